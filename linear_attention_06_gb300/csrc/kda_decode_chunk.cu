// kda_decode_chunk.cu -- a decode step of 2..16 tokens per sequence at dk = dv = 128, the
// step's tokens taken as one short chunk.
//
// The math (one head; tokens t = 0..T-1 of the step, S0 the state entering it, a_t = log
// alpha_t, g_t = sum_{s<=t} a_s, G = g_{T-1}) is the exact rewrite of the token recurrence of
// "Kimi K3 Architecture Teardown" (section "Hybrid Attention for 1M Tokens", Visual 5: decay,
// erase with beta, write with beta; the output read after the write) that the chunked prefill
// uses, with the decay of S0 moved onto the left factors so that S0 is used as it is read:
//
//   K_g = e^{g} o K,  Q_g = e^{g} o Q,  Kb = e^{G-g} o K,
//   A_ts = sum_c k_tc k_sc e^{g_tc - g_sc}  (s < t),  P_ts = sum_c q_tc k_sc e^{g_tc - g_sc}  (s <= t),
//   [W | U] = T [K_g | V] with T = (I + Diag(beta) A)^-1 Diag(beta)   (forward substitution),
//   Delta = U - W S0,   O = Q_g S0 + P Delta,   S = Diag(e^G) S0 + Kb^T Delta.
//
// A and P are formed as Khat Kb^T and Qhat Kb^T (Khat = e^{g-G} o K, Qhat = e^{g-G} o Q), so
// the form is taken while every key channel has G >= -60 (e^60 ~ 1e26, far inside the fp32
// range); a step that decays harder (log_alpha = -inf included) runs token by token in fp32
// instead, on the same register layout.  All other factors are e^{x} with x <= 0.
//
// Three products touch the state: W S0 and Q_g S0 (T x 128 by 128 x 128) and Kb^T Delta
// (128 x T by T x 128).  They run on the tensor cores (mma.sync m16n8k8, TF32 operands, fp32
// accumulation) with the state held in registers.  Warp w of the block owns the value columns
// 16w .. 16w+15 for all 128 key rows; lane 4 gi + qi holds S0[i][j] for
//   j in {16w + 2 gi, 16w + 2 gi + 1},  i in {8 b + 2 qi, 8 b + 2 qi + 1 : b = 0..15},
// which are, element for element, the A fragments of S0^T (fragment row gi <-> column
// 16w + 2 gi, row gi + 8 <-> column 16w + 2 gi + 1; fragment column qi <-> key row 8b + 2qi,
// column qi + 4 <-> key row 8b + 2qi + 1) for Delta^T = U^T - S0^T W^T and O^T = S0^T Q_g^T, and
// the accumulator fragments of S^T += Delta^T Kb.  The token index of Delta, P and Kb is
// permuted the same way (fragment k = qi <-> token 8kk + 2qi, k = qi + 4 <-> 8kk + 2qi + 1), so
// the accumulator of Delta^T is already the A fragment of the two products that read it.  The
// state therefore crosses HBM once in each direction, and no product needs a reduction across
// warps.  The small steps (cumulative decay, A and P, the solve) run in fp32 on the CUDA cores
// from shared memory; TF32 rounds the operands of the three state products to 11 significant
// bits while the carried state stays fp32 (the update adds into it in the fp32 accumulator).
//
// fp32 inputs always take that fp32 token loop (decay, the two column sums over the warp's own
// rows, the rank-one update), so they keep fp32 accuracy; in it a warp needs no other warp
// until the output store.
//
// One block of 256 threads per (sequence, head); two blocks fit an SM (84 KB of shared
// memory and at most 128 registers a thread each).
#include <atomic>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"
#include "sm103_primitives.cuh"

namespace kda {
namespace {
using namespace sm103;

constexpr int kD = 128;                 // dk = dv
constexpr int kThreads = 256;           // 8 warps x 16 value columns
constexpr int kTok = 16;                // tokens per step, padded with zero tokens
constexpr float kMaxExponent = 60.f;    // factored A and P while every channel has G >= -60
// Row strides (floats).  132 = 4 (mod 32): rows read as float4 by the A / P dot products, and
// the accumulator pairs of U (rows 2qi, columns 2gi); 136 = 8 (mod 32) and 24: the B fragments
// (eight rows gi, each read as a pair at column 2qi).  Each leaves the warp's loads without
// bank conflicts.
constexpr int kLd = 132, kLdB = 136, kLdT = 24;

struct Smem {
    float k[kTok][kLd];     // k; Khat for the factored A and P
    float q[kTok][kLd];     // q; Qhat
    float v[kTok][kLd];     // v; U after the solve
    float g[kTok][kLd];     // log alpha; then g_t (term-by-term A and P) or alpha (token loop)
    float kg[kTok][kLdB];   // K_g; -W in TF32 after the solve
    float kb[kTok][kLd];    // Kb
    float qg[kTok][kLdB];   // Q_g in TF32
    float kbt[kD][kLdT];    // Kb^T in TF32
    float pm[kTok][kLdT];   // P (s <= t, else 0) in TF32
    float am[kTok][kTok];   // A (s < t)
    float os[kTok][kLd];    // output rows
    float dec[kD];          // e^G per key channel
    float beta[kTok];
    float kq[kTok];         // k_t . q_t (token loop)
};

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void store8(float* s, const float (&x)[8]) {
    reinterpret_cast<float4*>(s)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(s)[1] = make_float4(x[4], x[5], x[6], x[7]);
}
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store4(float* p, float4 o) { *reinterpret_cast<float4*>(p) = o; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 o) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
}
__device__ __forceinline__ float4 load4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ float tf32f(float x) { return __uint_as_float(to_tf32(x)); }

// Position of (t, s) in the row-major lower triangle with (DIAG) or without the diagonal.
template <bool DIAG>
__device__ __forceinline__ void tri_index(int d, int& t, int& s) {
    t = DIAG ? 0 : 1;
    while ((DIAG ? (t + 1) * (t + 2) / 2 : (t + 1) * t / 2) <= d) ++t;
    s = d - (DIAG ? t * (t + 1) / 2 : t * (t - 1) / 2);
}

// sum_c x[c] y[c] over the 128 key channels (shared-memory rows).
__device__ __forceinline__ float row_dot(const float* x, const float* y) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
    for (int c = 0; c < kD; c += 4) {
        const float4 xv = *reinterpret_cast<const float4*>(x + c), yv = *reinterpret_cast<const float4*>(y + c);
        a0 = fmaf(xv.x, yv.x, a0);
        a1 = fmaf(xv.y, yv.y, a1);
        a0 = fmaf(xv.z, yv.z, a0);
        a1 = fmaf(xv.w, yv.w, a1);
    }
    return a0 + a1;
}

template <typename Tin>
struct Params {
    const Tin* q;
    const Tin* k;
    const Tin* v;
    const float* log_alpha;
    const Tin* beta;
    float* S;
    Tin* out;
    int H, T;
    const Tin* gate;
    const float* norm_w;
    float norm_eps;
    unsigned int* status;
};

// The step's token vectors into shared memory (rows T .. 15 zero: tokens that change nothing).
template <typename Tin>
__device__ __forceinline__ void stage_tokens(Smem& sm, const Params<Tin>& p, size_t row0, int64_t n_rows) {
    (void)n_rows;
    for (int i = threadIdx.x; i < kTok * (kD / 8); i += kThreads) {
        const int t = i / (kD / 8), c = (i % (kD / 8)) * 8;
        float kx[8], qx[8], vx[8], ax[8];
        const size_t e = (row0 + (size_t)t * p.H) * kD + c;
        if (t < p.T && KDA_INDEX_OK(e + 7, n_rows * kD, p.status)) {
            load8(p.k + e, kx); load8(p.q + e, qx); load8(p.v + e, vx); load8(p.log_alpha + e, ax);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) kx[u] = qx[u] = vx[u] = ax[u] = 0.f;
        }
        store8(&sm.k[t][c], kx); store8(&sm.q[t][c], qx); store8(&sm.v[t][c], vx); store8(&sm.g[t][c], ax);
    }
    if (threadIdx.x < kTok) {
        const int t = threadIdx.x;
        const size_t e = row0 + (size_t)t * p.H;
        sm.beta[t] = (t < p.T && KDA_INDEX_OK(e, n_rows, p.status)) ? to_f32(p.beta[e]) : 0.f;
    }
}

// out rows of the step from sm.os: plain, or gated (RMSNorm over the 128 channels x weight x
// sigmoid(gate)).  One warp per token, four channels a lane.
template <typename Tin>
__device__ __forceinline__ void store_outputs(const Smem& sm, const Params<Tin>& p, size_t row0, int64_t n_rows) {
    (void)n_rows;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = w; t < p.T; t += kThreads / 32) {
        const size_t e = (row0 + (size_t)t * p.H) * kD + 4 * lane;
        float4 o = *reinterpret_cast<const float4*>(&sm.os[t][4 * lane]);
        if (p.gate) {
            float ss = o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w;
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            const float rn = rsqrtf(ss * (1.f / kD) + p.norm_eps);
            if (KDA_INDEX_OK(e + 3, n_rows * kD, p.status)) {
                const float4 gv = load4(p.gate + e);
                const float* wp = p.norm_w + 4 * lane;   // the weight is only 4-byte aligned
                const float4 nw = make_float4(__ldg(wp), __ldg(wp + 1), __ldg(wp + 2), __ldg(wp + 3));
                o.x = o.x * rn * nw.x / (1.f + __expf(-gv.x));
                o.y = o.y * rn * nw.y / (1.f + __expf(-gv.y));
                o.z = o.z * rn * nw.z / (1.f + __expf(-gv.z));
                o.w = o.w * rn * nw.w / (1.f + __expf(-gv.w));
            }
        }
        if (KDA_INDEX_OK(e + 3, n_rows * kD, p.status)) store4(p.out + e, o);
    }
}

// fp32 token loop on the register layout: for each token, decay, the column sums S^T k and S^T q
// over the lane's rows (then across the four lanes qi that share the column pair), the erase /
// write delta, the output and the rank-one update.  Reads k, q, v, beta and log alpha from
// shared memory; writes the output rows to sm.os.
__device__ __forceinline__ void token_loop(Smem& sm, float (&s)[16][4], int T, int warp, int lane, int qi, int jc) {
    for (int i = threadIdx.x; i < T * kD; i += kThreads) {
        const int t = i / kD, c = i % kD;
        sm.g[t][c] = expf(sm.g[t][c]);
    }
    for (int t = warp; t < T; t += kThreads / 32) {
        const float4 kv = *reinterpret_cast<const float4*>(&sm.k[t][4 * lane]);
        const float4 qv = *reinterpret_cast<const float4*>(&sm.q[t][4 * lane]);
        float d = kv.x * qv.x + kv.y * qv.y + kv.z * qv.z + kv.w * qv.w;
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) d += __shfl_xor_sync(0xffffffffu, d, m);
        if (lane == 0) sm.kq[t] = d;
    }
    __syncthreads();
    for (int t = 0; t < T; ++t) {
        float2 r = make_float2(0.f, 0.f), y = r;
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            const int i = 8 * b + 2 * qi;
            const float2 al = *reinterpret_cast<const float2*>(&sm.g[t][i]);
            const float2 kv = *reinterpret_cast<const float2*>(&sm.k[t][i]);
            const float2 qv = *reinterpret_cast<const float2*>(&sm.q[t][i]);
            float2 s0 = make_float2(s[b][0], s[b][1]), s1 = make_float2(s[b][2], s[b][3]);
            s0 = __fmul2_rn(s0, make_float2(al.x, al.x));
            s1 = __fmul2_rn(s1, make_float2(al.y, al.y));
            r = __ffma2_rn(s0, make_float2(kv.x, kv.x), r);
            r = __ffma2_rn(s1, make_float2(kv.y, kv.y), r);
            y = __ffma2_rn(s0, make_float2(qv.x, qv.x), y);
            y = __ffma2_rn(s1, make_float2(qv.y, qv.y), y);
            s[b][0] = s0.x; s[b][1] = s0.y; s[b][2] = s1.x; s[b][3] = s1.y;
        }
#pragma unroll
        for (int m = 1; m < 4; m <<= 1) {
            r.x += __shfl_xor_sync(0xffffffffu, r.x, m);
            r.y += __shfl_xor_sync(0xffffffffu, r.y, m);
            y.x += __shfl_xor_sync(0xffffffffu, y.x, m);
            y.y += __shfl_xor_sync(0xffffffffu, y.y, m);
        }
        const float bt = sm.beta[t], kq = sm.kq[t];
        const float2 vv = *reinterpret_cast<const float2*>(&sm.v[t][jc]);
        const float2 dl = make_float2(bt * (vv.x - r.x), bt * (vv.y - r.y));
        if (qi == 0) *reinterpret_cast<float2*>(&sm.os[t][jc]) = make_float2(fmaf(kq, dl.x, y.x), fmaf(kq, dl.y, y.y));
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            const float2 kv = *reinterpret_cast<const float2*>(&sm.k[t][8 * b + 2 * qi]);
            float2 s0 = make_float2(s[b][0], s[b][1]), s1 = make_float2(s[b][2], s[b][3]);
            s0 = __ffma2_rn(make_float2(kv.x, kv.x), dl, s0);
            s1 = __ffma2_rn(make_float2(kv.y, kv.y), dl, s1);
            s[b][0] = s0.x; s[b][1] = s0.y; s[b][2] = s1.x; s[b][3] = s1.y;
        }
    }
}

// The chunk form after the scaled rows are in shared memory: A and P, the solve, and the three
// state products on the tensor cores; writes the output rows to sm.os and leaves the new state
// in s.
template <int NT>
__device__ __forceinline__ void chunk_products(Smem& sm, float (&s)[16][4], int T, int warp, int gi, int qi,
                                               int jc) {
    constexpr int kT8 = 8 * NT;
    (void)warp;
    // ---- A (s < t: 120 dot products) and P (s <= t: 136), one per thread ----
    {
        const int d = threadIdx.x;
        int t, s2;
        const bool isA = d < 120;
        if (isA) tri_index<false>(d, t, s2);
        else tri_index<true>(d - 120, t, s2);
        const float val = t < T ? row_dot(isA ? sm.k[t] : sm.q[t], sm.kb[s2]) : 0.f;
        if (isA) sm.am[t][s2] = val;
        else sm.pm[t][s2] = tf32f(val);
    }
    __syncthreads();

    // ---- forward substitution: thread col solves column col of [W | U] = T [K_g | V] ----
    {
        const int col = threadIdx.x;
        float* ycol = col < kD ? &sm.kg[0][col] : &sm.v[0][col - kD];
        const int ld = col < kD ? kLdB : kLd;
        float x[kT8];
#pragma unroll
        for (int t = 0; t < kT8; ++t) {
            float a0 = ycol[t * ld], a1 = 0.f;
#pragma unroll
            for (int u = 0; u < t; ++u) {
                if (u & 1) a1 = fmaf(-sm.am[t][u], x[u], a1);
                else a0 = fmaf(-sm.am[t][u], x[u], a0);
            }
            x[t] = sm.beta[t] * (a0 + a1);
            ycol[t * ld] = col < kD ? -tf32f(x[t]) : x[t];
        }
    }
    __syncthreads();

    // ---- the state products on the tensor cores ----
    float dt[NT][4], ot[NT][4];                      // Delta^T and O^T accumulators
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float2 u0 = *reinterpret_cast<const float2*>(&sm.v[8 * nt + 2 * qi][jc]);
        const float2 u1 = *reinterpret_cast<const float2*>(&sm.v[8 * nt + 2 * qi + 1][jc]);
        dt[nt][0] = u0.x; dt[nt][1] = u1.x; dt[nt][2] = u0.y; dt[nt][3] = u1.y;
        ot[nt][0] = ot[nt][1] = ot[nt][2] = ot[nt][3] = 0.f;
    }
#pragma unroll
    for (int b = 0; b < 16; ++b) {
        const uint32_t a[4] = {to_tf32(s[b][0]), to_tf32(s[b][1]), to_tf32(s[b][2]), to_tf32(s[b][3])};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint2 bw = *reinterpret_cast<const uint2*>(&sm.kg[8 * nt + gi][8 * b + 2 * qi]);
            const uint2 bq = *reinterpret_cast<const uint2*>(&sm.qg[8 * nt + gi][8 * b + 2 * qi]);
            const uint32_t fw[2] = {bw.x, bw.y}, fq[2] = {bq.x, bq.y};
            mma_tf32(dt[nt], a, fw);                 // Delta^T = U^T - S0^T W^T
            mma_tf32(ot[nt], a, fq);                 // O^T = S0^T Q_g^T
        }
    }
    uint32_t ad[NT][4];                              // Delta^T as the A fragment (token-permuted k)
#pragma unroll
    for (int kk = 0; kk < NT; ++kk) {
        ad[kk][0] = to_tf32(dt[kk][0]); ad[kk][1] = to_tf32(dt[kk][2]);
        ad[kk][2] = to_tf32(dt[kk][1]); ad[kk][3] = to_tf32(dt[kk][3]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int kk = 0; kk < NT; ++kk) {
            const uint2 bp = *reinterpret_cast<const uint2*>(&sm.pm[8 * nt + gi][8 * kk + 2 * qi]);
            const uint32_t fp[2] = {bp.x, bp.y};
            mma_tf32(ot[nt], ad[kk], fp);            // O^T += Delta^T P^T
        }
        *reinterpret_cast<float2*>(&sm.os[8 * nt + 2 * qi][jc]) = make_float2(ot[nt][0], ot[nt][2]);
        *reinterpret_cast<float2*>(&sm.os[8 * nt + 2 * qi + 1][jc]) = make_float2(ot[nt][1], ot[nt][3]);
    }
#pragma unroll
    for (int b = 0; b < 16; ++b) {                   // S^T = S0^T Diag(e^G) + Delta^T Kb
        const float2 dc = *reinterpret_cast<const float2*>(&sm.dec[8 * b + 2 * qi]);
        float acc[4] = {s[b][0] * dc.x, s[b][2] * dc.y, s[b][1] * dc.x, s[b][3] * dc.y};
#pragma unroll
        for (int kk = 0; kk < NT; ++kk) {
            const uint2 bk = *reinterpret_cast<const uint2*>(&sm.kbt[8 * b + gi][8 * kk + 2 * qi]);
            const uint32_t fk[2] = {bk.x, bk.y};
            mma_tf32(acc, ad[kk], fk);
        }
        s[b][0] = acc[0]; s[b][2] = acc[1]; s[b][1] = acc[2]; s[b][3] = acc[3];
    }
}

// NT = number of 8-token blocks the step's tokens fill (1: T <= 8, 2: T <= 16).
template <typename Tin, int NT>
__global__ void __launch_bounds__(kThreads, 2) decode_chunk_kernel(const Params<Tin> p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    constexpr bool kTensor = sizeof(Tin) == 2;     // bf16 inputs: the tensor-core form

    const size_t pair = blockIdx.x;                 // (sequence, head)
    const size_t n = pair / p.H, h = pair % p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, qi = lane & 3;
    const int jc = 16 * warp + 2 * gi;              // this lane's value columns jc, jc + 1
    float* Sp = p.S + pair * kD * kD;
    const int64_t n_state = (int64_t)gridDim.x * kD * kD;
    const int64_t n_rows = (int64_t)gridDim.x * p.T;  // rows of q, k, v, out: num_seqs x T x H
    const size_t row0 = n * (size_t)p.T * p.H + h;    // row of token 0; token t is row0 + t H

    // The state first, so its read overlaps everything up to the products.
    // s[b][0..1] = S0[8b + 2qi][jc, jc+1], s[b][2..3] = S0[8b + 2qi + 1][jc, jc+1].
    float s[16][4];
#pragma unroll
    for (int b = 0; b < 16; ++b) {
        const int i = 8 * b + 2 * qi;
        const bool ok = KDA_INDEX_OK((int64_t)pair * kD * kD + (int64_t)(i + 1) * kD + jc + 1, n_state, p.status);
        const float2 r0 = ok ? __ldcs(reinterpret_cast<const float2*>(Sp + (size_t)i * kD + jc)) : make_float2(0.f, 0.f);
        const float2 r1 = ok ? __ldcs(reinterpret_cast<const float2*>(Sp + (size_t)(i + 1) * kD + jc))
                             : make_float2(0.f, 0.f);
        s[b][0] = r0.x; s[b][1] = r0.y; s[b][2] = r1.x; s[b][3] = r1.y;
    }
    (void)n_state;                                  // read by the index checks of bounds-checked builds

    stage_tokens(sm, p, row0, n_rows);
    __syncthreads();

    bool chunk_form = false;
    if constexpr (kTensor) {
        // ---- per key channel c: the cumulative decay g_t and whether the chunk form holds ----
        constexpr int kT8 = 8 * NT;                  // token rows the products read
        const int c = threadIdx.x & (kD - 1);
        const bool kside = threadIdx.x < kD;
        float gt[kT8];
        float run = 0.f;
#pragma unroll
        for (int t = 0; t < kT8; ++t) { run += sm.g[t][c]; gt[t] = run; }
        const float G = gt[kT8 - 1];                 // padded tokens add log alpha = 0
        chunk_form = __syncthreads_and(G >= -kMaxExponent) != 0;   // false for NaN and -inf too
        if (chunk_form) {
            if (kside) {
#pragma unroll
                for (int t = 0; t < kT8; ++t) {
                    const float kv = sm.k[t][c];
                    const float kb = __expf(G - gt[t]) * kv;
                    sm.kb[t][c] = kb;
                    sm.kbt[c][t] = tf32f(kb);
                    sm.kg[t][c] = __expf(gt[t]) * kv;
                    sm.k[t][c] = __expf(gt[t] - G) * kv;
                }
                sm.dec[c] = __expf(G);
            } else {
#pragma unroll
                for (int t = 0; t < kT8; ++t) {
                    const float qv = sm.q[t][c];
                    sm.qg[t][c] = tf32f(__expf(gt[t]) * qv);
                    sm.q[t][c] = __expf(gt[t] - G) * qv;
                }
            }
            if (threadIdx.x < kTok * kTok / 8) {      // P above the diagonal stays 0
                const int i = threadIdx.x * 8, t = i / kTok, s0 = i % kTok;
                *reinterpret_cast<float4*>(&sm.pm[t][s0]) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4*>(&sm.pm[t][s0 + 4]) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            __syncthreads();
            chunk_products<NT>(sm, s, p.T, warp, gi, qi, jc);
        }
    }
    if (!chunk_form) {
        token_loop(sm, s, p.T, warp, lane, qi, jc);
    }

#pragma unroll
    for (int b = 0; b < 16; ++b) {
        const int i = 8 * b + 2 * qi;
        if (KDA_INDEX_OK((int64_t)pair * kD * kD + (int64_t)(i + 1) * kD + jc + 1, n_state, p.status)) {
            __stcs(reinterpret_cast<float2*>(Sp + (size_t)i * kD + jc), make_float2(s[b][0], s[b][1]));
            __stcs(reinterpret_cast<float2*>(Sp + (size_t)(i + 1) * kD + jc), make_float2(s[b][2], s[b][3]));
        }
    }
    __syncthreads();
    store_outputs(sm, p, row0, n_rows);
}

template <typename Tin, int NT>
cudaError_t launch_t(const Params<Tin>& p, unsigned blocks, cudaStream_t st) {
    static std::atomic<bool> attr_set[64];           // the shared-memory opt-in, once per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(decode_chunk_kernel<Tin, NT>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    decode_chunk_kernel<Tin, NT><<<blocks, kThreads, sizeof(Smem), st>>>(p);
    return cudaGetLastError();
}

template <typename Tin>
Params<Tin> params(const DecodeArgs& a) {
    return Params<Tin>{static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v),
                       a.log_alpha, static_cast<const Tin*>(a.beta), a.state, static_cast<Tin*>(a.out),
                       a.H, a.tokens_per_seq, static_cast<const Tin*>(a.gate), a.norm_w, a.norm_eps, a.status};
}

}  // namespace

bool decode_chunk_supported(const DecodeArgs& a) {
    return a.dk == kD && a.dv == kD && a.tokens_per_seq >= 2 && a.tokens_per_seq <= kTok;
}

cudaError_t launch_decode_chunk(const DecodeArgs& a, cudaStream_t st) {
    if (a.num_seqs == 0) return cudaSuccess;
    if (!decode_chunk_supported(a)) return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)((size_t)a.num_seqs * a.H);
    if (a.dtype == DType::F32) return launch_t<float, 2>(params<float>(a), blocks, st);
    return a.tokens_per_seq <= 8 ? launch_t<__nv_bfloat16, 1>(params<__nv_bfloat16>(a), blocks, st)
                                 : launch_t<__nv_bfloat16, 2>(params<__nv_bfloat16>(a), blocks, st);
}

}  // namespace kda
