// kda_decode_chunk.cu -- a decode step of 3..16 tokens per sequence at dk = dv = 128, the
// step's tokens taken as one short chunk (steps of one or two tokens run faster through the
// token loop of kda_decode.cu: 199 us against 234 us at two tokens, 256 x 32 heads).
//
// The math (one head; tokens t = 0..T-1 of the step, S0 the state entering it, a_t = log
// alpha_t, g_t = sum_{s<=t} a_s, G = g_{T-1}) is the exact rewrite of the token recurrence of
// "Kimi K3 Architecture Teardown" (section "Hybrid Attention for 1M Tokens", Visual 5: decay,
// erase with beta, write with beta; the output read after the write) that the chunked prefill
// uses, with the decay of S0 moved onto the left factors so that S0 is used as it is read:
//
//   K_g = e^{g} o K,  Q_g = e^{g} o Q,  Kb = e^{G-g} o K,
//   A_ts = sum_c k_tc k_sc e^{g_tc - g_sc}  (s < t),  P_ts = sum_c q_tc k_sc e^{g_tc - g_sc}  (s <= t),
//   R = V - K_g S0,   (I + Diag(beta) A) Delta = Diag(beta) R,
//   O = Q_g S0 + P Delta,   S = Diag(e^G) S0 + Kb^T Delta.
//
// (Delta = T R with T = (I + Diag(beta) A)^-1 Diag(beta) is the UT / WY form U - W S0 with
// U = T V and W = T K_g, applied in the other order: no T is formed; each warp solves the
// triangular system for its own columns of R by forward substitution.)  A and P are formed as
// Khat Kb^T and Qhat Kb^T (Khat = e^{g-G} o K, Qhat = e^{g-G} o Q), so the form is taken while
// every key channel has G >= -60 (e^60 ~ 1e26, far inside the fp32 range); a step that decays
// harder (log_alpha = -inf included) runs token by token in fp32 instead, on the same register
// layout.  All other factors are e^{x} with x <= 0.
//
// Products.  K_g S0 and Q_g S0 (T x 128 by 128 x 128) and Kb^T Delta (128 x T by T x 128) touch
// the state; they run on the tensor cores (mma.sync m16n8k8, TF32 operands, fp32 accumulation)
// with the state held in registers.  Warp w of the block owns the value columns 16w .. 16w+15
// for all 128 key rows; lane 4 gi + qi holds S0[i][j] for
//   j in {16w + 2 gi, 16w + 2 gi + 1},  i in {8 b + 2 qi, 8 b + 2 qi + 1 : b = 0..15},
// which are, element for element, the A fragments of S0^T (fragment row gi <-> column
// 16w + 2 gi, row gi + 8 <-> column 16w + 2 gi + 1; fragment column qi <-> key row 8b + 2qi,
// column qi + 4 <-> key row 8b + 2qi + 1) for R^T = V^T - S0^T K_g^T and O^T = S0^T Q_g^T, and
// the accumulator fragments of S^T += Delta^T Kb.  The token index of R, Delta, P and Kb is
// permuted the same way (fragment k = qi <-> token 8kk + 2qi, k = qi + 4 <-> 8kk + 2qi + 1), so
// an accumulator over tokens is already the A fragment of the next product that reads it.  The
// state crosses HBM once in each direction, and no product needs a reduction across warps.
// TF32 rounds the operands of these products to 11 significant bits; the carried state stays
// fp32 (the update adds into it in the fp32 accumulator).  A and P take TF32 operands too (Khat,
// Qhat and Kb rounded once when they are formed; the chunked prefill forms them from bf16
// operands, three bits fewer), and the triangular solve runs in fp32 on the accumulator of R:
// the lanes holding token s compute Delta_s and pass it by shuffle to the three other lanes of
// their column pair, which subtract A_ts Delta_s from their later tokens.
//
// Schedule of one (sequence, head): the state is loaded into registers while the step's token
// vectors are staged in shared memory; per key channel the cumulative decay and the scaled
// rows; A and P (2 NT warps) and the first pass over the state (every warp); then per warp the
// solve, the output and the state update.
//
// The token loop (decay, the two column sums over the warp's own rows, the rank-one update) is
// exact fp32 arithmetic; in it a warp needs no other warp until the output store.  Inputs in
// fp32 do not come here: they keep the one-token kernel's token loop, which is as fast for them
// and gives the same bits as T one-token steps.
//
// Blocks are persistent, two per SM (59,008 bytes of shared memory a block for 9..16 tokens,
// 35,968 for 3..8, and at most 128 registers a thread), and walk the (sequence, head) pairs
// with a stride of the grid size; each prefetches the state and token rows of its next pair
// into L2 when it starts a pair, so that their DRAM reads overlap its arithmetic.
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
constexpr float kMaxExponent = 60.f;    // chunk form while every channel has G >= -60
constexpr float kLog2e = 1.4426950408889634f;
// Row strides (floats).  136 = 8 (mod 32) and 24: fragments read as pairs by eight rows gi at
// column 2qi; 132 = 4 (mod 32): the accumulator pairs of V and O (rows 2qi, columns 2gi); 20: the
// rows 2qi (+1) of A read as float4 by the solve.  Each leaves the warp's shared-memory loads
// without bank conflicts.
constexpr int kLd = 132, kLdB = 136, kLdT = 24, kLdA = 20;

// Arrays whose lives do not overlap share storage: log alpha is dead once the barrier that
// decides the chunk form has passed, when Kb^T is written; -K_g is dead after the first state
// pass, before the output rows are written (the token loop uses neither Kb^T nor K_g).  A
// smaller block footprint measured faster (T = 16: 318 us at 66 KiB, 326 us at 83 KiB).  The
// Gram products read Kb from its transposed TF32 copy (no second Kb tile), and the token rows
// are sized to the instance (8 NT rows: a step of at most 8 tokens keeps half the rows).
template <int NT>
struct Smem {
    static constexpr int R = 8 * NT;   // token rows: the step's tokens padded to whole 8-token blocks
    float k[R][kLdB];     // k; Khat
    float q[R][kLdB];     // q; Qhat
    float v[R][kLd];      // v
    union {
        float g[R][kLd];      // log alpha; alpha in the token loop
        float kbt[kD][kLdT];     // Kb^T in TF32 (written once the chunk form is decided)
    };
    union {
        float kg[R][kLdB];    // -K_g in TF32 (read by the first state pass)
        float os[R][kLd];     // output rows (written after it; the token loop has no K_g)
    };
    float qg[R][kLdB];    // Q_g in TF32
    float am[R][kLdA];    // A (s < t, else 0)
    float pm[R][kLdT];    // P (s <= t, else 0) in TF32
    float dec[kD];           // e^G per key channel
    float beta[kTok];
    float kq[kTok];          // k_t . q_t (token loop)
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
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 o) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ float tf32f(float x) { return __uint_as_float(to_tf32(x)); }
__device__ __forceinline__ float ex2(float x) {       // 2^x, the SFU's approximation
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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
    int pairs, H, T;
    const Tin* gate;
    const float* norm_w;
    float norm_eps;
    unsigned int* status;
};

// State of one pair into registers, directly in the fragment layout: two 8-byte loads per b
// (rows 8b + 2qi and 8b + 2qi + 1, columns jc and jc + 1).
__device__ __forceinline__ void load_state(const float* Sp, float (&s)[16][4], int64_t first, int64_t n_state,
                                           unsigned int* status, int jc, int qi) {
    (void)first; (void)n_state; (void)status;
#pragma unroll
    for (int b = 0; b < 16; ++b) {
        const int i = 8 * b + 2 * qi;
        float2 r0 = make_float2(0.f, 0.f), r1 = r0;
        if (KDA_INDEX_OK(first + (i + 1) * kD + jc + 1, n_state, status)) {
            r0 = __ldcs(reinterpret_cast<const float2*>(Sp + i * kD + jc));
            r1 = __ldcs(reinterpret_cast<const float2*>(Sp + (i + 1) * kD + jc));
        }
        s[b][0] = r0.x; s[b][1] = r0.y; s[b][2] = r1.x; s[b][3] = r1.y;
    }
}
__device__ __forceinline__ void store_state(float* Sp, const float (&s)[16][4], int64_t first, int64_t n_state,
                                            unsigned int* status, int jc, int qi) {
    (void)first; (void)n_state; (void)status;
#pragma unroll
    for (int b = 0; b < 16; ++b) {
        const int i = 8 * b + 2 * qi;
        if (KDA_INDEX_OK(first + (i + 1) * kD + jc + 1, n_state, status)) {
            __stcs(reinterpret_cast<float2*>(Sp + i * kD + jc), make_float2(s[b][0], s[b][1]));
            __stcs(reinterpret_cast<float2*>(Sp + (i + 1) * kD + jc), make_float2(s[b][2], s[b][3]));
        }
    }
}

// L2 prefetch of a pair's state and token rows (no completion is waited for).
template <typename Tin>
__device__ __forceinline__ void prefetch_pair(const Params<Tin>& p, int pair) {
    const size_t n = (size_t)pair / p.H, h = (size_t)pair % p.H;
    const size_t row0 = n * (size_t)p.T * p.H + h;
    if (threadIdx.x == 0) bulk_prefetch_l2(p.S + (size_t)pair * kD * kD, kD * kD * sizeof(float));
    const int i = (int)threadIdx.x - 32;                 // warps 1 and 2: one token row each
    if (i >= 0 && i < 4 * p.T) {
        const int t = i >> 2, a = i & 3;
        const size_t e = (row0 + (size_t)t * p.H) * kD;
        if (a == 3) bulk_prefetch_l2(p.log_alpha + e, kD * sizeof(float));
        else bulk_prefetch_l2((a == 0 ? p.q : a == 1 ? p.k : p.v) + e, kD * sizeof(Tin));
    }
}

// The step's token vectors into shared memory (rows T .. 15 zero: tokens that change nothing).
template <int NT, typename Tin>
__device__ __forceinline__ void stage_tokens(Smem<NT>& sm, const Params<Tin>& p, size_t row0, int64_t n_rows) {
    (void)n_rows;
    for (int i = threadIdx.x; i < Smem<NT>::R * (kD / 8); i += kThreads) {
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
template <int NT, typename Tin>
__device__ __forceinline__ void store_outputs(const Smem<NT>& sm, const Params<Tin>& p, size_t row0, int64_t n_rows) {
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
template <int NT>
__device__ __forceinline__ void token_loop(Smem<NT>& sm, float (&s)[16][4], int T, int warp, int lane, int qi, int jc) {
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

// Per key channel c (threads c and c + 128, one half of the step's token rows each): the
// cumulative decay in base 2 and the scaled rows.  Returns whether the chunk form holds (the
// same answer in every thread).
template <int NT>
__device__ __forceinline__ bool scale_rows(Smem<NT>& sm) {
    constexpr int kT8 = 8 * NT, kTH = kT8 / 2;       // token rows, rows per half
    const int c = threadIdx.x & (kD - 1), half = threadIdx.x >> 7;
    float run = 0.f;
    for (int t = 0; t < half * kTH; ++t) run += sm.g[t][c];
    float gl[kTH];
#pragma unroll
    for (int i = 0; i < kTH; ++i) { run += sm.g[half * kTH + i][c]; gl[i] = run; }
    for (int t = (half + 1) * kTH; t < kT8; ++t) run += sm.g[t][c];
    const float G = run;                             // the same order of additions in both halves
    if (!__syncthreads_and(G >= -kMaxExponent)) return false;   // false for NaN and -inf too
    const float G2 = G * kLog2e;
    float kbt[kTH];
#pragma unroll
    for (int i = 0; i < kTH; ++i) {
        const int t = half * kTH + i;
        const float g2 = gl[i] * kLog2e;
        const float eg = ex2(g2), eb = ex2(G2 - g2), eh = ex2(g2 - G2);
        const float kv = sm.k[t][c], qv = sm.q[t][c];
        kbt[i] = tf32f(eb * kv);
        sm.kg[t][c] = -tf32f(eg * kv);
        sm.k[t][c] = tf32f(eh * kv);
        sm.qg[t][c] = tf32f(eg * qv);
        sm.q[t][c] = tf32f(eh * qv);
    }
#pragma unroll
    for (int i = 0; i < kTH; i += 4)
        *reinterpret_cast<float4*>(&sm.kbt[c][half * kTH + i]) = make_float4(kbt[i], kbt[i + 1], kbt[i + 2], kbt[i + 3]);
    if (half == 0) sm.dec[c] = ex2(G2);
    return true;
}

// A = Khat Kb^T and P = Qhat Kb^T, 16 x 8 tiles on the tensor cores, TF32 operands as stored
// (fragment k = qi <-> channel 8b + 2qi, k = qi + 4 <-> 8b + 2qi + 1); warp w < 2 NT takes tile
// w (A for w < NT, P after), two accumulators (even and odd channel blocks) over the 128 channels.
template <int NT>
__device__ __forceinline__ void gram_tile(Smem<NT>& sm, int warp, int gi, int qi) {
    const bool isP = warp >= NT;
    const int nt = warp % NT;
    const float* X = isP ? &sm.q[0][0] : &sm.k[0][0];
    float acc[2][4] = {};                            // two accumulators: even and odd channel blocks
#pragma unroll
    for (int b = 0; b < 16; ++b) {
        const uint2 x0 = *reinterpret_cast<const uint2*>(X + gi * kLdB + 8 * b + 2 * qi);
        const uint2 x1 = NT > 1 ? *reinterpret_cast<const uint2*>(X + (gi + 8) * kLdB + 8 * b + 2 * qi)
                                : make_uint2(0u, 0u);   // padding tokens 8-15 of a one-block step
        const uint32_t a[4] = {x0.x, x1.x, x0.y, x1.y};
        const uint32_t bb[2] = {__float_as_uint(sm.kbt[8 * b + 2 * qi][8 * nt + gi]),
                                __float_as_uint(sm.kbt[8 * b + 2 * qi + 1][8 * nt + gi])};
        mma_tf32(acc[b & 1], a, bb);
    }
    float c[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) c[e] = acc[0][e] + acc[1][e];
    // c: (t = gi, s = 8 nt + 2 qi, +1), (t = gi + 8, same s)
    const int s0 = 8 * nt + 2 * qi;
    if (isP) {
        *reinterpret_cast<float2*>(&sm.pm[gi][s0]) =
            make_float2(s0 <= gi ? tf32f(c[0]) : 0.f, s0 + 1 <= gi ? tf32f(c[1]) : 0.f);
        if (NT > 1)
            *reinterpret_cast<float2*>(&sm.pm[gi + 8][s0]) =
                make_float2(s0 <= gi + 8 ? tf32f(c[2]) : 0.f, s0 + 1 <= gi + 8 ? tf32f(c[3]) : 0.f);
    } else {
        *reinterpret_cast<float2*>(&sm.am[gi][s0]) = make_float2(s0 < gi ? c[0] : 0.f, s0 + 1 < gi ? c[1] : 0.f);
        if (NT > 1)
            *reinterpret_cast<float2*>(&sm.am[gi + 8][s0]) =
                make_float2(s0 < gi + 8 ? c[2] : 0.f, s0 + 1 < gi + 8 ? c[3] : 0.f);
    }
}

// (I + Diag(beta) A) Delta = Diag(beta) R on the warp's columns, in place on the accumulator rt
// of R^T (rt[nt][p] / rt[nt][2 + p]: token 8 nt + 2 qi + p, columns jc / jc + 1).  Step s: the
// lanes with qi = (s mod 8) / 2 hold token s and finish Delta_s = beta_s x (R_s - the terms
// already subtracted); a shuffle gives it to the other lanes of the column pair, which subtract
// A_ts Delta_s from every later token t they hold (A is zero on and above the diagonal).
template <int NT>
__device__ __forceinline__ void solve_delta(const Smem<NT>& sm, float (&rt)[NT][4], int lane, int qi) {
    constexpr int kT8 = 8 * NT;
#pragma unroll
    for (int s4 = 0; s4 < kT8; s4 += 4) {
        float4 a[NT][2];                             // A[8 nt + 2 qi + p][s4 .. s4 + 3]
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int p = 0; p < 2; ++p)
                if (nt >= s4 / 8)                    // earlier token blocks take no update from here
                    a[nt][p] = *reinterpret_cast<const float4*>(&sm.am[8 * nt + 2 * qi + p][s4]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int s = s4 + u, ns = s >> 3, ps = s & 1, qs = (s & 7) >> 1;
            const float bs = sm.beta[s];
            const bool own = qi == qs;
            const float d0 = bs * rt[ns][ps], d1 = bs * rt[ns][2 + ps];
            if (own) { rt[ns][ps] = d0; rt[ns][2 + ps] = d1; }
            const int src = (lane & ~3) | qs;
            const float D0 = __shfl_sync(0xffffffffu, d0, src), D1 = __shfl_sync(0xffffffffu, d1, src);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    if (nt < ns) continue;               // tokens of block nt < ns all precede token s
                    const float4 av = a[nt][p];
                    const float ats = u == 0 ? av.x : u == 1 ? av.y : u == 2 ? av.z : av.w;
                    rt[nt][p] = fmaf(-ats, D0, rt[nt][p]);
                    rt[nt][2 + p] = fmaf(-ats, D1, rt[nt][2 + p]);
                }
        }
    }
}

// Chunk form after scale_rows: returns with the output rows in sm.os and the new state in s.
template <int NT>
__device__ __forceinline__ void chunk_products(Smem<NT>& sm, float (&s)[16][4], int warp, int lane, int gi, int qi,
                                               int jc) {
    if (warp < 2 * NT) gram_tile<NT>(sm, warp, gi, qi);

    // R^T = V^T - S0^T K_g^T and O^T = S0^T Q_g^T (accumulator: row <-> column jc / jc + 1,
    // column <-> token 8 nt + 2 qi / + 1)
    float rt[NT][4], ot[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float2 v0 = *reinterpret_cast<const float2*>(&sm.v[8 * nt + 2 * qi][jc]);
        const float2 v1 = *reinterpret_cast<const float2*>(&sm.v[8 * nt + 2 * qi + 1][jc]);
        rt[nt][0] = v0.x; rt[nt][1] = v1.x; rt[nt][2] = v0.y; rt[nt][3] = v1.y;
        ot[nt][0] = ot[nt][1] = ot[nt][2] = ot[nt][3] = 0.f;
    }
#pragma unroll
    for (int b = 0; b < 16; ++b) {
        const uint32_t a[4] = {to_tf32(s[b][0]), to_tf32(s[b][1]), to_tf32(s[b][2]), to_tf32(s[b][3])};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint2 bk = *reinterpret_cast<const uint2*>(&sm.kg[8 * nt + gi][8 * b + 2 * qi]);
            const uint2 bq = *reinterpret_cast<const uint2*>(&sm.qg[8 * nt + gi][8 * b + 2 * qi]);
            const uint32_t fk[2] = {bk.x, bk.y}, fq[2] = {bq.x, bq.y};
            mma_tf32(rt[nt], a, fk);
            mma_tf32(ot[nt], a, fq);
        }
    }
    __syncthreads();                                 // A and P are in shared memory

    solve_delta<NT>(sm, rt, lane, qi);               // rt now holds Delta^T
    uint32_t ad[NT][4];                              // Delta^T as the A fragment (token-permuted k)
#pragma unroll
    for (int kk = 0; kk < NT; ++kk) {
        ad[kk][0] = to_tf32(rt[kk][0]); ad[kk][1] = to_tf32(rt[kk][2]);
        ad[kk][2] = to_tf32(rt[kk][1]); ad[kk][3] = to_tf32(rt[kk][3]);
    }
    // O^T += Delta^T P^T, then the output rows
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int kk = 0; kk < NT; ++kk) {
            const uint2 bp = *reinterpret_cast<const uint2*>(&sm.pm[8 * nt + gi][8 * kk + 2 * qi]);
            const uint32_t fp[2] = {bp.x, bp.y};
            mma_tf32(ot[nt], ad[kk], fp);
        }
        *reinterpret_cast<float2*>(&sm.os[8 * nt + 2 * qi][jc]) = make_float2(ot[nt][0], ot[nt][2]);
        *reinterpret_cast<float2*>(&sm.os[8 * nt + 2 * qi + 1][jc]) = make_float2(ot[nt][1], ot[nt][3]);
    }
    // S^T = S0^T Diag(e^G) + Delta^T Kb
#pragma unroll
    for (int b = 0; b < 16; ++b) {
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
    Smem<NT>& sm = *reinterpret_cast<Smem<NT>*>(smem_raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, qi = lane & 3;
    const int jc = 16 * warp + 2 * gi;               // this lane's value columns jc, jc + 1
    const int64_t n_state = (int64_t)p.pairs * kD * kD;
    const int64_t n_rows = (int64_t)p.pairs * p.T;   // rows of q, k, v, out: num_seqs x T x H
    (void)n_state;                                   // read by the index checks of bounds-checked builds

    for (int pair = blockIdx.x; pair < p.pairs; pair += gridDim.x) {
        const size_t n = (size_t)pair / p.H, h = (size_t)pair % p.H;
        const size_t row0 = n * (size_t)p.T * p.H + h;   // row of token 0; token t is row0 + t H
        float* Sp = p.S + (size_t)pair * kD * kD;
        if (pair + (int)gridDim.x < p.pairs) prefetch_pair(p, pair + gridDim.x);

        float s[16][4];
        load_state(Sp, s, (int64_t)pair * kD * kD, n_state, p.status, jc, qi);
        stage_tokens(sm, p, row0, n_rows);
        __syncthreads();

        const bool chunk_form = scale_rows<NT>(sm);
        if (chunk_form) {
            __syncthreads();
            chunk_products<NT>(sm, s, warp, lane, gi, qi, jc);
        } else {
            token_loop(sm, s, p.T, warp, lane, qi, jc);
        }
        store_state(Sp, s, (int64_t)pair * kD * kD, n_state, p.status, jc, qi);
        __syncthreads();
        store_outputs(sm, p, row0, n_rows);
    }
}

template <typename Tin, int NT>
cudaError_t launch_t(const Params<Tin>& p, cudaStream_t st) {
    static std::atomic<bool> attr_set[64];           // the shared-memory opt-in, once per device
    static std::atomic<int> sm_count[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(decode_chunk_kernel<Tin, NT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem<NT>));
        int sms = 0;
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        sm_count[dev].store(sms > 0 ? sms : 1, std::memory_order_relaxed);
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int resident = 2 * sm_count[dev].load(std::memory_order_relaxed);   // two blocks an SM
    const unsigned blocks = (unsigned)(p.pairs < resident ? p.pairs : resident);
    decode_chunk_kernel<Tin, NT><<<blocks, kThreads, sizeof(Smem<NT>), st>>>(p);
    return cudaGetLastError();
}

template <typename Tin>
Params<Tin> params(const DecodeArgs& a) {
    return Params<Tin>{static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v),
                       a.log_alpha, static_cast<const Tin*>(a.beta), a.state, static_cast<Tin*>(a.out),
                       a.num_seqs * a.H, a.H, a.tokens_per_seq, static_cast<const Tin*>(a.gate), a.norm_w,
                       a.norm_eps, a.status};
}

}  // namespace

bool decode_chunk_supported(const DecodeArgs& a) {
    return a.dtype == DType::BF16 && a.dk == kD && a.dv == kD && a.tokens_per_seq >= 3 && a.tokens_per_seq <= kTok;
}

cudaError_t launch_decode_chunk(const DecodeArgs& a, cudaStream_t st) {
    if (a.num_seqs == 0) return cudaSuccess;
    if (!decode_chunk_supported(a) || (int64_t)a.num_seqs * a.H > INT32_MAX / 2) return cudaErrorInvalidValue;
    return a.tokens_per_seq <= 8 ? launch_t<__nv_bfloat16, 1>(params<__nv_bfloat16>(a), st)
                                 : launch_t<__nv_bfloat16, 2>(params<__nv_bfloat16>(a), st);
}

}  // namespace kda
