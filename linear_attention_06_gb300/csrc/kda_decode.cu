// kda_decode.cu -- one KDA decode step, memory-bound.
//
// For each (sequence, head) the fp32 state S (dk x dv) is streamed from HBM
// once and written back once, in place.  With alpha = exp(log_alpha):
//   S' = Diag(alpha) S                         decay ("Kimi K3 Architecture
//                                              Teardown", Visual 5, step one)
//   r  = S'^T k,  y = S'^T q                   one pass over S'
//   delta = beta (v - r)                       erase + write with one beta
//                                              ("Kimi K3 Architecture: KDA,
//                                              MoE, and Attention", section
//                                              "Memory as a First-Class Problem")
//   S  = S' + k delta^T                        written back in place
//   o  = S^T q = y + (k . q) delta             read after write
//
// Several tokens per sequence (tokens_per_seq = T, at most 16) run through the
// same block one after another with the state held in registers, so a short
// multi-token step costs the same state traffic as a single token; the T tokens'
// vectors are staged in shared memory up front, so the token loop waits on no
// global load.  Instances: one token (compile-time trip count), two tokens, and up to
// kMaxDecodeTokens (bf16 steps of 3..16 tokens at d = 128 take the chunk form instead).
//
// Layout of the work: one block of 256 threads per (sequence, head).  A row of
// S (dv fp32) is covered by dv/4 threads with 16-byte loads, so each warp
// instruction moves whole 512-byte rows; each thread keeps its rows (a run of
// consecutive key rows, so the per-row decay, k and q come as 16-byte shared
// broadcasts) in registers between the read and the write, so S crosses HBM
// exactly twice.
// The two column reductions are done per thread over its rows, then across
// row groups through shared memory.  Loads and stores use the streaming cache
// hints (each byte is touched once).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_as(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_as(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// MAXT: the largest T the instance takes (1 for the single-token step, whose shared
// memory then stays small, or kMaxDecodeTokens).
template <int DK, int DV, typename Tin, int MAXT>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
              const float* __restrict__ log_alpha, const Tin* __restrict__ beta,
              float* __restrict__ S, Tin* __restrict__ out, int H, int T,
              const Tin* __restrict__ gate, const float* __restrict__ norm_w, float norm_eps,
              unsigned int* status) {
    constexpr int LANES = DV / 4;          // threads per row (float4 each)
    constexpr int RG = kThreads / LANES;   // row groups
    constexpr int RPT = DK / RG;           // rows per thread
    constexpr int kWarps = kThreads / 32;
    static_assert(RPT * RG == DK && RPT % 4 == 0, "row split in groups of four rows");

    const size_t p = blockIdx.x;           // (sequence, head) pair
    const size_t n = p / H, h = p % H;
    const int c4 = threadIdx.x % LANES;
    const int g = threadIdx.x / LANES;
    float4* Sp = reinterpret_cast<float4*>(S + p * DK * DV);

    // Issue the whole state read first so it overlaps the small loads.
    (void)status;                          // read by the index checks of bounds-checked builds
    const int64_t n_state4 = (int64_t)gridDim.x * DK * DV / 4;   // float4s of S over all pairs
    (void)n_state4;
    float4 s[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int64_t i4 = (int64_t)p * DK * DV / 4 + (int64_t)(g * RPT + m) * LANES + c4;
        (void)i4;
        s[m] = KDA_INDEX_OK(i4, n_state4, status) ? __ldcs(Sp + (size_t)(g * RPT + m) * LANES + c4)
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // The vectors of all T tokens of this sequence (rows n*T .. n*T+T-1) are staged in
    // shared memory once, next to the state read, so the token loop below waits on no
    // global load; the state stays in registers and crosses HBM once in each direction.
    // (dl, red_r and red_y are accessed as float4: every array is 16-byte aligned, whatever
    // the sizes of the ones before it)
    __shared__ __align__(16) float ks[MAXT][DK];
    __shared__ __align__(16) float qs[MAXT][DK];
    __shared__ __align__(16) float al[MAXT][DK];
    __shared__ __align__(16) float vs[MAXT][DV];
    __shared__ __align__(16) float bt[MAXT];
    __shared__ __align__(16) float kq[MAXT];
    __shared__ __align__(16) float dl[DV];
    __shared__ __align__(16) float red_r[RG][DV];
    __shared__ __align__(16) float red_y[RG][DV];
    __shared__ __align__(16) float red_n[DV / 32];
    if (MAXT == 1) T = 1;                   // a compile-time trip count for the single-token step
    const size_t row0 = n * (size_t)T * H + h;         // row of token 0; token t is row0 + t * H
    const int64_t n_rows = (int64_t)gridDim.x * T;     // rows of q, k, v, out: num_seqs x T x H
    (void)n_rows;
    for (int i = threadIdx.x; i < T * DK; i += kThreads) {
        const int tok = i / DK, c = i % DK;
        const size_t e = (row0 + (size_t)tok * H) * DK + c;
        const bool ok = KDA_INDEX_OK(e, n_rows * DK, status);
        ks[tok][c] = ok ? to_f32(k[e]) : 0.f;
        qs[tok][c] = ok ? to_f32(q[e]) : 0.f;
        al[tok][c] = ok ? expf(log_alpha[e]) : 1.f;
    }
    for (int i = threadIdx.x; i < T * DV; i += kThreads) {
        const int tok = i / DV, j = i % DV;
        const size_t e = (row0 + (size_t)tok * H) * DV + j;
        vs[tok][j] = KDA_INDEX_OK(e, n_rows * DV, status) ? to_f32(v[e]) : 0.f;
    }
    if (threadIdx.x < T) {
        const size_t e = row0 + (size_t)threadIdx.x * H;
        bt[threadIdx.x] = KDA_INDEX_OK(e, n_rows, status) ? to_f32(beta[e]) : 0.f;
    }
    __syncthreads();
    {                                       // k . q of every token, one warp per token
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int tok = w; tok < T; tok += kWarps) {
            float acc = 0.f;
            for (int i = lane; i < DK; i += 32) acc = fmaf(ks[tok][i], qs[tok][i], acc);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) kq[tok] = acc;
        }
    }                                       // (read after the first barrier of the token loop)

    for (int tok = 0; tok < T; ++tok) {
        const size_t row = row0 + (size_t)tok * H;
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f), y = r;
#pragma unroll
        for (int m = 0; m < RPT; m += 4) {         // a warp shares its rows: 16-byte broadcasts
            const int i = g * RPT + m;
            const float4 a4 = *reinterpret_cast<const float4*>(&al[tok][i]);
            const float4 k4 = *reinterpret_cast<const float4*>(&ks[tok][i]);
            const float4 q4 = *reinterpret_cast<const float4*>(&qs[tok][i]);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w},
                        qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float4& e = s[m + u];
                e.x *= av[u]; e.y *= av[u]; e.z *= av[u]; e.w *= av[u];
                r.x = fmaf(e.x, kv[u], r.x); r.y = fmaf(e.y, kv[u], r.y);
                r.z = fmaf(e.z, kv[u], r.z); r.w = fmaf(e.w, kv[u], r.w);
                y.x = fmaf(e.x, qv[u], y.x); y.y = fmaf(e.y, qv[u], y.y);
                y.z = fmaf(e.z, qv[u], y.z); y.w = fmaf(e.w, qv[u], y.w);
            }
        }
        // (every thread read the previous token's partial sums before that token's second
        // barrier, so they can be overwritten now)
        *reinterpret_cast<float4*>(&red_r[g][4 * c4]) = r;
        *reinterpret_cast<float4*>(&red_y[g][4 * c4]) = y;
        __syncthreads();

        static_assert(DV <= kThreads, "one output channel per thread");
        const int j = threadIdx.x;
        float oj = 0.f;
        if (j < DV) {
            float rj = 0.f, yj = 0.f;
#pragma unroll
            for (int gg = 0; gg < RG; ++gg) { rj += red_r[gg][j]; yj += red_y[gg][j]; }
            const float d = bt[tok] * (vs[tok][j] - rj);
            dl[j] = d;
            oj = fmaf(kq[tok], d, yj);
            if (!gate && KDA_INDEX_OK(row * DV + j, n_rows * DV, status)) store_as(&out[row * DV + j], oj);
        }
        if (gate) {   // gated output: RMSNorm over the DV channels (warps 0 .. DV/32-1) x weight x sigmoid(gate)
            float ss = oj * oj;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if ((j & 31) == 0 && j < DV) red_n[j >> 5] = ss;
            __syncthreads();
            if (j < DV) {
                float tot = 0.f;
#pragma unroll
                for (int w = 0; w < DV / 32; ++w) tot += red_n[w];
                const float rn = rsqrtf(tot * (1.f / DV) + norm_eps);
                if (KDA_INDEX_OK(row * DV + j, n_rows * DV, status)) {
                    const float gv = to_f32(gate[row * DV + j]);
                    store_as(&out[row * DV + j], oj * rn * norm_w[j] / (1.f + __expf(-gv)));
                }
            }
        }
        __syncthreads();

        const float4 d4 = *reinterpret_cast<const float4*>(&dl[4 * c4]);
#pragma unroll
        for (int m = 0; m < RPT; m += 4) {
            const float4 k4 = *reinterpret_cast<const float4*>(&ks[tok][g * RPT + m]);
            const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float4& e = s[m + u];
                e.x = fmaf(kv[u], d4.x, e.x); e.y = fmaf(kv[u], d4.y, e.y);
                e.z = fmaf(kv[u], d4.z, e.z); e.w = fmaf(kv[u], d4.w, e.w);
            }
        }
        // the next token's dl and red_n are written only after its first barrier, which every
        // thread reaches after this update
    }
#pragma unroll
    for (int m = 0; m < RPT; ++m)
        if (KDA_INDEX_OK((int64_t)p * DK * DV / 4 + (int64_t)(g * RPT + m) * LANES + c4, n_state4, status))
            __stcs(Sp + (size_t)(g * RPT + m) * LANES + c4, s[m]);
}

template <int DK, int DV, int MAXT>
cudaError_t launch_dims_t(const DecodeArgs& a, cudaStream_t st) {
    const unsigned blocks = (unsigned)((size_t)a.num_seqs * a.H);
    if (a.dtype == DType::F32) {
        decode_kernel<DK, DV, float, MAXT><<<blocks, kThreads, 0, st>>>(
            static_cast<const float*>(a.q), static_cast<const float*>(a.k),
            static_cast<const float*>(a.v), a.log_alpha, static_cast<const float*>(a.beta),
            a.state, static_cast<float*>(a.out), a.H, a.tokens_per_seq, static_cast<const float*>(a.gate),
            a.norm_w, a.norm_eps, a.status);
    } else {
        decode_kernel<DK, DV, __nv_bfloat16, MAXT><<<blocks, kThreads, 0, st>>>(
            static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
            static_cast<const __nv_bfloat16*>(a.v), a.log_alpha,
            static_cast<const __nv_bfloat16*>(a.beta), a.state, static_cast<__nv_bfloat16*>(a.out), a.H,
            a.tokens_per_seq, static_cast<const __nv_bfloat16*>(a.gate), a.norm_w, a.norm_eps, a.status);
    }
    return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t launch_dims(const DecodeArgs& a, cudaStream_t st) {
    if (a.tokens_per_seq < 1 || a.tokens_per_seq > kMaxDecodeTokens) return cudaErrorInvalidValue;
    if (a.tokens_per_seq == 1) return launch_dims_t<DK, DV, 1>(a, st);
    return a.tokens_per_seq == 2 ? launch_dims_t<DK, DV, 2>(a, st) : launch_dims_t<DK, DV, kMaxDecodeTokens>(a, st);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
    if (a.num_seqs == 0) return cudaSuccess;
    if (decode_chunk_supported(a)) return launch_decode_chunk(a, st);
    if (a.dk == 128 && a.dv == 128) return launch_dims<128, 128>(a, st);
    if (a.dk == 128 && a.dv == 64) return launch_dims<128, 64>(a, st);
    if (a.dk == 64 && a.dv == 128) return launch_dims<64, 128>(a, st);
    return launch_dims<64, 64>(a, st);
}

}  // namespace kda
