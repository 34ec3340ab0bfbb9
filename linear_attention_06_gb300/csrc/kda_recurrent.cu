// kda_recurrent.cu -- fp32 token-by-token KDA prefill on CUDA cores.
//
// Computes, per (sequence, head), the recurrence of "Kimi K3 Architecture
// Teardown" (section "Hybrid Attention for 1M Tokens", Visual 5) in the order
// the pages give: decay each key channel, erase beta * (what the decayed
// state holds under k), write beta * k v^T, then read the updated state with q
// ("Kimi K3 Architecture: KDA, MoE, and Attention", section "Memory as a
// First-Class Problem").
//
// Design: one thread per value column j of S.  Thread j keeps column j of the
// fp32 state (dk values) in registers, so the two reductions over the key
// channel (r_j = sum_i S'_ij k_i and y_j = sum_i S'_ij q_i) stay inside the
// thread and need no shuffles.  The output uses o_j = y_j + (k.q) delta_j,
// the updated state read with q, written without a second pass.  The
// per-token vectors k, q and alpha = exp(log_alpha) are staged through a
// double-buffered shared-memory slot that the block refills one token ahead,
// so there is one barrier per token.  This path serves fp32 inputs (tolerance
// 1e-4 against the fp64 oracle) and every shape the tensor-core kernel does
// not take.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kCols = 64;   // value columns (threads) per block

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_as(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_as(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ void seq_range(const int32_t* cu, int n, int num_seqs, int64_t T,
                                          int64_t& bos, int64_t& eos) {
    if (cu) {
        int64_t b = cu[n], e = cu[n + 1];
        b = b < 0 ? 0 : (b > T ? T : b);
        e = e < 0 ? 0 : (e > T ? T : e);
        bos = b;
        eos = e < b ? b : e;
    } else {
        const int64_t len = T / num_seqs;
        bos = len * n;
        eos = bos + len;
    }
}

template <int DK, typename Tin>
__global__ void __launch_bounds__(kCols)
recurrent_prefill_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                         const Tin* __restrict__ v, const float* __restrict__ log_alpha,
                         const Tin* __restrict__ beta, const float* __restrict__ h0,
                         const int32_t* __restrict__ cu, Tin* __restrict__ out,
                         float* __restrict__ hT, int64_t T, int num_seqs, int H, int dv,
                         const int32_t* __restrict__ ck_cu, const int32_t* __restrict__ ck_pos,
                         float* __restrict__ ck_states, unsigned int* status) {
    (void)status;                          // read by the index checks of bounds-checked builds
    const int tiles = dv / kCols;
    const int n = blockIdx.x / tiles;
    const int j = (blockIdx.x % tiles) * kCols + threadIdx.x;
    const int h = blockIdx.y;
    int64_t bos, eos;
    seq_range(cu, n, num_seqs, T, bos, eos);

    __shared__ __align__(16) float ks[2][DK];
    __shared__ __align__(16) float qs[2][DK];
    __shared__ __align__(16) float as[2][DK];

    float s[DK];
    const size_t sbase = ((size_t)n * H + h) * DK * dv + j;
    const int64_t n_state = (int64_t)num_seqs * H * DK * dv, n_k = T * H * DK, n_v = T * H * dv;
    (void)n_state; (void)n_k; (void)n_v;                 // read by the index checks of bounds-checked builds
#pragma unroll
    for (int i = 0; i < DK; ++i)
        s[i] = (h0 && KDA_INDEX_OK(sbase + (size_t)i * dv, n_state, status)) ? h0[sbase + (size_t)i * dv] : 0.f;

    constexpr int PER = DK / kCols;   // vector elements each thread stages
    auto stage = [&](int64_t t, int buf) {
        const size_t base = ((size_t)t * H + h) * DK;
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const int i = threadIdx.x + m * kCols;
            const bool ok = KDA_INDEX_OK(base + i, n_k, status);
            ks[buf][i] = ok ? to_f32(k[base + i]) : 0.f;
            qs[buf][i] = ok ? to_f32(q[base + i]) : 0.f;
            as[buf][i] = ok ? expf(log_alpha[base + i]) : 1.f;
        }
    };
    if (bos < eos) stage(bos, 0);
    __syncthreads();

    // checkpoints of this sequence: the state after ck_pos[ck] tokens goes to ck_states[ck]
    int ck = 0, ck_end = 0;
    int64_t ck_next = -1;
    if (ck_states) {
        ck = ck_cu[n];
        ck_end = ck_cu[n + 1];
        ck_next = (ck < ck_end) ? ck_pos[ck] : -1;
    }
    int buf = 0;
    for (int64_t t = bos; t < eos; ++t) {
        // prefetch the next token's vectors into registers
        float pk[PER], pq[PER], pa[PER];
        const bool more = (t + 1 < eos);
        if (more) {
            const size_t base = ((size_t)(t + 1) * H + h) * DK;
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int i = threadIdx.x + m * kCols;
                const bool ok = KDA_INDEX_OK(base + i, n_k, status);
                pk[m] = ok ? to_f32(k[base + i]) : 0.f;
                pq[m] = ok ? to_f32(q[base + i]) : 0.f;
                pa[m] = ok ? log_alpha[base + i] : 0.f;
            }
        }
        const size_t th = (size_t)t * H + h;
        const float vj = KDA_INDEX_OK(th * dv + j, n_v, status) ? to_f32(v[th * dv + j]) : 0.f;
        const float b = KDA_INDEX_OK(th, T * H, status) ? to_f32(beta[th]) : 0.f;

        float r[4] = {0.f, 0.f, 0.f, 0.f}, y[4] = {0.f, 0.f, 0.f, 0.f}, kq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < DK; i += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(&as[buf][i]);
            const float4 k4 = *reinterpret_cast<const float4*>(&ks[buf][i]);
            const float4 q4 = *reinterpret_cast<const float4*>(&qs[buf][i]);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
            const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
            const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                s[i + u] *= av[u];                       // decay
                r[u] = fmaf(s[i + u], kv[u], r[u]);      // what S' holds under k
                y[u] = fmaf(s[i + u], qv[u], y[u]);      // S'^T q
                kq[u] = fmaf(kv[u], qv[u], kq[u]);
            }
        }
        const float rj = (r[0] + r[1]) + (r[2] + r[3]);
        const float yj = (y[0] + y[1]) + (y[2] + y[3]);
        const float kqs = (kq[0] + kq[1]) + (kq[2] + kq[3]);
        const float delta = b * (vj - rj);               // erase + write, same beta
#pragma unroll
        for (int i = 0; i < DK; i += 4) {
            const float4 k4 = *reinterpret_cast<const float4*>(&ks[buf][i]);
            s[i + 0] = fmaf(k4.x, delta, s[i + 0]);
            s[i + 1] = fmaf(k4.y, delta, s[i + 1]);
            s[i + 2] = fmaf(k4.z, delta, s[i + 2]);
            s[i + 3] = fmaf(k4.w, delta, s[i + 3]);
        }
        if (KDA_INDEX_OK(th * dv + j, n_v, status)) store_as(&out[th * dv + j], fmaf(kqs, delta, yj));   // read after write
        if (ck < ck_end) {                       // positions <= 0 are passed over like any other bad one
            const int64_t done = t - bos + 1;
            while (ck < ck_end && ck_next <= done) {   // positions not on a chunk end are skipped
                if (ck_next == done && (done % 64 == 0 || t + 1 == eos)) {
                    const size_t cb = ((size_t)ck * H + h) * DK * dv + j;
                    const int64_t n_ck = (int64_t)ck_cu[num_seqs] * H * DK * dv;
                    (void)n_ck;
#pragma unroll
                    for (int i = 0; i < DK; ++i)
                        if (KDA_INDEX_OK(cb + (size_t)i * dv, n_ck, status)) ck_states[cb + (size_t)i * dv] = s[i];
                }
                ++ck;
                ck_next = (ck < ck_end) ? ck_pos[ck] : -1;
            }
        }

        if (more) {
            const int nb = buf ^ 1;
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int i = threadIdx.x + m * kCols;
                ks[nb][i] = pk[m];
                qs[nb][i] = pq[m];
                as[nb][i] = expf(pa[m]);
            }
        }
        __syncthreads();
        buf ^= 1;
    }
    if (hT) {
#pragma unroll
        for (int i = 0; i < DK; ++i)
            if (KDA_INDEX_OK(sbase + (size_t)i * dv, n_state, status)) hT[sbase + (size_t)i * dv] = s[i];
    }
}

template <int DK, typename Tin>
cudaError_t launch_typed(const PrefillArgs& a, cudaStream_t st) {
    const int tiles = a.dv / kCols;
    dim3 grid((unsigned)(a.num_seqs * tiles), (unsigned)a.H);
    recurrent_prefill_kernel<DK, Tin><<<grid, kCols, 0, st>>>(
        static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v),
        a.log_alpha, static_cast<const Tin*>(a.beta), a.initial_state, a.cu_seqlens,
        static_cast<Tin*>(a.out), a.final_state, a.total_tokens, a.num_seqs, a.H, a.dv, a.ckpt_cu,
        a.ckpt_pos, a.ckpt_states, a.status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent_prefill(const PrefillArgs& a, cudaStream_t st) {
    if (a.num_seqs == 0) return cudaSuccess;
    if (a.dtype == DType::F32) {
        return a.dk == 64 ? launch_typed<64, float>(a, st) : launch_typed<128, float>(a, st);
    }
    return a.dk == 64 ? launch_typed<64, __nv_bfloat16>(a, st)
                      : launch_typed<128, __nv_bfloat16>(a, st);
}

}  // namespace kda
