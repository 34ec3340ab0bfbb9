// kda_frontend.cu -- the steps of a KDA layer between its projections and the
// recurrence: causal depthwise short convolution, SiLU and L2 norm for q and k,
// convolution and SiLU for v, logsigmoid for the decay, sigmoid for beta
// ("Kimi K3 architecture: KDA, MLA and MoE", section "Scale: Total vs Active
// Parameters and Serving Economics", Visual 1, the KDA inset).
//
// Memory-bound.  One warp walks a run of 32 consecutive tokens of one head;
// lane l holds channels [l*CPL, l*CPL + CPL) of each row, so every row access is
// one coalesced 256-byte (bf16, d = 128) segment.  The W-1 previous raw rows of
// q, k and v stay in registers as the warp advances, so each raw row is read
// once (plus W-1 halo rows per run), and the convolution restarts from zeros at
// every sequence start.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kRun = 32;       // tokens per warp
constexpr int kWarps = 4;      // warps per block

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Row segments of CPL consecutive channels as single vector accesses (the
// caller's buffers are 16-byte aligned and CPL * sizeof(T) divides 16).
template <typename T, int CPL>
__device__ __forceinline__ void load_row(const T* p, float (&x)[CPL]) {
    if constexpr (sizeof(T) == 2 && CPL == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
        x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
    } else if constexpr (sizeof(T) == 2 && CPL == 2) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
        x[0] = __uint_as_float(u << 16); x[1] = __uint_as_float(u & 0xffff0000u);
    } else if constexpr (sizeof(T) == 4 && CPL == 4) {
        const float4 f = *reinterpret_cast<const float4*>(p);
        x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    } else if constexpr (sizeof(T) == 4 && CPL == 2) {
        const float2 f = *reinterpret_cast<const float2*>(p);
        x[0] = f.x; x[1] = f.y;
    } else {
#pragma unroll
        for (int i = 0; i < CPL; ++i) x[i] = to_f(p[i]);
    }
}
template <typename T, int CPL>
__device__ __forceinline__ void store_row(T* p, const float (&x)[CPL]) {
    if constexpr (sizeof(T) == 2 && CPL == 4) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]), hi = __floats2bfloat162_rn(x[2], x[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(p) = u;
    } else if constexpr (sizeof(T) == 2 && CPL == 2) {
        __nv_bfloat162 v = __floats2bfloat162_rn(x[0], x[1]);
        *reinterpret_cast<__nv_bfloat162*>(p) = v;
    } else if constexpr (sizeof(T) == 4 && CPL == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    } else if constexpr (sizeof(T) == 4 && CPL == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    } else {
#pragma unroll
        for (int i = 0; i < CPL; ++i) p[i] = from_f<T>(x[i]);
    }
}

__device__ __forceinline__ float silu(float y) { return y / (1.f + __expf(-y)); }
__device__ __forceinline__ float logsigmoid(float x) {
    return -(fmaxf(-x, 0.f) + log1pf(__expf(-fabsf(x))));
}
__device__ __forceinline__ float sigmoid(float x) { return 1.f / (1.f + __expf(-x)); }

// Sequence containing token t: largest n with cu[n] <= t (offsets clamped into
// [0, T]); returns its start and end.
__device__ __forceinline__ void find_seq(const int32_t* cu, int N, int64_t T, int64_t t, int& n,
                                         int64_t& bos, int64_t& eos) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const int64_t c = min(max((int64_t)cu[mid], (int64_t)0), T);
        if (c <= t) lo = mid;
        else hi = mid - 1;
    }
    n = lo;
    bos = min(max((int64_t)cu[n], (int64_t)0), T);
    eos = min(max((int64_t)cu[n + 1], (int64_t)0), T);
}

// One tensor of one (token, head): convolve the current raw row with the held
// history, advance the history, apply SiLU.
template <int CPL, int W>
__device__ __forceinline__ void conv_step(const float (&x)[CPL], float (&hist)[W > 1 ? W - 1 : 1][CPL],
                                          const float (&w)[W][CPL], float (&y)[CPL]) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        float acc = w[W - 1][c] * x[c];
#pragma unroll
        for (int i = 0; i < W - 1; ++i) acc = fmaf(w[i][c], hist[i][c], acc);
        y[c] = silu(acc);
    }
#pragma unroll
    for (int i = 0; i + 1 < W - 1; ++i)
#pragma unroll
        for (int c = 0; c < CPL; ++c) hist[i][c] = hist[i + 1][c];
    if (W > 1) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) hist[W > 1 ? W - 2 : 0][c] = x[c];
    }
}

template <int CPL>
__device__ __forceinline__ void l2_normalize(float (&y)[CPL], float eps) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) ss = fmaf(y[c], y[c], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss + eps);
#pragma unroll
    for (int c = 0; c < CPL; ++c) y[c] *= r;
}

template <typename T, int CPK, int CPV, int W>
__global__ void __launch_bounds__(kWarps * 32) frontend_kernel(FrontendArgs a) {
    const int lane = threadIdx.x & 31;
    const int h = blockIdx.y;
    const int64_t t_begin = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * kRun;
    if (t_begin >= a.total_tokens) return;
    const int64_t t_end = min(t_begin + kRun, a.total_tokens);
    const int H = a.H, dk = a.dk, dv = a.dv;
    const int ck = lane * CPK, cv = lane * CPV;

    // taps of this lane's channels
    float wq[W][CPK], wk[W][CPK], wv[W][CPV];
#pragma unroll
    for (int c = 0; c < CPK; ++c)
#pragma unroll
        for (int i = 0; i < W; ++i) {
            wq[i][c] = a.conv_q[((int64_t)h * dk + ck + c) * W + i];
            wk[i][c] = a.conv_k[((int64_t)h * dk + ck + c) * W + i];
        }
#pragma unroll
    for (int c = 0; c < CPV; ++c)
#pragma unroll
        for (int i = 0; i < W; ++i) wv[i][c] = a.conv_v[((int64_t)h * dv + cv + c) * W + i];

    const T* __restrict__ qr = static_cast<const T*>(a.q_raw);
    const T* __restrict__ kr = static_cast<const T*>(a.k_raw);
    const T* __restrict__ vr = static_cast<const T*>(a.v_raw);
    const T* __restrict__ br = static_cast<const T*>(a.b_raw);
    T* __restrict__ qo = static_cast<T*>(a.q);
    T* __restrict__ ko = static_cast<T*>(a.k);
    T* __restrict__ vo = static_cast<T*>(a.v);
    T* __restrict__ bo = static_cast<T*>(a.beta);

    int n = 0;
    int64_t bos = 0, eos = a.total_tokens;
    if (a.cu_seqlens) {
        find_seq(a.cu_seqlens, a.num_seqs, a.total_tokens, t_begin, n, bos, eos);
    } else {
        const int64_t len = a.total_tokens / a.num_seqs;
        bos = (t_begin / len) * len;
        eos = bos + len;
    }

    constexpr int WH = W > 1 ? W - 1 : 1;
    float hq[WH][CPK], hk[WH][CPK], hv[WH][CPV];
#pragma unroll
    for (int i = 0; i < WH; ++i) {                       // raw rows t_begin-(W-1) .. t_begin-1
        const int64_t src = t_begin - (W - 1) + i;
        const bool in = W > 1 && src >= bos;
#pragma unroll
        for (int c = 0; c < CPK; ++c) hq[i][c] = hk[i][c] = 0.f;
#pragma unroll
        for (int c = 0; c < CPV; ++c) hv[i][c] = 0.f;
        if (in) {
            load_row<T, CPK>(qr + (src * H + h) * dk + ck, hq[i]);
            load_row<T, CPK>(kr + (src * H + h) * dk + ck, hk[i]);
            load_row<T, CPV>(vr + (src * H + h) * dv + cv, hv[i]);
        }
    }

    // software pipeline: the raw rows of token t+1 are in flight while token t is computed
    float cq[CPK], ckk[CPK], cvv[CPV], ca[CPK], cb = 0.f;
    auto fetch = [&](int64_t t, float (&xq)[CPK], float (&xk)[CPK], float (&xv)[CPV], float (&xa)[CPK], float& xb) {
        const int64_t rk = (t * H + h) * dk + ck, rv = (t * H + h) * dv + cv;
        load_row<T, CPK>(qr + rk, xq);
        load_row<T, CPK>(kr + rk, xk);
        load_row<T, CPV>(vr + rv, xv);
        load_row<float, CPK>(a.a_raw + rk, xa);
        xb = lane == 0 ? to_f(br[t * H + h]) : 0.f;
    };
    fetch(t_begin, cq, ckk, cvv, ca, cb);
    for (int64_t t = t_begin; t < t_end; ++t) {
        float nq[CPK], nk[CPK], nv[CPV], na[CPK], nb = 0.f;
        if (t + 1 < t_end) fetch(t + 1, nq, nk, nv, na, nb);
        if (t >= eos) {                                  // a new sequence starts here
            if (a.cu_seqlens) {
                find_seq(a.cu_seqlens, a.num_seqs, a.total_tokens, t, n, bos, eos);
            } else {
                bos = eos;
                eos = bos + a.total_tokens / a.num_seqs;
            }
#pragma unroll
            for (int i = 0; i < WH; ++i) {
#pragma unroll
                for (int c = 0; c < CPK; ++c) hq[i][c] = hk[i][c] = 0.f;
#pragma unroll
                for (int c = 0; c < CPV; ++c) hv[i][c] = 0.f;
            }
        }
        const int64_t rk = (t * H + h) * dk + ck, rv = (t * H + h) * dv + cv;
        float y[CPK], yv[CPV], la[CPK];
        conv_step<CPK, W>(cq, hq, wq, y);
        l2_normalize<CPK>(y, a.eps);
        store_row<T, CPK>(qo + rk, y);
        conv_step<CPK, W>(ckk, hk, wk, y);
        l2_normalize<CPK>(y, a.eps);
        store_row<T, CPK>(ko + rk, y);
        conv_step<CPV, W>(cvv, hv, wv, yv);
        store_row<T, CPV>(vo + rv, yv);
#pragma unroll
        for (int c = 0; c < CPK; ++c) la[c] = logsigmoid(ca[c]);
        store_row<float, CPK>(a.log_alpha + rk, la);
        if (lane == 0) bo[t * H + h] = from_f<T>(sigmoid(cb));
#pragma unroll
        for (int c = 0; c < CPK; ++c) { cq[c] = nq[c]; ckk[c] = nk[c]; ca[c] = na[c]; }
#pragma unroll
        for (int c = 0; c < CPV; ++c) cvv[c] = nv[c];
        cb = nb;
    }
}

template <typename T, int CPK, int CPV>
cudaError_t launch_w(const FrontendArgs& a, dim3 grid, cudaStream_t s) {
    switch (a.conv_width) {
        case 1: frontend_kernel<T, CPK, CPV, 1><<<grid, kWarps * 32, 0, s>>>(a); break;
        case 2: frontend_kernel<T, CPK, CPV, 2><<<grid, kWarps * 32, 0, s>>>(a); break;
        case 3: frontend_kernel<T, CPK, CPV, 3><<<grid, kWarps * 32, 0, s>>>(a); break;
        case 4: frontend_kernel<T, CPK, CPV, 4><<<grid, kWarps * 32, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const FrontendArgs& a, dim3 grid, cudaStream_t s) {
    if (a.dk == 128 && a.dv == 128) return launch_w<T, 4, 4>(a, grid, s);
    if (a.dk == 128 && a.dv == 64) return launch_w<T, 4, 2>(a, grid, s);
    if (a.dk == 64 && a.dv == 128) return launch_w<T, 2, 4>(a, grid, s);
    return launch_w<T, 2, 2>(a, grid, s);
}

}  // namespace

cudaError_t launch_frontend(const FrontendArgs& a, cudaStream_t s) {
    if (a.total_tokens == 0) return cudaSuccess;
    const int64_t runs = (a.total_tokens + kRun - 1) / kRun;
    const dim3 grid((unsigned)((runs + kWarps - 1) / kWarps), (unsigned)a.H);
    return a.dtype == DType::BF16 ? launch_t<__nv_bfloat16>(a, grid, s) : launch_t<float>(a, grid, s);
}

}  // namespace kda
