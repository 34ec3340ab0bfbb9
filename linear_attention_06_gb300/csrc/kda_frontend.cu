// kda_frontend.cu -- the steps of a KDA layer between its projections and the
// recurrence: causal depthwise short convolution, SiLU and L2 norm for q and k,
// convolution and SiLU for v, logsigmoid for the decay, sigmoid for beta
// ("Kimi K3 architecture: KDA, MLA and MoE", section "Scale: Total vs Active
// Parameters and Serving Economics", Visual 1, the KDA inset).
//
// Memory-bound.  A convolution warp walks a run of about 256 consecutive tokens of
// one head for one of q, k, v (bf16 rows: each half warp its own half run; the launch
// sizes the run so the grid ends just under a whole number of waves); the
// LPR lanes of a row hold CPL channels each, so every row access is one coalesced
// segment.  Raw rows are copied into shared memory eight at a time by cp.async,
// two stages in flight, so the next stage's loads overlap the current stage's
// arithmetic; the W-1 previous raw rows stay in registers as the warp advances, so
// each raw row is read once (plus W-1 halo rows per run), and the convolution
// restarts from zeros at every sequence start.  Runs of 32 tokens with one staged
// copy each measured 566 us for the bench's front end, fixed 256-token runs 468 us
// (a last wave of 32 blocks), runs sized to whole waves 454 us.
// The decay and beta gates are a separate elementwise kernel.
#include <atomic>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kRun = 256;      // tokens per warp (target; the launch rounds it to fill whole waves)
constexpr int kStageRows = 8;  // rows per cp.async stage (two stages in flight)
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
    if constexpr (sizeof(T) == 2 && CPL == 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else if constexpr (sizeof(T) == 2 && CPL == 4) {
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
    if constexpr (sizeof(T) == 2 && CPL == 8) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 v = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&v);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (sizeof(T) == 2 && CPL == 4) {
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

__device__ __forceinline__ float silu(float y) { return __fdividef(y, 1.f + __expf(-y)); }
// SiLU through one hardware tanh (y sigmoid(y) = y/2 (1 + tanh(y/2))): half the
// special-function work of silu(); its ~2^-11 relative error is below the bf16
// rounding of the outputs it is used for.
__device__ __forceinline__ float silu_tanh(float y) {
    float th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * y));
    return 0.5f * y * (1.f + th);
}
// log sigmoid(x) = min(x, 0) - log(1 + e^{-|x|}), with the fast exp and log: the absolute error
// (about 2e-7) is what the decay e^{log alpha} sees, and the accurate log1pf made this
// elementwise pass bound by issue rather than by HBM.
__device__ __forceinline__ float logsigmoid(float x) {
    return fminf(x, 0.f) - __logf(1.f + __expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

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
template <int CPL, int W, bool kFastSilu = false>
__device__ __forceinline__ void conv_step(const float (&x)[CPL], float (&hist)[W > 1 ? W - 1 : 1][CPL],
                                          const float (&w)[W][CPL], float (&y)[CPL]) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        float acc = w[W - 1][c] * x[c];
#pragma unroll
        for (int i = 0; i < W - 1; ++i) acc = fmaf(w[i][c], hist[i][c], acc);
        y[c] = kFastSilu ? silu_tanh(acc) : silu(acc);
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

// The LPR lanes of `mask` (an aligned group) hold one row between them.
template <int CPL, int LPR>
__device__ __forceinline__ void l2_normalize(float (&y)[CPL], float eps, unsigned mask) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) ss = fmaf(y[c], y[c], ss);
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(mask, ss, o);
    const float r = rsqrtf(ss + eps);
#pragma unroll
    for (int c = 0; c < CPL; ++c) y[c] *= r;
}

// Sequence bounds of token t (clamped offsets, or the equal split).
__device__ __forceinline__ void seq_of(const FrontendArgs& a, int64_t t, int64_t& bos, int64_t& eos) {
    if (a.cu_seqlens) {
        int n;
        find_seq(a.cu_seqlens, a.num_seqs, a.total_tokens, t, n, bos, eos);
    } else {
        const int64_t len = a.total_tokens / a.num_seqs;
        bos = (t / len) * len;
        eos = bos + len;
    }
}

// Asynchronous global -> shared copy of one lane's row segment (bytes = 4, 8 or 16).
template <int BYTES>
__device__ __forceinline__ void cp_async(void* dst_smem, const void* src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem));
    if constexpr (BYTES == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(d), "l"(src), "n"(BYTES) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// One of q (tensor z0 + blockIdx.z = 0), k (1) or v (2) for kRun tokens of one head
// per warp.  LPR lanes hold a row (CPL channels each); with LPR = 16 the two halves of
// a warp walk two runs of kRun / 2 tokens side by side.  A run's raw rows are copied
// into shared memory kStage at a time into two alternating buffers (every lane its own
// channels, no registers held), then convolved with the history kept in registers,
// passed through SiLU and (q, k) normalised.
template <typename T, int CPL, int W, int LPR>
__global__ void __launch_bounds__(kWarps * 32, 5) conv_kernel(FrontendArgs a, int z0, int run) {
    static_assert(LPR == 16 || LPR == 32, "a row is half a warp or a warp");
    constexpr int RPW = 32 / LPR;                                 // runs per warp
    const int kSub = run / RPW;                                   // tokens per run
    constexpr int kSeg = CPL * (int)sizeof(T);                    // bytes per lane and row
    constexpr int kRow = LPR * kSeg;                              // bytes per staged row
    constexpr int kStage = kStageRows;
    __shared__ __align__(16) uint8_t stage[kWarps][RPW][2][kStage][kRow];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / LPR, ll = lane % LPR;
    const unsigned mask = LPR == 32 ? 0xffffffffu : (0xffffu << (16 * sub));
    const int h = blockIdx.y, which = z0 + (int)blockIdx.z;
    const int64_t t_begin = ((int64_t)blockIdx.x * kWarps + warp) * run + (int64_t)sub * kSub;
    if (t_begin >= a.total_tokens) return;
    const int64_t t_end = min(t_begin + kSub, a.total_tokens);
    const int H = a.H, d = which == 2 ? a.dv : a.dk;
    const int c0 = ll * CPL;
    const T* __restrict__ src = static_cast<const T*>(which == 0 ? a.q_raw : which == 1 ? a.k_raw : a.v_raw);
    T* __restrict__ dst = static_cast<T*>(which == 0 ? a.q : which == 1 ? a.k : a.v);
    const float* __restrict__ conv = which == 0 ? a.conv_q : which == 1 ? a.conv_k : a.conv_v;
    const bool norm = which != 2;

    const int64_t n_elems = a.total_tokens * H * d;      // elements of src and dst
    (void)n_elems;                                       // read by the index checks of bounds-checked builds
    float wt[W][CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const int64_t e = ((int64_t)h * d + c0 + c) * W + i;
            wt[i][c] = KDA_INDEX_OK(e, (int64_t)H * d * W, a.status) ? conv[e] : 0.f;
        }

    int64_t bos, eos;
    seq_of(a, t_begin, bos, eos);
    constexpr int WH = W > 1 ? W - 1 : 1;
    float hist[WH][CPL];
#pragma unroll
    for (int i = 0; i < WH; ++i) {                       // raw rows t_begin-(W-1) .. t_begin-1
        const int64_t sr = t_begin - (W - 1) + i;
#pragma unroll
        for (int c = 0; c < CPL; ++c) hist[i][c] = 0.f;
        if (W > 1 && sr >= bos && KDA_INDEX_OK((sr * H + h) * d + c0 + CPL - 1, n_elems, a.status))
            load_row<T, CPL>(src + (sr * H + h) * d + c0, hist[i]);
    }
    const int64_t rstride = (int64_t)H * d;              // elements from one token's row to the next
    const T* sp = src + (t_begin * H + h) * d + c0;
    T* dp = dst + (t_begin * H + h) * d + c0;
    // stage k (rows t_begin + k kStage ...) goes to buffer k & 1; stages k and k + 1 are in flight
    // while stage k - 1 is convolved.  Each lane copies and reads back only its own bytes.
    const int nstages = (int)((t_end - t_begin + kStage - 1) / kStage);
    auto issue = [&](int k) {
        if (k < nstages) {
            const int64_t ts = t_begin + (int64_t)k * kStage;
            const int n = (int)min((int64_t)kStage, t_end - ts);
            uint8_t* buf = &stage[warp][sub][k & 1][0][ll * kSeg];
            const T* p = sp + (int64_t)k * kStage * rstride;
            for (int j = 0; j < n; ++j, p += rstride)
                if (KDA_INDEX_OK(((ts + j) * H + h) * d + c0 + CPL - 1, n_elems, a.status))
                    cp_async<kSeg>(buf + j * kRow, p);
        }
        cp_async_commit();                               // an empty group past the end keeps the count
    };
    issue(0);
    issue(1);
    for (int k = 0; k < nstages; ++k) {
        cp_async_wait<1>();                              // stage k landed (k + 1 may be in flight)
        const int64_t ts = t_begin + (int64_t)k * kStage;
        const int n = (int)min((int64_t)kStage, t_end - ts);
        const uint8_t* buf = &stage[warp][sub][k & 1][0][ll * kSeg];
#pragma unroll 4
        for (int j = 0; j < n; ++j, dp += rstride) {
            const int64_t t = ts + j;
            if (t >= eos) {                              // a new sequence starts here
                seq_of(a, t, bos, eos);
#pragma unroll
                for (int i = 0; i < WH; ++i)
#pragma unroll
                    for (int c = 0; c < CPL; ++c) hist[i][c] = 0.f;
            }
            float xr[CPL], y[CPL];
            load_row<T, CPL>(reinterpret_cast<const T*>(buf + j * kRow), xr);
            conv_step<CPL, W, sizeof(T) == 2>(xr, hist, wt, y);   // bf16 outputs: the tanh form
            if (norm) l2_normalize<CPL, LPR>(y, a.eps, mask);
            if (KDA_INDEX_OK((t * H + h) * d + c0 + CPL - 1, n_elems, a.status)) store_row<T, CPL>(dp, y);
        }
        issue(k + 2);                                    // into the buffer just read
    }
    cp_async_wait<0>();
}

// log_alpha = logsigmoid(a_raw) and beta = sigmoid(b_raw): elementwise over rows
// of dk channels (one warp per row, CPL channels per lane) and the beta column.
template <typename T, int CPL>
__global__ void __launch_bounds__(kWarps * 32) gate_kernel(FrontendArgs a) {
    constexpr int kRowsPerWarp = 8;
    const int lane = threadIdx.x & 31;
    const int64_t rows = a.total_tokens * a.H;
    const int64_t r0 = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * kRowsPerWarp;
    const int c0 = lane * CPL;
    float x[kRowsPerWarp][CPL];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j)
        if (r0 + j < rows && KDA_INDEX_OK((r0 + j) * a.dk + c0 + CPL - 1, rows * a.dk, a.status))
            load_row<float, CPL>(a.a_raw + (r0 + j) * a.dk + c0, x[j]);
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
        if (r0 + j >= rows) break;
        float y[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) y[c] = logsigmoid(x[j][c]);
        if (KDA_INDEX_OK((r0 + j) * a.dk + c0 + CPL - 1, rows * a.dk, a.status))
            store_row<float, CPL>(a.log_alpha + (r0 + j) * a.dk + c0, y);
    }
    if (lane < kRowsPerWarp && r0 + lane < rows && KDA_INDEX_OK(r0 + lane, rows, a.status)) {
        const T* br = static_cast<const T*>(a.b_raw);
        static_cast<T*>(a.beta)[r0 + lane] = from_f<T>(sigmoid(to_f(br[r0 + lane])));
    }
}

template <typename T, int CPL, int LPR>
cudaError_t launch_conv(const FrontendArgs& a, dim3 grid, int z0, int run, cudaStream_t s) {
    switch (a.conv_width) {
        case 1: conv_kernel<T, CPL, 1, LPR><<<grid, kWarps * 32, 0, s>>>(a, z0, run); break;
        case 2: conv_kernel<T, CPL, 2, LPR><<<grid, kWarps * 32, 0, s>>>(a, z0, run); break;
        case 3: conv_kernel<T, CPL, 3, LPR><<<grid, kWarps * 32, 0, s>>>(a, z0, run); break;
        case 4: conv_kernel<T, CPL, 4, LPR><<<grid, kWarps * 32, 0, s>>>(a, z0, run); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// A row of d channels: bf16 rows are split over half a warp (16-byte accesses), fp32 rows over
// a warp.
template <typename T>
cudaError_t launch_rows(const FrontendArgs& a, int d, dim3 grid, int z0, int run, cudaStream_t s) {
    if constexpr (sizeof(T) == 2)
        return d == 128 ? launch_conv<T, 8, 16>(a, grid, z0, run, s) : launch_conv<T, 4, 16>(a, grid, z0, run, s);
    else
        return d == 128 ? launch_conv<T, 4, 32>(a, grid, z0, run, s) : launch_conv<T, 2, 32>(a, grid, z0, run, s);
}

// Tokens per convolution warp: about kRun, rounded so that the grid ends just under a whole
// number of waves of resident blocks (a last wave of a few blocks would leave the GPU idle), in
// multiples of 2 kStageRows (whole stages for both half-warp runs).
int run_length(int64_t tokens, int tensors, int H, int resident_blocks) {
    const int64_t res_warps = (int64_t)resident_blocks * kWarps;
    const int64_t per = (int64_t)tensors * H;                     // independent (tensor, head) columns
    const int64_t want_warps = per * ((tokens + kRun - 1) / kRun);
    const int64_t waves = want_warps <= res_warps ? 1 : (want_warps + res_warps / 2) / res_warps;
    const int64_t warps_per_col = (res_warps * waves) / per;      // whole waves, split over the columns
    if (warps_per_col <= 0) return kRun;
    const int64_t step = 2 * kStageRows;
    const int64_t rl = ((tokens + warps_per_col - 1) / warps_per_col + step - 1) / step * step;
    return (int)(rl < step ? step : (rl > (1 << 20) ? (1 << 20) : rl));
}

// Resident blocks of the bf16 / fp32 d = 128 convolution instance on this device (once per device).
template <typename T>
int resident_conv_blocks() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    int per_sm = 0, sms = 0;
    constexpr int CPL = sizeof(T) == 2 ? 8 : 4, LPR = sizeof(T) == 2 ? 16 : 32;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, conv_kernel<T, CPL, 4, LPR>, kWarps * 32, 0) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || per_sm <= 0 || sms <= 0)
        return 0;
    v = per_sm * sms;
    cached[dev].store(v, std::memory_order_relaxed);
    return v;
}

template <typename T>
cudaError_t launch_t(const FrontendArgs& a, cudaStream_t s) {
    const int resident = resident_conv_blocks<T>();
    const int tensors = a.dk == a.dv ? 3 : 2;
    const int run = resident > 0 ? run_length(a.total_tokens, tensors, a.H, resident) : kRun;
    const int64_t runs = (a.total_tokens + run - 1) / run;
    const unsigned bx = (unsigned)((runs + kWarps - 1) / kWarps);
    cudaError_t e;
    if (a.dk == a.dv) {                                  // q, k, v: grid.z = 0, 1, 2
        e = launch_rows<T>(a, a.dk, dim3(bx, a.H, 3), 0, run, s);
    } else {                                             // q and k, then v with its own width
        e = launch_rows<T>(a, a.dk, dim3(bx, a.H, 2), 0, run, s);
        if (e == cudaSuccess)
            e = launch_rows<T>(a, a.dv, dim3(bx, a.H, 1), 2, run, s);
    }
    if (e != cudaSuccess) return e;
    const int64_t rows = a.total_tokens * a.H;
    const unsigned gb = (unsigned)((rows + kWarps * 8 - 1) / (kWarps * 8));
    if (a.dk == 128) gate_kernel<T, 4><<<gb, kWarps * 32, 0, s>>>(a);
    else gate_kernel<T, 2><<<gb, kWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_frontend(const FrontendArgs& a, cudaStream_t s) {
    if (a.total_tokens == 0) return cudaSuccess;
    return a.dtype == DType::BF16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace kda
