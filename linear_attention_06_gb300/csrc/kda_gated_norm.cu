// kda_gated_norm.cu -- the step after the KDA box in a KDA layer: an RMSNorm
// over the value channels of each (token, head), times a per-channel weight,
// times sigmoid(gate) ("Kimi K3 architecture: KDA, MLA and MoE", section
// "Scale: Total vs Active Parameters and Serving Economics", Visual 1: the KDA
// output passes a norm and is multiplied by the sigmoid gate).
//
// Prefill applies it with these row kernels, in place on `out`, after the
// recurrence: one read of o and of the gate and one write, memory-bound.  (The
// decode step applies it inside its own output store.)  Done inside the
// tensor-core prefill's output stores instead, the gate loads, the cross-warp
// sums and their barriers lengthen the output warps' per-chunk loop, which is
// on that kernel's critical path, and cost more than this pass.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kWarps = 8;
constexpr int kRows = 2;       // rows per warp, loads of both issued first

template <typename T, int CPL> struct Vec;
template <> struct Vec<__nv_bfloat16, 2> {
    static __device__ __forceinline__ void ld(const __nv_bfloat16* p, float (&x)[2]) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
        x[0] = __uint_as_float(u << 16); x[1] = __uint_as_float(u & 0xffff0000u);
    }
    static __device__ __forceinline__ void st(__nv_bfloat16* p, const float (&x)[2]) {
        *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(x[0], x[1]);
    }
};
template <> struct Vec<float, 4> {
    static __device__ __forceinline__ void ld(const float* p, float (&x)[4]) {
        const float4 f = *reinterpret_cast<const float4*>(p);
        x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    }
    static __device__ __forceinline__ void st(float* p, const float (&x)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};
template <> struct Vec<float, 2> {
    static __device__ __forceinline__ void ld(const float* p, float (&x)[2]) {
        const float2 f = *reinterpret_cast<const float2*>(p);
        x[0] = f.x; x[1] = f.y;
    }
    static __device__ __forceinline__ void st(float* p, const float (&x)[2]) {
        *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    }
};

// Lane l owns the CPL consecutive channels [l*CPL, l*CPL + CPL) of each row, so a
// row is one contiguous 32*CPL-element segment per warp instruction.
template <typename T, int CPL>
__global__ void __launch_bounds__(kWarps * 32) gated_norm_kernel(T* __restrict__ out, const T* __restrict__ gate,
                                                                 const float* __restrict__ w, float eps,
                                                                 int64_t rows, unsigned int* status) {
    (void)status;                          // read by the index checks of bounds-checked builds
    constexpr int DV = 32 * CPL;
    const int lane = threadIdx.x & 31;
    const int64_t row0 = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * kRows;
    const int c0 = lane * CPL;
    float wv[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) wv[i] = w[c0 + i];
    float x[kRows][CPL], g[kRows][CPL];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        if (row0 + r < rows && KDA_INDEX_OK((row0 + r) * DV + c0 + CPL - 1, rows * DV, status)) {
            Vec<T, CPL>::ld(out + (row0 + r) * DV + c0, x[r]);
            Vec<T, CPL>::ld(gate + (row0 + r) * DV + c0, g[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        if (row0 + r >= rows) break;
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) ss = fmaf(x[r][i], x[r][i], ss);
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
        const float rr = rsqrtf(ss * (1.f / DV) + eps);
        float y[CPL];
#pragma unroll
        for (int i = 0; i < CPL; ++i) y[i] = x[r][i] * rr * wv[i] * __fdividef(1.f, 1.f + __expf(-g[r][i]));
        if (KDA_INDEX_OK((row0 + r) * DV + c0 + CPL - 1, rows * DV, status)) Vec<T, CPL>::st(out + (row0 + r) * DV + c0, y);
    }
}

// bf16 rows of 128 channels: a row over half a warp (8 channels a lane, 16-byte accesses),
// kHalfRows rows a half warp with all their loads issued first.
constexpr int kHalfRows = 4;
__global__ void __launch_bounds__(kWarps * 32) gated_norm_bf16_128(__nv_bfloat16* __restrict__ out,
                                                                   const __nv_bfloat16* __restrict__ gate,
                                                                   const float* __restrict__ w, float eps,
                                                                   int64_t rows, unsigned int* status) {
    (void)status;
    constexpr int DV = 128;
    const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
    const unsigned mask = 0xffffu << (16 * half);
    const int64_t row0 = (((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * 2 + half) * kHalfRows;
    const int c0 = hl * 8;
    float wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) wv[i] = w[c0 + i];
    uint4 xu[kHalfRows], gu[kHalfRows];
#pragma unroll
    for (int r = 0; r < kHalfRows; ++r) {
        xu[r] = gu[r] = make_uint4(0u, 0u, 0u, 0u);
        if (row0 + r < rows && KDA_INDEX_OK((row0 + r) * DV + c0 + 7, rows * DV, status)) {
            xu[r] = *reinterpret_cast<const uint4*>(out + (row0 + r) * DV + c0);
            gu[r] = *reinterpret_cast<const uint4*>(gate + (row0 + r) * DV + c0);
        }
    }
#pragma unroll
    for (int r = 0; r < kHalfRows; ++r) {
        if (row0 + r >= rows) break;
        const uint32_t xw[4] = {xu[r].x, xu[r].y, xu[r].z, xu[r].w}, gw[4] = {gu[r].x, gu[r].y, gu[r].z, gu[r].w};
        float x[8], g[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(xw[i] << 16); x[2 * i + 1] = __uint_as_float(xw[i] & 0xffff0000u);
            g[2 * i] = __uint_as_float(gw[i] << 16); g[2 * i + 1] = __uint_as_float(gw[i] & 0xffff0000u);
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(mask, ss, o);
        const float rr = rsqrtf(ss * (1.f / DV) + eps);
        uint32_t yw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float y0 = x[2 * i] * rr * wv[2 * i] * __fdividef(1.f, 1.f + __expf(-g[2 * i]));
            const float y1 = x[2 * i + 1] * rr * wv[2 * i + 1] * __fdividef(1.f, 1.f + __expf(-g[2 * i + 1]));
            __nv_bfloat162 v = __floats2bfloat162_rn(y0, y1);
            yw[i] = *reinterpret_cast<uint32_t*>(&v);
        }
        if (KDA_INDEX_OK((row0 + r) * DV + c0 + 7, rows * DV, status))
            *reinterpret_cast<uint4*>(out + (row0 + r) * DV + c0) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
    }
}

}  // namespace

cudaError_t launch_gated_norm(void* out, const void* gate, const float* w, float eps, int64_t rows, int dv,
                              DType dt, cudaStream_t s, unsigned int* status) {
    if (rows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((rows + kWarps * kRows - 1) / (kWarps * kRows));
    if (dt == DType::BF16) {
        auto* o = static_cast<__nv_bfloat16*>(out);
        auto* g = static_cast<const __nv_bfloat16*>(gate);
        if (dv == 128) {
            const unsigned b16 = (unsigned)((rows + kWarps * 2 * kHalfRows - 1) / (kWarps * 2 * kHalfRows));
            gated_norm_bf16_128<<<b16, kWarps * 32, 0, s>>>(o, g, w, eps, rows, status);
        } else {
            gated_norm_kernel<__nv_bfloat16, 2><<<blocks, kWarps * 32, 0, s>>>(o, g, w, eps, rows, status);
        }
    } else {
        auto* o = static_cast<float*>(out);
        auto* g = static_cast<const float*>(gate);
        if (dv == 128) gated_norm_kernel<float, 4><<<blocks, kWarps * 32, 0, s>>>(o, g, w, eps, rows, status);
        else gated_norm_kernel<float, 2><<<blocks, kWarps * 32, 0, s>>>(o, g, w, eps, rows, status);
    }
    return cudaGetLastError();
}

}  // namespace kda
