// kda_gated_norm.cu -- the step after the KDA box in a KDA layer: an RMSNorm
// over the value channels of each (token, head), times a per-channel weight,
// times sigmoid(gate) ("Kimi K3 architecture: KDA, MLA and MoE", section
// "Scale: Total vs Active Parameters and Serving Economics", Visual 1: the KDA
// output passes a norm and is multiplied by the sigmoid gate).
//
// This row kernel finishes the fp32 recurrent prefill path, whose blocks each
// own a slice of the value channels; the tensor-core prefill and the decode
// step apply the same epilogue inside their own output stores.  One warp per
// (token, head) row, in place on `out`.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float x) { *p = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename T, int CPL>
__global__ void __launch_bounds__(kWarps * 32) gated_norm_kernel(T* out, const T* gate, const float* w,
                                                                 float eps, int64_t rows) {
    const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    constexpr int DV = 32 * CPL;
    T* o = out + row * DV;
    const T* g = gate + row * DV;
    float x[CPL];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        x[i] = ld(o + lane + 32 * i);
        ss = fmaf(x[i], x[i], ss);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
    const float r = rsqrtf(ss * (1.f / DV) + eps);
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        const float gv = ld(g + c);
        st(o + c, x[i] * r * w[c] / (1.f + __expf(-gv)));
    }
}

}  // namespace

cudaError_t launch_gated_norm(void* out, const void* gate, const float* w, float eps, int64_t rows, int dv,
                              DType dt, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((rows + kWarps - 1) / kWarps);
    if (dt == DType::BF16) {
        auto* o = static_cast<__nv_bfloat16*>(out);
        auto* g = static_cast<const __nv_bfloat16*>(gate);
        if (dv == 128) gated_norm_kernel<__nv_bfloat16, 4><<<blocks, kWarps * 32, 0, s>>>(o, g, w, eps, rows);
        else gated_norm_kernel<__nv_bfloat16, 2><<<blocks, kWarps * 32, 0, s>>>(o, g, w, eps, rows);
    } else {
        auto* o = static_cast<float*>(out);
        auto* g = static_cast<const float*>(gate);
        if (dv == 128) gated_norm_kernel<float, 4><<<blocks, kWarps * 32, 0, s>>>(o, g, w, eps, rows);
        else gated_norm_kernel<float, 2><<<blocks, kWarps * 32, 0, s>>>(o, g, w, eps, rows);
    }
    return cudaGetLastError();
}

}  // namespace kda
