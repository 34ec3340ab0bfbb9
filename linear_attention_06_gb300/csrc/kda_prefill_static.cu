// kda_prefill_static.cu -- kda_prefill_split_static: the split prefill with its scratch
// in a fixed device array of this library instead of a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run a prefill: code
// that runs inside another framework's memory pool or under a strict budget where a
// cudaMalloc would fail or is forbidden, code whose allocation calls would synchronise or
// fragment a pool it does not own, or a caller that simply has no allocator handle.  For
// them this entry point runs the two split kernels (chunk-local records, then the state
// chain) on a scratch array that the library itself owns, a file-scope __device__ array of
// kStaticScratchBytes (64 MiB).  Every GPU that loads the library holds that array until the
// process exits, and every call shares it.
#include <atomic>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "kda.h"
#include "kda_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)KDA_PREFILL_SPLIT_STATIC_BYTES;
static_assert(kStaticScratchBytes % 256 == 0, "scratch size");

// The scratch: record mode words and chunk records of kda_prefill_split, for shapes whose
// workspace fits.  In host code this name only stands for the array; its device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_split_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once per device
// (with that device current) and cached; nullptr if the lookup fails.
void* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p) return p;
    void* q = nullptr;
    if (cudaGetSymbolAddress((void**)&q, g_split_scratch) != cudaSuccess || !q) return nullptr;
    g_scratch_addr[dev].store(q, std::memory_order_release);
    return q;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" kda_status kda_prefill_split_static(const kda_shape* shape, const void* q, const void* k,
                                               const void* v, const float* log_alpha, const void* beta,
                                               const float* initial_state, const int32_t* cu_seqlens,
                                               void* out, float* final_state, kda_stream_t stream) {
    // argument rules of kda_prefill_split, on the host, before any CUDA call
    if (!shape) return KDA_ERR_INVALID_ARG;
    if (shape->num_seqs < 0 || shape->total_tokens < 0 || shape->H <= 0 || shape->dk <= 0 || shape->dv <= 0)
        return KDA_ERR_INVALID_ARG;
    if (shape->dtype != KDA_BF16 || shape->dk != 128 || shape->dv != 128) return KDA_ERR_UNSUPPORTED;
    if (shape->H > 65535 || (int64_t)shape->num_seqs * shape->H > (int64_t)INT32_MAX ||
        shape->total_tokens > (int64_t)INT32_MAX)
        return KDA_ERR_UNSUPPORTED;
    if (shape->total_tokens > 0 && shape->num_seqs == 0) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && shape->num_seqs > 0 && shape->total_tokens % shape->num_seqs != 0)
        return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && !aligned(cu_seqlens, 4)) return KDA_ERR_UNSUPPORTED;
    if (shape->total_tokens > 0) {
        if (!q || !k || !v || !log_alpha || !beta || !out) return KDA_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
            !aligned(log_alpha, 16) || !aligned(beta, 2))
            return KDA_ERR_UNSUPPORTED;
    }
    if ((initial_state && !aligned(initial_state, 16)) || (final_state && !aligned(final_state, 16)))
        return KDA_ERR_UNSUPPORTED;
    // the one limit of this entry point: the shape's scratch must fit the fixed array (one pass
    // for every shape: the segmented run of a long sequence would create a stream and events)
    if (kda::split_workspace_bytes(shape->total_tokens, shape->num_seqs, shape->H, false) > kStaticScratchBytes)
        return KDA_ERR_UNSUPPORTED;
    if (shape->num_seqs == 0) return KDA_OK;

    void* scratch = scratch_address();
    unsigned int* status = kda::device_status_word();
    if (!scratch || !status) return KDA_ERR_CUDA;
    kda::PrefillArgs a{q, k, v, log_alpha, beta, initial_state, cu_seqlens, out, final_state,
                       shape->total_tokens, shape->num_seqs, shape->H, shape->dk, shape->dv, kda::DType::BF16,
                       status};
    if (!kda::split_supported(a)) return KDA_ERR_UNSUPPORTED;
    // Nothing in the array has to start at zero: every mode word and record the chain kernel
    // reads is written by this call's chunk-local kernel first.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return kda::launch_split_prefill(a, scratch, s, false) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
