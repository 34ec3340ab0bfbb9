// kda_api.cu -- the extern "C" boundary of libkda (declared in include/kda.h).
//
// Validates every argument on the host before any CUDA call, picks the kernel
// (chunkwise tensor-core prefill for bf16 with dk = dv = 128, the fp32
// recurrent kernel otherwise) and enqueues it on the caller's stream.  Nothing
// is allocated; the only library state is one device status word that the
// tensor-core kernel sets if one of its bounded waits gives up.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "kda.h"
#include "kda_internal.h"
#include "sm103_primitives.cuh"

// Device status word; bit kda::kStatusTimeout is set by a kernel whose bounded
// wait ran out.  Read and cleared by kda_device_status.
__device__ unsigned int g_kda_status_word;

namespace {

constexpr int kMaxDevices = 64;
unsigned int* g_status_ptr[kMaxDevices] = {};

// Address of the status word on the current device (looked up once per
// device with that device current; cudaGetSymbolAddress does not allocate).
unsigned int* status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kda_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned int*>(p);
    }
    return g_status_ptr[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// One thread waits, with the library's bounded wait, on an mbarrier that nothing
// arrives on; when the wait gives up it records the timeout as every kernel does.
__global__ void selftest_timeout_kernel(unsigned int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        kda::sm103::mbar_init(&bar, 1);
        kda::sm103::fence_mbar_init();
        if (!kda::sm103::mbar_wait_bounded(&bar, 0, limit_ns)) atomicOr(status, kda::kStatusTimeout);
    }
}

// Clears the given bits of the status word and nothing else: a bit that a kernel on
// another stream sets between the host's read and this clear is kept for the next read.
__global__ void status_clear_kernel(unsigned int* status, unsigned int bits) {
    atomicAnd(status, ~bits);
}

bool env_flag(const char* name) {
    const char* v = getenv(name);
    return v && v[0] && strcmp(v, "0") != 0;
}

// Common shape checks.  Returns KDA_OK or the error to report.
kda_status check_shape(const kda_shape* s) {
    if (!s) return KDA_ERR_INVALID_ARG;
    if (s->num_seqs < 0 || s->total_tokens < 0 || s->H <= 0 || s->dk <= 0 || s->dv <= 0)
        return KDA_ERR_INVALID_ARG;
    if (s->dtype != KDA_BF16 && s->dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
    if ((s->dk != 64 && s->dk != 128) || (s->dv != 64 && s->dv != 128)) return KDA_ERR_UNSUPPORTED;
    if (s->H > 65535) return KDA_ERR_UNSUPPORTED;   // grid.y
    if ((int64_t)s->num_seqs * s->H > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

kda_status check_tensor_ptrs(const kda_shape* s, const void* q, const void* k, const void* v,
                             const float* log_alpha, const void* beta, const void* out) {
    if (!q || !k || !v || !log_alpha || !beta || !out) return KDA_ERR_INVALID_ARG;
    const size_t esz = s->dtype == KDA_BF16 ? 2 : 4;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        !aligned(log_alpha, 16) || !aligned(beta, esz))
        return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

// Gated-output arguments: gate [T, H, dv] like out, weight [dv] fp32, eps finite and > 0
// (a zero eps would turn an all-zero output row into 0 / 0).
kda_status check_gate(const kda_shape* s, const void* gate, const float* norm_w, float eps) {
    if (!gate || !norm_w) return KDA_ERR_INVALID_ARG;
    if (!(eps > 0.f) || !(eps < INFINITY)) return KDA_ERR_INVALID_ARG;
    if (!aligned(gate, 16) || !aligned(norm_w, 4)) return KDA_ERR_UNSUPPORTED;
    (void)s;
    return KDA_OK;
}

kda_status finish(cudaError_t e, cudaStream_t st) {
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if (env_flag("KDA_DEBUG_SYNC")) return kda_device_status(st);
    return KDA_OK;
}

}  // namespace

unsigned int* kda::device_status_word() { return status_word(); }

extern "C" {

kda_status kda_check_cu_seqlens(const int32_t* cu, int32_t num_seqs, int64_t total_tokens) {
    if (!cu || num_seqs < 0 || total_tokens < 0) return KDA_ERR_INVALID_ARG;
    if (cu[0] != 0) return KDA_ERR_INVALID_ARG;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu[n + 1] < cu[n]) return KDA_ERR_INVALID_ARG;
    if ((int64_t)cu[num_seqs] != total_tokens) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

}  // extern "C"

namespace {
kda_status prefill_impl(const kda_shape* shape, const void* q, const void* k, const void* v,
                        const float* log_alpha, const void* beta, const float* initial_state,
                        const int32_t* cu_seqlens, void* out, float* final_state,
                        const int32_t* ckpt_cu, const int32_t* ckpt_pos, float* ckpt_states,
                        kda_stream_t stream, const void* gate = nullptr, const float* norm_w = nullptr,
                        float norm_eps = 0.f) {
    kda_status st = check_shape(shape);
    if (st != KDA_OK) return st;
    if (shape->total_tokens > 0 && shape->num_seqs == 0) return KDA_ERR_INVALID_ARG;
    if (shape->total_tokens > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (!cu_seqlens && shape->num_seqs > 0 && shape->total_tokens % shape->num_seqs != 0)
        return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && !aligned(cu_seqlens, 4)) return KDA_ERR_UNSUPPORTED;
    if (shape->total_tokens > 0) {
        st = check_tensor_ptrs(shape, q, k, v, log_alpha, beta, out);
        if (st != KDA_OK) return st;
    }
    if ((initial_state && !aligned(initial_state, 16)) || (final_state && !aligned(final_state, 16)))
        return KDA_ERR_UNSUPPORTED;
    if (shape->num_seqs == 0) return KDA_OK;

    unsigned int* status = status_word();
    if (!status) return KDA_ERR_CUDA;
    kda::PrefillArgs a{q, k, v, log_alpha, beta, initial_state, cu_seqlens, out, final_state,
                       shape->total_tokens, shape->num_seqs, shape->H, shape->dk, shape->dv,
                       shape->dtype == KDA_BF16 ? kda::DType::BF16 : kda::DType::F32, status,
                       ckpt_cu, ckpt_pos, ckpt_states, gate, norm_w, norm_eps};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const char* force = getenv("KDA_PREFILL_IMPL");
    const bool want_recurrent = force && strcmp(force, "recurrent") == 0;
    cudaError_t e;
    if (!want_recurrent && kda::chunk_tc_supported(a))
        e = kda::launch_chunk_tc_prefill(a, s);
    else
        e = kda::launch_recurrent_prefill(a, s);
    if (e == cudaSuccess && gate)                          // gated output: one row pass over out
        e = kda::launch_gated_norm(out, gate, norm_w, norm_eps, shape->total_tokens * shape->H,
                                   shape->dv, a.dtype, s, a.status);
    return finish(e, s);
}
}  // namespace

extern "C" {

kda_status kda_prefill(const kda_shape* shape, const void* q, const void* k, const void* v,
                       const float* log_alpha, const void* beta, const float* initial_state,
                       const int32_t* cu_seqlens, void* out, float* final_state,
                       kda_stream_t stream) {
    return prefill_impl(shape, q, k, v, log_alpha, beta, initial_state, cu_seqlens, out, final_state,
                        nullptr, nullptr, nullptr, stream);
}

kda_status kda_prefill_checkpointed(const kda_shape* shape, const void* q, const void* k,
                                    const void* v, const float* log_alpha, const void* beta,
                                    const float* initial_state, const int32_t* cu_seqlens,
                                    void* out, float* final_state, const int32_t* ckpt_cu,
                                    const int32_t* ckpt_pos, float* ckpt_states,
                                    kda_stream_t stream) {
    if (!ckpt_cu || !ckpt_pos || !ckpt_states) return KDA_ERR_INVALID_ARG;
    if (!aligned(ckpt_cu, 4) || !aligned(ckpt_pos, 4) || !aligned(ckpt_states, 16))
        return KDA_ERR_UNSUPPORTED;
    return prefill_impl(shape, q, k, v, log_alpha, beta, initial_state, cu_seqlens, out, final_state,
                        ckpt_cu, ckpt_pos, ckpt_states, stream);
}

kda_status kda_prefill_gated(const kda_shape* shape, const void* q, const void* k, const void* v,
                             const float* log_alpha, const void* beta, const float* initial_state,
                             const int32_t* cu_seqlens, const void* gate, const float* norm_weight,
                             float norm_eps, void* out, float* final_state, kda_stream_t stream) {
    if (shape && shape->total_tokens > 0) {
        const kda_status st = check_gate(shape, gate, norm_weight, norm_eps);
        if (st != KDA_OK) return st;
    }
    return prefill_impl(shape, q, k, v, log_alpha, beta, initial_state, cu_seqlens, out, final_state,
                        nullptr, nullptr, nullptr, stream, gate, norm_weight, norm_eps);
}

kda_status kda_prefill_split_workspace_size(const kda_shape* shape, size_t* bytes) {
    if (!bytes) return KDA_ERR_INVALID_ARG;
    *bytes = 0;
    const kda_status st = check_shape(shape);
    if (st != KDA_OK) return st;
    if (shape->total_tokens > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    *bytes = kda::split_workspace_bytes(shape->total_tokens, shape->num_seqs, shape->H);
    return KDA_OK;
}

kda_status kda_prefill_split(const kda_shape* shape, const void* q, const void* k, const void* v,
                             const float* log_alpha, const void* beta, const float* initial_state,
                             const int32_t* cu_seqlens, void* out, float* final_state, void* workspace,
                             size_t workspace_bytes, kda_stream_t stream) {
    kda_status st = check_shape(shape);
    if (st != KDA_OK) return st;
    if (shape->total_tokens > 0 && shape->num_seqs == 0) return KDA_ERR_INVALID_ARG;
    if (shape->total_tokens > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (!cu_seqlens && shape->num_seqs > 0 && shape->total_tokens % shape->num_seqs != 0)
        return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && !aligned(cu_seqlens, 4)) return KDA_ERR_UNSUPPORTED;
    if (shape->total_tokens > 0) {
        st = check_tensor_ptrs(shape, q, k, v, log_alpha, beta, out);
        if (st != KDA_OK) return st;
    }
    if ((initial_state && !aligned(initial_state, 16)) || (final_state && !aligned(final_state, 16)))
        return KDA_ERR_UNSUPPORTED;
    const bool split_shape = shape->dtype == KDA_BF16 && shape->dk == 128 && shape->dv == 128;
    if (split_shape && shape->total_tokens > 0) {
        if (!workspace) return KDA_ERR_INVALID_ARG;
        if (!aligned(workspace, 256)) return KDA_ERR_UNSUPPORTED;
        if (workspace_bytes < kda::split_workspace_bytes(shape->total_tokens, shape->num_seqs, shape->H))
            return KDA_ERR_INVALID_ARG;
    }
    if (shape->num_seqs == 0) return KDA_OK;
    unsigned int* status = status_word();
    if (!status) return KDA_ERR_CUDA;
    kda::PrefillArgs a{q, k, v, log_alpha, beta, initial_state, cu_seqlens, out, final_state,
                       shape->total_tokens, shape->num_seqs, shape->H, shape->dk, shape->dv,
                       shape->dtype == KDA_BF16 ? kda::DType::BF16 : kda::DType::F32, status};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!split_shape || !kda::split_supported(a)) {   // the shapes the split kernels do not take
        const cudaError_t e = kda::chunk_tc_supported(a) ? kda::launch_chunk_tc_prefill(a, s)
                                                         : kda::launch_recurrent_prefill(a, s);
        return finish(e, s);
    }
    return finish(kda::launch_split_prefill(a, workspace, s), s);
}

kda_status kda_check_checkpoints(const int32_t* cu, int32_t num_seqs, int64_t total_tokens,
                                 const int32_t* ckpt_cu, const int32_t* ckpt_pos) {
    if (kda_check_cu_seqlens(cu, num_seqs, total_tokens) != KDA_OK) return KDA_ERR_INVALID_ARG;
    if (!ckpt_cu || (ckpt_cu[num_seqs] > 0 && !ckpt_pos) || ckpt_cu[0] != 0) return KDA_ERR_INVALID_ARG;
    for (int32_t n = 0; n < num_seqs; ++n) {
        if (ckpt_cu[n + 1] < ckpt_cu[n]) return KDA_ERR_INVALID_ARG;
        const int64_t len = (int64_t)cu[n + 1] - cu[n];
        int64_t prev = 0;
        for (int32_t c = ckpt_cu[n]; c < ckpt_cu[n + 1]; ++c) {
            const int64_t p = ckpt_pos[c];
            if (p <= prev || p > len || (p % 64 != 0 && p != len)) return KDA_ERR_INVALID_ARG;
            prev = p;
        }
    }
    return KDA_OK;
}

}  // extern "C"

namespace {
kda_status decode_impl(const kda_shape* shape, const void* q, const void* k, const void* v,
                       const float* log_alpha, const void* beta, float* state_inout, void* out,
                       kda_stream_t stream, const void* gate, const float* norm_w, float norm_eps) {
    kda_status st = check_shape(shape);
    if (st != KDA_OK) return st;
    if (shape->num_seqs == 0) return shape->total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (shape->total_tokens <= 0 || shape->total_tokens % shape->num_seqs != 0) return KDA_ERR_INVALID_ARG;
    const int64_t tps = shape->total_tokens / shape->num_seqs;
    if (tps > kda::kMaxDecodeTokens) return KDA_ERR_UNSUPPORTED;
    if (!state_inout) return KDA_ERR_INVALID_ARG;
    st = check_tensor_ptrs(shape, q, k, v, log_alpha, beta, out);
    if (st != KDA_OK) return st;
    if (!aligned(state_inout, 16)) return KDA_ERR_UNSUPPORTED;
    kda::DecodeArgs a{q, k, v, log_alpha, beta, state_inout, out, shape->num_seqs, (int32_t)tps, shape->H,
                      shape->dk, shape->dv,
                      shape->dtype == KDA_BF16 ? kda::DType::BF16 : kda::DType::F32, gate, norm_w, norm_eps};
    a.status = status_word();
    if (!a.status) return KDA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return finish(kda::launch_decode(a, s), s);
}
}  // namespace

extern "C" {

kda_status kda_decode_step(const kda_shape* shape, const void* q, const void* k, const void* v,
                           const float* log_alpha, const void* beta, float* state_inout,
                           void* out, kda_stream_t stream) {
    return decode_impl(shape, q, k, v, log_alpha, beta, state_inout, out, stream, nullptr, nullptr, 0.f);
}

kda_status kda_decode_step_gated(const kda_shape* shape, const void* q, const void* k, const void* v,
                                 const float* log_alpha, const void* beta, const void* gate,
                                 const float* norm_weight, float norm_eps, float* state_inout, void* out,
                                 kda_stream_t stream) {
    if (shape && shape->total_tokens > 0) {
        const kda_status st = check_gate(shape, gate, norm_weight, norm_eps);
        if (st != KDA_OK) return st;
    }
    return decode_impl(shape, q, k, v, log_alpha, beta, state_inout, out, stream, gate, norm_weight, norm_eps);
}

kda_status kda_frontend(const kda_shape* shape, int32_t conv_width, float eps, const void* q_raw,
                        const void* k_raw, const void* v_raw, const float* a_raw, const void* b_raw,
                        const float* conv_q, const float* conv_k, const float* conv_v,
                        const int32_t* cu_seqlens, void* q, void* k, void* v, float* log_alpha,
                        void* beta, kda_stream_t stream) {
    kda_status st = check_shape(shape);
    if (st != KDA_OK) return st;
    if (shape->total_tokens > 0 && shape->num_seqs == 0) return KDA_ERR_INVALID_ARG;
    if (shape->total_tokens > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (!cu_seqlens && shape->num_seqs > 0 && shape->total_tokens % shape->num_seqs != 0)
        return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && !aligned(cu_seqlens, 4)) return KDA_ERR_UNSUPPORTED;
    if (conv_width < 1 || conv_width > 4) return KDA_ERR_UNSUPPORTED;
    if (!(eps > 0.f) || !(eps < INFINITY)) return KDA_ERR_INVALID_ARG;   // an all-zero row needs eps > 0
    if (shape->total_tokens == 0) return KDA_OK;
    // the raw inputs and the outputs follow kda_prefill's pointer rules
    st = check_tensor_ptrs(shape, q_raw, k_raw, v_raw, a_raw, b_raw, q);
    if (st != KDA_OK) return st;
    st = check_tensor_ptrs(shape, q, k, v, log_alpha, beta, v);
    if (st != KDA_OK) return st;
    if (!conv_q || !conv_k || !conv_v) return KDA_ERR_INVALID_ARG;
    if (!aligned(conv_q, 4) || !aligned(conv_k, 4) || !aligned(conv_v, 4)) return KDA_ERR_UNSUPPORTED;
    kda::FrontendArgs a{q_raw, k_raw, v_raw, conv_q, conv_k, conv_v, a_raw, b_raw, cu_seqlens,
                        q, k, v, log_alpha, beta, shape->total_tokens, shape->num_seqs, shape->H,
                        shape->dk, shape->dv, conv_width, eps,
                        shape->dtype == KDA_BF16 ? kda::DType::BF16 : kda::DType::F32};
    a.status = status_word();
    if (!a.status) return KDA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return finish(kda::launch_frontend(a, s), s);
}

kda_status kda_prefill_frontend(const kda_shape* shape, int32_t conv_width, float eps, const void* q_raw,
                                const void* k_raw, const void* v_raw, const float* a_raw, const void* b_raw,
                                const float* conv_q, const float* conv_k, const float* conv_v,
                                const float* initial_state, const int32_t* cu_seqlens, void* out,
                                float* final_state, kda_stream_t stream) {
    kda_status st = check_shape(shape);
    if (st != KDA_OK) return st;
    if (shape->dtype != KDA_BF16 || shape->dk != 128 || shape->dv != 128) return KDA_ERR_UNSUPPORTED;
    if (shape->total_tokens > 0 && shape->num_seqs == 0) return KDA_ERR_INVALID_ARG;
    if (shape->total_tokens > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (!cu_seqlens && shape->num_seqs > 0 && shape->total_tokens % shape->num_seqs != 0)
        return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && !aligned(cu_seqlens, 4)) return KDA_ERR_UNSUPPORTED;
    if (conv_width < 1 || conv_width > 4) return KDA_ERR_UNSUPPORTED;
    if (!(eps > 0.f) || !(eps < INFINITY)) return KDA_ERR_INVALID_ARG;
    if ((initial_state && !aligned(initial_state, 16)) || (final_state && !aligned(final_state, 16)))
        return KDA_ERR_UNSUPPORTED;
    if (shape->total_tokens > 0) {
        st = check_tensor_ptrs(shape, q_raw, k_raw, v_raw, a_raw, b_raw, out);
        if (st != KDA_OK) return st;
        if (!conv_q || !conv_k || !conv_v) return KDA_ERR_INVALID_ARG;
        if (!aligned(conv_q, 4) || !aligned(conv_k, 4) || !aligned(conv_v, 4)) return KDA_ERR_UNSUPPORTED;
    }
    if (shape->num_seqs == 0) return KDA_OK;
    unsigned int* status = status_word();
    if (!status) return KDA_ERR_CUDA;
    kda::PrefillArgs a{q_raw, k_raw, v_raw, a_raw, b_raw, initial_state, cu_seqlens, out, final_state,
                       shape->total_tokens, shape->num_seqs, shape->H, shape->dk, shape->dv, kda::DType::BF16,
                       status};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!kda::chunk_tc_supported(a)) return KDA_ERR_UNSUPPORTED;
    kda::FrontendArgs f{q_raw, k_raw, v_raw, conv_q, conv_k, conv_v, a_raw, b_raw, cu_seqlens,
                        nullptr, nullptr, nullptr, nullptr, nullptr, shape->total_tokens, shape->num_seqs,
                        shape->H, shape->dk, shape->dv, conv_width, eps, kda::DType::BF16};
    f.status = status;
    return finish(kda::launch_chunk_tc_frontend(a, f, s), s);
}

kda_status kda_selftest_timeout(uint64_t limit_ns, kda_stream_t stream) {
    if (limit_ns < 1000ull || limit_ns > 1000000000ull) return KDA_ERR_INVALID_ARG;
    unsigned int* p = status_word();
    if (!p) return KDA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    selftest_timeout_kernel<<<1, 32, 0, s>>>(p, limit_ns);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_device_status(kda_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    unsigned int* p = status_word();
    if (!p) return KDA_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (word) {                       // clear exactly the bits that were read, atomically
        status_clear_kernel<<<1, 1, 0, s>>>(p, word);
        if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    if (word & kda::kStatusTimeout) return KDA_ERR_TIMEOUT;
    return (word & kda::kStatusBounds) ? KDA_ERR_BOUNDS : KDA_OK;
}

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_BOUNDS: return "KDA_ERR_BOUNDS";
    }
    return "KDA_ERR_UNKNOWN";
}

const char* kda_version(void) { return "kda-gb300 0.1.0 sm_103a"; }

}  // extern "C"
