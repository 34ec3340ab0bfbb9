// kda_internal.h -- launchers shared between the translation units of libkda.
// Not part of the public ABI (that is include/kda.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

enum class DType : int { BF16 = 0, F32 = 1 };

// Everything a prefill launch needs; pointers are device pointers.
struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const void* beta;
    const float* initial_state;   // may be null (zeros)
    const int32_t* cu_seqlens;    // may be null (equal split)
    void* out;
    float* final_state;           // may be null
    int64_t total_tokens;
    int32_t num_seqs;
    int32_t H, dk, dv;
    DType dtype;
    unsigned int* status;         // device status word (timeouts)
    // optional state checkpoints (all null when not requested): checkpoints
    // ckpt_cu[n] .. ckpt_cu[n+1]-1 of sequence n are saved after ckpt_pos[c]
    // tokens of that sequence into ckpt_states[c] ([H, dk, dv] fp32 each)
    const int32_t* ckpt_cu = nullptr;
    const int32_t* ckpt_pos = nullptr;
    float* ckpt_states = nullptr;
    // optional gated output: out = o / sqrt(mean_j o_j^2 + norm_eps) * norm_w * sigmoid(gate)
    // per (token, head); gate [T, H, dv] in dtype, norm_w [dv] fp32 (all null when not requested)
    const void* gate = nullptr;
    const float* norm_w = nullptr;
    float norm_eps = 0.f;
};

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const void* beta;
    float* state;
    void* out;
    int32_t num_seqs;
    int32_t tokens_per_seq;       // T >= 1: rows n*T .. n*T+T-1 belong to sequence n
    int32_t H, dk, dv;
    DType dtype;
    const void* gate = nullptr;   // optional gated output, as in PrefillArgs
    const float* norm_w = nullptr;
    float norm_eps = 0.f;
    unsigned int* status = nullptr;   // device status word (bounds-checked builds)
};
// In-place gated RMSNorm over rows of dv values (after the fp32 recurrent prefill).
cudaError_t launch_gated_norm(void* out, const void* gate, const float* w, float eps, int64_t rows, int dv,
                              DType dt, cudaStream_t s, unsigned int* status = nullptr);

// Layer front end: projections -> recurrence inputs (see kda_frontend in kda.h).
struct FrontendArgs {
    const void* q_raw;            // [T, H, dk] dtype
    const void* k_raw;            // [T, H, dk] dtype
    const void* v_raw;            // [T, H, dv] dtype
    const float* conv_q;          // [H, dk, W]
    const float* conv_k;          // [H, dk, W]
    const float* conv_v;          // [H, dv, W]
    const float* a_raw;           // [T, H, dk] fp32 decay logits
    const void* b_raw;            // [T, H] dtype beta logits
    const int32_t* cu_seqlens;    // may be null (equal split)
    void* q;                      // outputs in kda_prefill's layout
    void* k;
    void* v;
    float* log_alpha;
    void* beta;
    int64_t total_tokens;
    int32_t num_seqs;
    int32_t H, dk, dv;
    int32_t conv_width;           // 1..4
    float eps;                    // L2-norm epsilon
    DType dtype;
    unsigned int* status = nullptr;   // device status word (bounds-checked builds)
};
cudaError_t launch_frontend(const FrontendArgs& a, cudaStream_t s);
// The chunkwise tensor-core prefill reading the raw projections (q, k, v, log_alpha and
// beta of `a` point at q_raw, k_raw, v_raw, a_raw and b_raw), the front end done in place
// on each chunk's tiles before the recurrence (bf16, dk = dv = 128).
struct PrefillArgs;
cudaError_t launch_chunk_tc_frontend(const PrefillArgs& a, const FrontendArgs& f, cudaStream_t s);

// fp32 recurrent prefill (any supported dtype / head size).
cudaError_t launch_recurrent_prefill(const PrefillArgs& a, cudaStream_t s);
// Chunkwise tensor-core prefill: bf16, dk = dv = 128.
bool chunk_tc_supported(const PrefillArgs& a);
cudaError_t launch_chunk_tc_prefill(const PrefillArgs& a, cudaStream_t s);
// The same prefill split into a chunk-local kernel over every (head, chunk) and a
// state-chain kernel per (sequence, head), with per-chunk records in a caller workspace.
bool split_supported(const PrefillArgs& a);
// segments = false keeps one pass for every shape (no second stream or events: the entry
// point on the library's fixed scratch array uses it).
size_t split_workspace_bytes(int64_t total_tokens, int num_seqs, int H, bool segments = true);
cudaError_t launch_split_prefill(const PrefillArgs& a, void* workspace, cudaStream_t s, bool segments = true);
// The library's device status word on the current device (nullptr if it cannot be found).
unsigned int* device_status_word();
// One decode step of T tokens per sequence (state in place).
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
// Decode steps of 3..16 tokens per sequence at dk = dv = 128, the tokens taken as one chunk
// (kda_decode_chunk.cu); launch_decode sends those shapes there.
bool decode_chunk_supported(const DecodeArgs& a);
cudaError_t launch_decode_chunk(const DecodeArgs& a, cudaStream_t s);

// Longest run of tokens per sequence that kda_decode_step accepts.
constexpr int kMaxDecodeTokens = 16;

// Bits of the device status word.
constexpr unsigned int kStatusTimeout = 1u;
constexpr unsigned int kStatusBounds = 2u;    // bounds-checked builds: an index left its buffer

// Index check of a global-memory access computed from indices (not TMA, whose tensor
// maps bound it in hardware).  In a build with -DKDA_CHECK_BOUNDS an index outside
// [0, n) sets kStatusBounds in the status word and the access is skipped; otherwise it
// is always true and compiles away.
#ifdef KDA_CHECK_BOUNDS
__device__ __forceinline__ bool index_ok(int64_t i, int64_t n, unsigned int* status) {
    if (i >= 0 && i < n) return true;
    if (status) atomicOr(status, kStatusBounds);
    return false;
}
#define KDA_INDEX_OK(i, n, status) ::kda::index_ok((int64_t)(i), (int64_t)(n), (status))
#else
#define KDA_INDEX_OK(i, n, status) true
#endif

}  // namespace kda
