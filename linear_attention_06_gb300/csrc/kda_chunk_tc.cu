// kda_chunk_tc.cu -- chunkwise KDA prefill on sm_103a tensor cores (tcgen05).
//
// Scope: bf16 q, k, v, beta; fp32 log_alpha; dk = dv = 128; fp32 state.
//
// The math (one head, one chunk of C = 64 tokens r = 1..C, state S0 entering
// the chunk, a_r = log alpha_r, g_r = sum_{t<=r} a_t, G = g_C):
//
//   Unrolling S_r = Diag(alpha_r)(I - ...) gives S_r = Diag(e^{g_r}) S0 +
//   sum_{s<=r} Diag(e^{g_r-g_s}) k_s d_s^T with
//     d_r = beta_r (v_r - S0^T (e^{g_r} o k_r) - sum_{s<r} A_rs d_s),
//     A_rs = sum_c k_rc k_sc e^{g_rc - g_sc}.
//   So (I + Diag(beta) L(A)) Delta = Diag(beta)(V - (e^g o K) S0) with L the
//   strictly lower part: Delta = U - W S0 with T = (I + Diag(beta) L(A))^-1
//   Diag(beta), U = T V, W = T (e^g o K)  (the UT / WY form of the product of
//   the chunk's (I - beta k k^T) Diag(alpha) factors).  Then
//     O   = (e^g o Q) S0 + (mask_{s<=r} o P) Delta,  P_rs = sum_c q_rc k_sc e^{g_rc-g_sc}
//     S_C = Diag(e^G) S0 + ((e^{G-g}) o K)^T Delta.
//   This is an exact rewrite of the token recurrence of "Kimi K3 Architecture
//   Teardown" (section "Hybrid Attention for 1M Tokens", Visual 5: decay,
//   erase with beta, write with beta; output read after the write, as in
//   "Kimi K3 Architecture: KDA, MoE, and Attention", section "Memory as a
//   First-Class Problem").  The same section of the Teardown says K3 tiles the
//   decay so a 16-token tile stays in BF16 range on tensor cores; this kernel
//   uses its own exact scheme instead (below) and needs no floor on alpha.
//
// Decay factoring.  Everything is referred to the chunk END: with
// e_r = g_C - g_r = sum_{r<t<=C} a_t (<= 0),
//   Khat = e^{-e} o K, Qhat = e^{-e} o Q   (>= 1 in magnitude scale)
//   Kb   = e^{ e} o K                      (<= 1)
//   A = Khat Kb^T, P = Qhat Kb^T, W = (T Khat) Diag(e^G),
//   (e^g o Q) S0 = Qhat (Diag(e^G) S0).
// With Ss = Diag(e^G) S0 (the decayed state, computed once per chunk):
//   Delta = U - (T Khat) Ss,  O = Qhat Ss + (mask o P) Delta,  S_C = Ss + Kb^T Delta.
// All exponents lie in [-|G|, |G|].  A chunk is used whole only when every
// channel has |G| <= 60 (e^60 ~ 1e26, far inside the bf16 / fp32 range, and
// the factored products lose nothing).  Otherwise the chunk is split greedily
// into runs of consecutive tokens that each satisfy the bound; a single
// token always qualifies (its exponents are 0), so the kernel is exact for any
// log_alpha <= 0, including -inf.
//
// Work layout.  One CTA (128 threads = 4 warps, TMEM lanes 0..127) per
// (sequence, head); it walks the sequence's chunks in order.  TMA loads the
// next chunk's q, k, v and log_alpha tiles into the other of two shared-memory
// stages while the current chunk is processed.  Matrices that end in TMEM with
// a 128-wide dimension are computed transposed so that dimension lies on the
// 128 TMEM lanes (M = 128 everywhere):
//   AP      [Khat;Qhat](128x128) x Kb^T        -> lanes 0-63 = A rows, 64-127 = P rows
//   W'^T    Khat^T (MN-major) x T^T        -> lanes = key channel
//   U^T     V^T (MN-major) x T^T        -> lanes = value channel
//   Delta^T U^T += Ss^T(TMEM) x (-W'^T)   (A operand read from TMEM)
//   O^T     Ss^T(TMEM) x Qhat^T, += Delta^T(TMEM) x P^T
//   S^T     += Delta^T(TMEM) x Kb (MN-major)
// The state lives in TMEM as fp32 S^T (lane = value channel, column = key
// channel) for the whole sequence; a bf16 copy of Ss^T is packed into TMEM as
// the A operand of the two products that read it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "kda_internal.h"
#include "sm103_primitives.cuh"

namespace kda {
namespace {

using namespace sm103;

constexpr int C = 64;          // chunk length (tokens)
constexpr int D = 128;         // dk = dv
constexpr int kThreads = 128;
constexpr float kMaxExponent = 60.f;
constexpr uint64_t kWaitLimitNs = 4000000000ull;   // 4 s per bounded wait

// ---- dynamic shared memory layout (offsets from a 1024-byte aligned base)
// stage s (two stages): QK [k_h0 | q_h0 | k_h1 | q_h1] (8 KB each, 64 rows x
// 128 B, 128-byte swizzle), V [v_h0 | v_h1], A (log_alpha, fp32 [64][128]).
constexpr uint32_t kQK = 0, kV = 32768, kA = 49152, kStageBytes = 81920;
constexpr uint32_t kKB = 2 * kStageBytes;          // Kb  [v-style halves] 16 KB
constexpr uint32_t kTT = kKB + 16384;              // T   64 x 128 B        8 KB
constexpr uint32_t kPP = kTT + 8192;               // P   64 x 128 B        8 KB
constexpr uint32_t kWT = kPP + 8192;               // -W'^T 128 x 128 B    16 KB
constexpr uint32_t kSmemUsed = kWT + 16384;        // 212992
constexpr uint32_t kSmemDynamic = kSmemUsed + 1024;
constexpr uint32_t kNStride = 68;                  // fp32 row stride of the N matrix
constexpr uint32_t kLoadBytes = 81920;             // q, k, v, log_alpha tiles of one chunk
constexpr uint32_t kReloadBytes = 65536;           // q, k, log_alpha again (split chunks)

// ---- TMEM columns
constexpr uint32_t kTmS = 0, kTmSbf = 128, kTmAP = 192, kTmU = 256, kTmDbf = 320, kTmO = 384;
constexpr uint32_t kTmCols = 512;

struct Maps {
    CUtensorMap q, k, v, a;
};

__device__ __forceinline__ uint32_t qk_off(bool is_q, uint32_t r, uint32_t c) {
    return kQK + (c >> 6) * 16384u + (is_q ? 8192u : 0u) + sw128_offset(r, (c & 63u) * 2u);
}
__device__ __forceinline__ uint32_t half_off(uint32_t r, uint32_t c) {   // V and Kb
    return (c >> 6) * 8192u + sw128_offset(r, (c & 63u) * 2u);
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void seq_bounds(const int32_t* cu, int n, int num_seqs, int64_t T,
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

// Every thread waits (bounded); the block agrees on the outcome.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity) {
    const bool ok = mbar_wait_bounded(bar, parity, kWaitLimitNs);
    return __syncthreads_and(ok) != 0;
}

// TMA: q, k (and v) and log_alpha tiles of tokens [t0, t0+64) of head h.
__device__ __forceinline__ void issue_tile_loads(uint8_t* stage, const Maps& m, int h, int t0,
                                                 uint64_t* bar, bool with_v) {
    mbar_arrive_expect_tx(bar, with_v ? kLoadBytes : kReloadBytes);
    tma_load_3d(stage + kQK + 0, &m.k, 0, h, t0, bar);
    tma_load_3d(stage + kQK + 8192, &m.q, 0, h, t0, bar);
    tma_load_3d(stage + kQK + 16384, &m.k, 64, h, t0, bar);
    tma_load_3d(stage + kQK + 24576, &m.q, 64, h, t0, bar);
    if (with_v) {
        tma_load_3d(stage + kV, &m.v, 0, h, t0, bar);
        tma_load_3d(stage + kV + 8192, &m.v, 64, h, t0, bar);
    }
    tma_load_3d(stage + kA, &m.a, 0, h, t0, bar);
}

// Length of the next run [r0, r1) whose per-channel decay total stays within
// +-kMaxExponent (a single token is always accepted).  Thread = key channel.
__device__ int next_run(const float* A, int r0, int L) {
    const int c = threadIdx.x;
    if (r0 == 0) {
        float tot = 0.f;
        for (int r = 0; r < L; ++r) tot += A[r * D + c];
        if (!__syncthreads_or(!(fabsf(tot) <= kMaxExponent))) return L;
    }
    float acc = 0.f;
    int r1 = r0 + 1;
    for (int r = r0; r < L; ++r) {
        acc += A[r * D + c];
        if (__syncthreads_or(!(fabsf(acc) <= kMaxExponent))) {
            r1 = (r == r0) ? r0 + 1 : r;
            break;
        }
        r1 = r + 1;
    }
    return r1;
}

// Khat, Qhat (in place over k, q) and Kb for the rows [r0, r1); other rows are
// zeroed.  gam[c] = e^{G_c}, the decay of the whole run.  Thread = key channel.
__device__ void build_operands(uint8_t* sm, uint32_t stage, int r0, int r1, float* gam) {
    const int c = threadIdx.x;
    uint8_t* stg = sm + stage;
    const float* A = reinterpret_cast<const float*>(stg + kA);
    const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
    float e = 0.f;   // sum of log_alpha over the run's tokens after row r
    for (int r = C - 1; r >= 0; --r) {
        __nv_bfloat16* kp = reinterpret_cast<__nv_bfloat16*>(stg + qk_off(false, r, c));
        __nv_bfloat16* qp = reinterpret_cast<__nv_bfloat16*>(stg + qk_off(true, r, c));
        __nv_bfloat16* bp = reinterpret_cast<__nv_bfloat16*>(sm + kKB + half_off(r, c));
        if (r >= r0 && r < r1) {
            const float kv = bf2f(*kp), qv = bf2f(*qp);
            const float up = __expf(-e), dn = __expf(e);
            *kp = __float2bfloat16_rn(kv * up);
            *qp = __float2bfloat16_rn(qv * up);
            *bp = __float2bfloat16_rn(kv * dn);
            e += A[r * D + c];
        } else {
            *kp = zero;
            *qp = zero;
            *bp = zero;
        }
    }
    gam[c] = __expf(e);
}

// TMEM S^T (lane j = value channel, column c = key channel): S <- S Diag(gam)
// in fp32, and the bf16 copy of the decayed state packed as an A operand.
__device__ void decay_state(uint32_t tb, const float* gam) {
    const uint32_t lane0 = (threadIdx.x >> 5) * 32;
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
        uint32_t v0[32], v1[32], pk[32];
        tmem_ld32(tmem_addr(tb, lane0, kTmS + 64 * hf), v0);
        tmem_ld32(tmem_addr(tb, lane0, kTmS + 64 * hf + 32), v1);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            v0[i] = __float_as_uint(__uint_as_float(v0[i]) * gam[64 * hf + i]);
            v1[i] = __float_as_uint(__uint_as_float(v1[i]) * gam[64 * hf + 32 + i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            pk[i] = pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
            pk[16 + i] = pack_bf16x2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
        }
        tmem_st32(tmem_addr(tb, lane0, kTmS + 64 * hf), v0);
        tmem_st32(tmem_addr(tb, lane0, kTmS + 64 * hf + 32), v1);
        tmem_st32(tmem_addr(tb, lane0, kTmSbf + 32 * hf), pk);
    }
    tmem_wait_st();
}

// ---- MMA groups (issued by one thread) -------------------------------------
// AP = [Khat; Qhat] x Kb^T : M = 128, N = 64, K = 128 (both K-major).
__device__ __forceinline__ void mma_gram(uint32_t tb, uint32_t sQK, uint32_t sKB) {
    constexpr uint32_t id = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
    for (uint32_t ks = 0; ks < 8; ++ks) {
        const uint64_t a = smem_desc(sQK + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, kSwizzle128B);
        const uint64_t b = smem_desc(sKB + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, kSwizzle128B);
        mma_ss(tb + kTmAP, a, b, id, ks > 0);
    }
}

// W'^T = Khat^T T^T -> AP columns; U^T = V^T T^T -> U columns.  M = 128, N = 64,
// K = 64 tokens; A operands MN-major (channel halves LBO apart), B = T K-major.
__device__ __forceinline__ void mma_wu(uint32_t tb, uint32_t sQK, uint32_t sV, uint32_t sTT) {
    constexpr uint32_t id = idesc_bf16_f32(128, 64, true, false);
#pragma unroll
    for (uint32_t ks = 0; ks < 4; ++ks) {
        const uint64_t b = smem_desc(sTT + ks * 32, 16, 1024, kSwizzle128B);
        mma_ss(tb + kTmAP, smem_desc(sQK + ks * 2048, 16384, 1024, kSwizzle128B), b, id, ks > 0);
        mma_ss(tb + kTmU, smem_desc(sV + ks * 2048, 8192, 1024, kSwizzle128B), b, id, ks > 0);
    }
}

// Delta^T = U^T + Ss^T (-W'^T)  and  O^T = Ss^T Qhat^T : A = Ss^T from TMEM, K = 128.
__device__ __forceinline__ void mma_delta_out(uint32_t tb, uint32_t sWT, uint32_t sQK) {
    constexpr uint32_t idw = idesc_bf16_f32(128, 64, false, true);
    constexpr uint32_t idq = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
    for (uint32_t ks = 0; ks < 8; ++ks)
        mma_ts(tb + kTmU, tb + kTmSbf + ks * 8, smem_desc(sWT + ks * 2048, 16384, 1024, kSwizzle128B),
               idw, 1);
#pragma unroll
    for (uint32_t ks = 0; ks < 8; ++ks)
        mma_ts(tb + kTmO, tb + kTmSbf + ks * 8,
               smem_desc(sQK + 8192 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, kSwizzle128B), idq,
               ks > 0);
}

// S^T += Delta^T Kb (N = 128, Kb MN-major) and O^T += Delta^T P^T (N = 64):
// A = Delta^T from TMEM, K = 64 tokens.
__device__ __forceinline__ void mma_state_out(uint32_t tb, uint32_t sKB, uint32_t sPP) {
    constexpr uint32_t ids = idesc_bf16_f32(128, 128, false, true);
    constexpr uint32_t idp = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
    for (uint32_t ks = 0; ks < 4; ++ks)
        mma_ts(tb + kTmS, tb + kTmDbf + ks * 8, smem_desc(sKB + ks * 2048, 8192, 1024, kSwizzle128B),
               ids, 1);
#pragma unroll
    for (uint32_t ks = 0; ks < 4; ++ks)
        mma_ts(tb + kTmO, tb + kTmDbf + ks * 8, smem_desc(sPP + ks * 32, 16, 1024, kSwizzle128B), idp, 1);
}

// ---- TMEM readouts (thread = TMEM lane) --------------------------------------
__device__ __forceinline__ void ld64(uint32_t tb, uint32_t col, uint32_t (&v)[64]) {
    const uint32_t lane0 = (threadIdx.x >> 5) * 32;
    uint32_t* lo = v;
    tmem_ld32(tmem_addr(tb, lane0, col), *reinterpret_cast<uint32_t(*)[32]>(lo));
    tmem_ld32(tmem_addr(tb, lane0, col + 32), *reinterpret_cast<uint32_t(*)[32]>(lo + 32));
    tmem_wait_ld();
}

// Lanes 0-63 hold A rows r: N[r][s] = beta_r A_rs (s < r) -> fp32 matrix in the
// stage's log_alpha slot.  Lanes 64-127 hold P rows r: P_rs (s <= r) -> bf16,
// K-major operand tile PP.
__device__ void read_gram(uint32_t tb, uint8_t* stage, uint8_t* sm, const float* beta_s) {
    uint32_t v[64];
    ld64(tb, kTmAP, v);
    const int tid = threadIdx.x;
    if (tid < 64) {
        const int r = tid;
        const float b = beta_s[r];
        float* Nr = reinterpret_cast<float*>(stage + kA) + r * kNStride;
#pragma unroll
        for (int s = 0; s < 64; s += 4) {
            float4 f;
            f.x = (s + 0 < r) ? b * __uint_as_float(v[s + 0]) : 0.f;
            f.y = (s + 1 < r) ? b * __uint_as_float(v[s + 1]) : 0.f;
            f.z = (s + 2 < r) ? b * __uint_as_float(v[s + 2]) : 0.f;
            f.w = (s + 3 < r) ? b * __uint_as_float(v[s + 3]) : 0.f;
            *reinterpret_cast<float4*>(Nr + s) = f;
        }
    } else {
        const int r = tid - 64;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int s = 8 * ch + 2 * u;
                const float lo = (s <= r) ? __uint_as_float(v[s]) : 0.f;
                const float hi = (s + 1 <= r) ? __uint_as_float(v[s + 1]) : 0.f;
                w[u] = pack_bf16x2(lo, hi);
            }
            *reinterpret_cast<uint4*>(sm + kPP + sw128_offset(r, 16 * ch)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// T = (I + N)^{-1} Diag(beta) by forward substitution, one column per thread
// (threads 0..63), fp32; written as the bf16 K-major operand TT (row r).
__device__ void solve_T(const uint8_t* stage, uint8_t* sm, const float* beta_s) {
    const int j = threadIdx.x;
    const float* Nm = reinterpret_cast<const float*>(stage + kA);
    float x[64];
#pragma unroll
    for (int r = 0; r < 64; ++r) x[r] = 0.f;
#pragma unroll
    for (int r = 0; r < 64; ++r) {
        float acc = (r == j) ? 1.f : 0.f;
#pragma unroll
        for (int s = 0; s < r; s += 4) {
            const float4 n4 = *reinterpret_cast<const float4*>(Nm + r * kNStride + s);
            acc = fmaf(-n4.x, x[s + 0], acc);
            acc = fmaf(-n4.y, x[s + 1], acc);
            acc = fmaf(-n4.z, x[s + 2], acc);
            acc = fmaf(-n4.w, x[s + 3], acc);
        }
        x[r] = acc;
    }
    const float bj = beta_s[j];
#pragma unroll
    for (int r = 0; r < 64; ++r)
        *reinterpret_cast<__nv_bfloat16*>(sm + kTT + sw128_offset(r, 2 * j)) =
            __float2bfloat16_rn(x[r] * bj);
}

// Lane c holds W'^T row c (64 tokens): store -W'^T as bf16, MN-major B operand.
__device__ void read_w(uint32_t tb, uint8_t* sm) {
    uint32_t v[64];
    ld64(tb, kTmAP, v);
    const int c = threadIdx.x;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            w[u] = pack_bf16x2(-__uint_as_float(v[8 * ch + 2 * u]), -__uint_as_float(v[8 * ch + 2 * u + 1]));
        *reinterpret_cast<uint4*>(sm + kWT + sw128_offset(c, 16 * ch)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Lane j holds Delta^T row j (fp32): pack to bf16 in TMEM as an A operand.
__device__ void pack_delta(uint32_t tb) {
    uint32_t v[64], pk[32];
    ld64(tb, kTmU, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    tmem_st32(tmem_addr(tb, (threadIdx.x >> 5) * 32, kTmDbf), pk);
    tmem_wait_st();
}

// Lane j holds O^T row j: write out[t0 + r, h, j] for r in [r0, r1).
__device__ void store_out(uint32_t tb, __nv_bfloat16* out, int64_t t0, int H, int h, int r0, int r1) {
    uint32_t v[64];
    ld64(tb, kTmO, v);
    const int j = threadIdx.x;
#pragma unroll
    for (int r = 0; r < 64; ++r)
        if (r >= r0 && r < r1)
            out[((t0 + r) * H + h) * D + j] = __float2bfloat16_rn(__uint_as_float(v[r]));
}

__device__ void load_state(uint32_t tb, const float* h0, size_t base) {
    const int j = threadIdx.x;
    const uint32_t lane0 = (threadIdx.x >> 5) * 32;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            r[i] = h0 ? __float_as_uint(h0[base + (size_t)(32 * cb + i) * D + j]) : 0u;
        tmem_st32(tmem_addr(tb, lane0, kTmS + 32 * cb), r);
    }
    tmem_wait_st();
}

__device__ void store_state(uint32_t tb, float* hT, size_t base) {
    const int j = threadIdx.x;
    const uint32_t lane0 = (threadIdx.x >> 5) * 32;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tb, lane0, kTmS + 32 * cb), r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) hT[base + (size_t)(32 * cb + i) * D + j] = __uint_as_float(r[i]);
    }
}

// Make this thread's shared-memory and TMEM writes visible to the tensor core,
// then synchronise the block.
__device__ __forceinline__ void publish_to_mma() {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ Maps maps, const __nv_bfloat16* __restrict__ beta,
                const float* __restrict__ h0, const int32_t* __restrict__ cu,
                __nv_bfloat16* __restrict__ out, float* __restrict__ hT, int64_t T, int num_seqs,
                int H, unsigned int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t full_bar[2], mma_bar, reload_bar;
    __shared__ uint32_t tmem_base;
    __shared__ float beta_s[C], gam[D];

    const int tid = threadIdx.x;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    int64_t bos, eos;
    seq_bounds(cu, n, num_seqs, T, bos, eos);
    const int nchunks = (int)((eos - bos + C - 1) / C);
    const size_t sbase = ((size_t)n * H + h) * D * D;

    if (tid == 0) {
        mbar_init(&full_bar[0], 1);
        mbar_init(&full_bar[1], 1);
        mbar_init(&mma_bar, 1);
        mbar_init(&reload_bar, 1);
        fence_mbar_init();
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
        tma_prefetch_desc(&maps.a);
    }
    if ((tid >> 5) == 0) {
        tmem_alloc(&tmem_base, kTmCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;

    bool pending[2] = {false, false};
    if (tid == 0) {
        for (int c = 0; c < 2 && c < nchunks; ++c)
            issue_tile_loads(sm + c * kStageBytes, maps, h, (int)(bos + (int64_t)c * C), &full_bar[c], true);
    }
    for (int c = 0; c < 2 && c < nchunks; ++c) pending[c] = true;
    load_state(tb, h0, sbase);

    uint32_t full_ph[2] = {0u, 0u}, mma_ph = 0u, reload_ph = 0u;
    bool mma_pending = false, reload_pending = false;
    const uint32_t sQKbase = smem_u32(sm);
    const uint32_t sKB = smem_u32(sm + kKB), sTT = smem_u32(sm + kTT), sPP = smem_u32(sm + kPP),
                   sWT = smem_u32(sm + kWT);
    bool ok = true;

    for (int c = 0; c < nchunks && ok; ++c) {
        const int st = c & 1;
        uint8_t* stage = sm + st * kStageBytes;
        const uint32_t sQK = sQKbase + st * kStageBytes + kQK, sV = sQKbase + st * kStageBytes + kV;
        const int64_t t0 = bos + (int64_t)c * C;
        const int L = (int)((eos - t0) < C ? (eos - t0) : C);
        float braw = 0.f;
        if (tid < L) braw = bf2f(beta[(t0 + tid) * H + h]);

        ok = wait_all(&full_bar[st], full_ph[st]);
        if (!ok) break;
        full_ph[st] ^= 1u;
        pending[st] = false;

        for (int r0 = 0; r0 < L && ok;) {
            if (r0 > 0) {   // split chunk: restore the raw q, k, log_alpha tiles
                if (tid == 0) issue_tile_loads(stage, maps, h, (int)t0, &reload_bar, false);
                reload_pending = true;
                ok = wait_all(&reload_bar, reload_ph);
                if (!ok) break;
                reload_ph ^= 1u;
                reload_pending = false;
            }
            const int r1 = next_run(reinterpret_cast<const float*>(stage + kA), r0, L);
            if (tid < C) beta_s[tid] = (tid >= r0 && tid < r1) ? braw : 0.f;
            build_operands(sm, st * kStageBytes, r0, r1, gam);
            __syncthreads();
            decay_state(tb, gam);
            publish_to_mma();

            if (tid == 0) {
                mma_gram(tb, sQK, sKB);
                mma_commit(&mma_bar);
            }
            mma_pending = true;
            if (!(ok = wait_all(&mma_bar, mma_ph))) break;
            mma_ph ^= 1u;
            mma_pending = false;
            tc_fence_after();
            read_gram(tb, stage, sm, beta_s);
            fence_proxy_async_smem();
            __syncthreads();
            if (tid < 64) solve_T(stage, sm, beta_s);
            publish_to_mma();

            if (tid == 0) {
                mma_wu(tb, sQK, sV, sTT);
                mma_commit(&mma_bar);
            }
            mma_pending = true;
            if (!(ok = wait_all(&mma_bar, mma_ph))) break;
            mma_ph ^= 1u;
            mma_pending = false;
            tc_fence_after();
            read_w(tb, sm);
            publish_to_mma();

            if (tid == 0) {
                mma_delta_out(tb, sWT, sQK);
                mma_commit(&mma_bar);
            }
            mma_pending = true;
            if (!(ok = wait_all(&mma_bar, mma_ph))) break;
            mma_ph ^= 1u;
            mma_pending = false;
            tc_fence_after();
            pack_delta(tb);
            publish_to_mma();

            if (tid == 0) {
                mma_state_out(tb, sKB, sPP);
                mma_commit(&mma_bar);
            }
            mma_pending = true;
            if (!(ok = wait_all(&mma_bar, mma_ph))) break;
            mma_ph ^= 1u;
            mma_pending = false;
            tc_fence_after();
            store_out(tb, out, t0, H, h, r0, r1);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            r0 = r1;
        }
        if (ok && c + 2 < nchunks) {
            if (tid == 0)
                issue_tile_loads(stage, maps, h, (int)(t0 + 2 * C), &full_bar[st], true);
            pending[st] = true;
        }
    }

    if (ok) {
        if (hT) store_state(tb, hT, sbase);
    } else {
        if (tid == 0) atomicOr(status, kStatusTimeout);
        // let in-flight copies land before the block exits (bounded)
        for (int s = 0; s < 2; ++s)
            if (pending[s]) mbar_wait_bounded(&full_bar[s], full_ph[s], kWaitLimitNs);
        if (mma_pending) mbar_wait_bounded(&mma_bar, mma_ph, kWaitLimitNs);
        if (reload_pending) mbar_wait_bounded(&reload_bar, reload_ph, kWaitLimitNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if ((tid >> 5) == 0) tmem_dealloc(tb, kTmCols);
}

// ---- host side ------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// [T, H, 128] tensor, box {inner, 1, 64}.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esz, int64_t T, int H,
              uint32_t inner, CUtensorMapSwizzle sw) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)H * D * esz};
    cuuint32_t box[3] = {inner, 1, (cuuint32_t)C}, es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_supported(const PrefillArgs& a) {
    return a.dtype == DType::BF16 && a.dk == D && a.dv == D && a.total_tokens > 0 &&
           encode_fn() != nullptr;
}

cudaError_t launch_chunk_tc_prefill(const PrefillArgs& a, cudaStream_t s) {
    Maps maps;
    if (!make_map(&maps.q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&maps.k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&maps.v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&maps.a, a.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.total_tokens, a.H, 128,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemDynamic);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const unsigned blocks = (unsigned)((int64_t)a.num_seqs * a.H);
    chunk_tc_kernel<<<blocks, kThreads, kSmemDynamic, s>>>(
        maps, static_cast<const __nv_bfloat16*>(a.beta), a.initial_state, a.cu_seqlens,
        static_cast<__nv_bfloat16*>(a.out), a.final_state, a.total_tokens, a.num_seqs, a.H, a.status);
    return cudaGetLastError();
}

}  // namespace kda
