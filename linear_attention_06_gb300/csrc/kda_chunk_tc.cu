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
// The UT solve works on 16x16 blocks of the strictly lower 64x64 matrix
// N = Diag(beta) L(A) and of X = (I + N)^-1, kept in the stage's log_alpha slot
// (free by then) as the 10 lower-triangular blocks each, row stride 20 floats.
constexpr uint32_t kBlkStride = 20, kBlkBytes = 16 * kBlkStride * 4;          // 1280
constexpr uint32_t kSolveN = 0, kSolveX = 10 * kBlkBytes, kSolveY = 20 * kBlkBytes;
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
        float t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < C; ++r) t4[r & 3] += (r < L) ? A[r * D + c] : 0.f;
        const float tot = (t4[0] + t4[1]) + (t4[2] + t4[3]);
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
// The 64 log-decays are first pulled into registers and turned into suffix
// sums, so the exponentials and the tile stores carry no loop dependency.
__device__ void build_operands(uint8_t* sm, uint32_t stage, int r0, int r1, float* gam) {
    const int c = threadIdx.x;
    uint8_t* stg = sm + stage;
    const float* A = reinterpret_cast<const float*>(stg + kA);
    float e[C];
#pragma unroll
    for (int r = 0; r < C; ++r) e[r] = (r >= r0 && r < r1) ? A[r * D + c] : 0.f;
    float run = 0.f;   // sum of log_alpha over the run's tokens after row r
#pragma unroll
    for (int r = C - 1; r >= 0; --r) {
        const float ar = e[r];
        e[r] = run;
        run += ar;
    }
    gam[c] = __expf(run);
    const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
#pragma unroll
    for (int r = 0; r < C; ++r) {
        __nv_bfloat16* kp = reinterpret_cast<__nv_bfloat16*>(stg + qk_off(false, r, c));
        __nv_bfloat16* qp = reinterpret_cast<__nv_bfloat16*>(stg + qk_off(true, r, c));
        __nv_bfloat16* bp = reinterpret_cast<__nv_bfloat16*>(sm + kKB + half_off(r, c));
        if (r >= r0 && r < r1) {
            const float kv = bf2f(*kp), qv = bf2f(*qp);
            const float up = __expf(-e[r]), dn = __expf(e[r]);
            *kp = __float2bfloat16_rn(kv * up);
            *qp = __float2bfloat16_rn(qv * up);
            *bp = __float2bfloat16_rn(kv * dn);
        } else {
            *kp = zero;
            *qp = zero;
            *bp = zero;
        }
    }
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
        const int r = tid, bi = r >> 4, rr = r & 15;
        const float b = beta_s[r];
        float* Nbase = reinterpret_cast<float*>(stage + kA + kSolveN);
#pragma unroll
        for (int bj = 0; bj < 4; ++bj) {
            if (bj > bi) break;
            float* dst = Nbase + (bi * (bi + 1) / 2 + bj) * (kBlkBytes / 4) + rr * kBlkStride;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int s0 = 16 * bj + 4 * q4;
                float4 f;
                f.x = (s0 + 0 < r) ? b * __uint_as_float(v[s0 + 0]) : 0.f;
                f.y = (s0 + 1 < r) ? b * __uint_as_float(v[s0 + 1]) : 0.f;
                f.z = (s0 + 2 < r) ? b * __uint_as_float(v[s0 + 2]) : 0.f;
                f.w = (s0 + 3 < r) ? b * __uint_as_float(v[s0 + 3]) : 0.f;
                *reinterpret_cast<float4*>(dst + 4 * q4) = f;
            }
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

__device__ __forceinline__ float* blk(float* base, int i, int j) {
    return base + (i * (i + 1) / 2 + j) * (kBlkBytes / 4);
}

// One warp computes rows [rb, rb + NR) of C = sign * sum_p A_p B_p for 16x16
// blocks (NP pairs); each lane owns NR/2 consecutive columns of one row.
template <int NR, int NP>
__device__ __forceinline__ void blk_product(float* Cb, float* const (&Ab)[NP], float* const (&Bb)[NP],
                                            int rb, float sign) {
    constexpr int NC = NR / 2;                  // columns per lane
    constexpr int LPR = 16 / NC;                // lanes per row
    const int lane = threadIdx.x & 31;
    const int rr = rb + lane / LPR, c0 = (lane % LPR) * NC;
    float acc[NC];
#pragma unroll
    for (int u = 0; u < NC; ++u) acc[u] = 0.f;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        float arow[16];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const float4 a4 = *reinterpret_cast<const float4*>(Ab[p] + rr * kBlkStride + 4 * k4);
            arow[4 * k4] = a4.x; arow[4 * k4 + 1] = a4.y; arow[4 * k4 + 2] = a4.z; arow[4 * k4 + 3] = a4.w;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float* brow = Bb[p] + k * kBlkStride + c0;
#pragma unroll
            for (int u = 0; u < NC; u += 2) {
                const float2 b2 = *reinterpret_cast<const float2*>(brow + u);
                acc[u] = fmaf(arow[k], b2.x, acc[u]);
                acc[u + 1] = fmaf(arow[k], b2.y, acc[u + 1]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < NC; u += 2)
        *reinterpret_cast<float2*>(Cb + rr * kBlkStride + c0 + u) = make_float2(sign * acc[u], sign * acc[u + 1]);
}

// T = (I + N)^{-1} Diag(beta), N strictly lower (64 x 64), by 16x16 blocks:
// the four diagonal blocks D_i = (I + N_ii)^{-1} by forward substitution, then
// X_ij = -D_i sum_{k=j}^{i-1} N_ik X_kj one block sub-diagonal at a time.
// All 128 threads take part; fp32 throughout.  T goes to the bf16 K-major
// operand tile TT (row r = token, column s).
__device__ void solve_T(uint8_t* stage, uint8_t* sm, const float* beta_s) {
    float* Nb = reinterpret_cast<float*>(stage + kA + kSolveN);
    float* Xb = reinterpret_cast<float*>(stage + kA + kSolveX);
    float* Yb = reinterpret_cast<float*>(stage + kA + kSolveY);
    const int tid = threadIdx.x, w = tid >> 5;
    if (tid < 64) {                                  // diagonal blocks
        const int i = tid >> 4, jl = tid & 15;
        const float* Nii = blk(Nb, i, i);
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == jl) ? 1.f : 0.f;
#pragma unroll
            for (int q = 0; q < r; ++q) acc = fmaf(-Nii[r * kBlkStride + q], x[q], acc);
            x[r] = acc;
        }
        float* Xii = blk(Xb, i, i);
#pragma unroll
        for (int r = 0; r < 16; ++r) Xii[r * kBlkStride + jl] = x[r];
    }
    __syncthreads();
    // first sub-diagonal: Y_i = N_{i+1,i} D_i, X_{i+1,i} = -D_{i+1} Y_i
    if (w < 3) {
        float* const A1[1] = {blk(Nb, w + 1, w)};
        float* const B1[1] = {blk(Xb, w, w)};
        blk_product<16, 1>(Yb + w * (kBlkBytes / 4), A1, B1, 0, 1.f);
    }
    __syncthreads();
    if (w < 3) {
        float* const A1[1] = {blk(Xb, w + 1, w + 1)};
        float* const B1[1] = {Yb + w * (kBlkBytes / 4)};
        blk_product<16, 1>(blk(Xb, w + 1, w), A1, B1, 0, -1.f);
    }
    __syncthreads();
    // second sub-diagonal: Z_i = N_{i+2,i} D_i + N_{i+2,i+1} X_{i+1,i}; X_{i+2,i} = -D_{i+2} Z_i
    {
        const int i = w >> 1, rb = (w & 1) * 8;
        float* const A2[2] = {blk(Nb, i + 2, i), blk(Nb, i + 2, i + 1)};
        float* const B2[2] = {blk(Xb, i, i), blk(Xb, i + 1, i)};
        blk_product<8, 2>(Yb + i * (kBlkBytes / 4), A2, B2, rb, 1.f);
    }
    __syncthreads();
    {
        const int i = w >> 1, rb = (w & 1) * 8;
        float* const A1[1] = {blk(Xb, i + 2, i + 2)};
        float* const B1[1] = {Yb + i * (kBlkBytes / 4)};
        blk_product<8, 1>(blk(Xb, i + 2, i), A1, B1, rb, -1.f);
    }
    __syncthreads();
    // third sub-diagonal: Z = N_30 D_0 + N_31 X_10 + N_32 X_20; X_30 = -D_3 Z
    {
        float* const A3[3] = {blk(Nb, 3, 0), blk(Nb, 3, 1), blk(Nb, 3, 2)};
        float* const B3[3] = {blk(Xb, 0, 0), blk(Xb, 1, 0), blk(Xb, 2, 0)};
        blk_product<4, 3>(Yb, A3, B3, 4 * w, 1.f);
    }
    __syncthreads();
    {
        float* const A1[1] = {blk(Xb, 3, 3)};
        float* const B1[1] = {Yb};
        blk_product<4, 1>(blk(Xb, 3, 0), A1, B1, 4 * w, -1.f);
    }
    __syncthreads();
    // T[r][s] = X[r][s] beta_s, bf16, row r: thread (r, half) writes 32 columns
    {
        const int r = tid >> 1, hf = tid & 1, bi = r >> 4, rr = r & 15;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            const int s0 = 32 * hf + 8 * ch, bj = s0 >> 4;
            uint32_t wv[4];
            if (bj <= bi) {
                const float* xr = blk(Xb, bi, bj) + rr * kBlkStride + (s0 & 15);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    wv[u] = pack_bf16x2(xr[2 * u] * beta_s[s0 + 2 * u], xr[2 * u + 1] * beta_s[s0 + 2 * u + 1]);
            } else {
                wv[0] = wv[1] = wv[2] = wv[3] = 0u;
            }
            *reinterpret_cast<uint4*>(sm + kTT + sw128_offset(r, 16 * (4 * hf + ch))) =
                make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
    }
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

// Lane j holds O^T row j.  The rows are transposed through a 64 x 256-byte
// staging tile (the -W'^T slot, dead after the Delta product) and written as
// 16-byte row segments, rows [r0, r1) only.
__device__ void store_out(uint32_t tb, uint8_t* sm, __nv_bfloat16* out, int64_t t0, int H, int h,
                          int r0, int r1) {
    uint32_t v[64];
    ld64(tb, kTmO, v);
    const int tid = threadIdx.x;
    uint8_t* stg = sm + kWT;
#pragma unroll
    for (int r = 0; r < 64; ++r)
        *reinterpret_cast<__nv_bfloat16*>(stg + r * 256 + tid * 2) = __float2bfloat16_rn(__uint_as_float(v[r]));
    __syncthreads();
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const int id = tid + kThreads * m, row = id >> 4, ch = id & 15;
        if (row >= r0 && row < r1) {
            const uint4 val = *reinterpret_cast<const uint4*>(stg + row * 256 + ch * 16);
            *reinterpret_cast<uint4*>(out + ((t0 + row) * H + h) * D + ch * 8) = val;
        }
    }
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

#ifdef KDA_PHASE_TIMING
// Diagnostic build only: cycles spent per phase by thread 0 of block 0.
__device__ unsigned long long g_phase_cycles[16];
#define KDA_PHASE(i)                                                        \
    do {                                                                    \
        if (blockIdx.x == 0 && threadIdx.x == 0) {                          \
            const long long t_ = clock64();                                 \
            g_phase_cycles[i] += (unsigned long long)(t_ - phase_t_);       \
            phase_t_ = t_;                                                  \
        }                                                                   \
    } while (0)
#else
#define KDA_PHASE(i) do {} while (0)
#endif

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
#ifdef KDA_PHASE_TIMING
    long long phase_t_ = clock64();
#endif

    float braw_next = (tid < C && bos + tid < eos) ? bf2f(beta[(bos + tid) * H + h]) : 0.f;
    for (int c = 0; c < nchunks && ok; ++c) {
        const int st = c & 1;
        uint8_t* stage = sm + st * kStageBytes;
        const uint32_t sQK = sQKbase + st * kStageBytes + kQK, sV = sQKbase + st * kStageBytes + kV;
        const int64_t t0 = bos + (int64_t)c * C;
        const int L = (int)((eos - t0) < C ? (eos - t0) : C);
        const float braw = braw_next;                 // beta of this chunk, loaded one chunk ahead
        if (c + 1 < nchunks) {
            const int64_t tn = t0 + C + tid;
            braw_next = (tid < C && tn < eos) ? bf2f(beta[tn * H + h]) : 0.f;
        }

        ok = wait_all(&full_bar[st], full_ph[st]);
        KDA_PHASE(0);
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
            KDA_PHASE(1);
            if (tid < C) beta_s[tid] = (tid >= r0 && tid < r1) ? braw : 0.f;
            build_operands(sm, st * kStageBytes, r0, r1, gam);
            __syncthreads();
            KDA_PHASE(2);
            decay_state(tb, gam);
            publish_to_mma();
            KDA_PHASE(3);

            if (tid == 0) {
                mma_gram(tb, sQK, sKB);
                mma_commit(&mma_bar);
            }
            mma_pending = true;
            if (!(ok = wait_all(&mma_bar, mma_ph))) break;
            mma_ph ^= 1u;
            mma_pending = false;
            tc_fence_after();
            KDA_PHASE(4);
            read_gram(tb, stage, sm, beta_s);
            fence_proxy_async_smem();
            __syncthreads();
            KDA_PHASE(5);
            solve_T(stage, sm, beta_s);
            publish_to_mma();
            KDA_PHASE(6);

            if (tid == 0) {
                mma_wu(tb, sQK, sV, sTT);
                mma_commit(&mma_bar);
            }
            mma_pending = true;
            if (!(ok = wait_all(&mma_bar, mma_ph))) break;
            mma_ph ^= 1u;
            mma_pending = false;
            tc_fence_after();
            KDA_PHASE(7);
            read_w(tb, sm);
            publish_to_mma();
            KDA_PHASE(8);

            if (tid == 0) {
                mma_delta_out(tb, sWT, sQK);
                mma_commit(&mma_bar);
            }
            mma_pending = true;
            if (!(ok = wait_all(&mma_bar, mma_ph))) break;
            mma_ph ^= 1u;
            mma_pending = false;
            tc_fence_after();
            KDA_PHASE(9);
            pack_delta(tb);
            publish_to_mma();
            KDA_PHASE(10);

            if (tid == 0) {
                mma_state_out(tb, sKB, sPP);
                mma_commit(&mma_bar);
            }
            mma_pending = true;
            if (!(ok = wait_all(&mma_bar, mma_ph))) break;
            mma_ph ^= 1u;
            mma_pending = false;
            tc_fence_after();
            KDA_PHASE(11);
            store_out(tb, sm, out, t0, H, h, r0, r1);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            KDA_PHASE(12);
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

#ifdef KDA_PHASE_TIMING
extern "C" int kda_debug_phase_cycles(unsigned long long* host16, int reset) {
    if (cudaMemcpyFromSymbol(host16, g_phase_cycles, 16 * sizeof(unsigned long long)) != cudaSuccess)
        return -1;
    if (reset) {
        unsigned long long z[16] = {};
        if (cudaMemcpyToSymbol(g_phase_cycles, z, sizeof(z)) != cudaSuccess) return -1;
    }
    return 0;
}
#endif

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
