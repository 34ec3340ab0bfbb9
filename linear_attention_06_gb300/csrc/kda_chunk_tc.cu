// kda_chunk_tc.cu -- chunkwise KDA prefill on sm_103a tensor cores (tcgen05).
//
// Scope: bf16 q, k, v, beta; fp32 log_alpha; dk = dv = 128; fp32 state.
//
// The math (one head, one chunk of C = 64 tokens r = 1..C, state S0 entering
// the chunk, a_r = log alpha_r, g_r = sum_{t<=r} a_t, G = g_C):
//
//   Unrolling the recurrence gives S_r = Diag(e^{g_r}) S0 +
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
//   First-Class Problem").  The same section of the Teardown says K3 floors the
//   decay so a 16-token tile stays in BF16 range on tensor cores; this kernel
//   uses its own exact scheme instead (below) and needs no floor on alpha.
//
// Decay factoring.  Everything is referred to the chunk END: with
// e_r = g_C - g_r = sum_{r<t<=C} a_t (<= 0),
//   Khat = e^{-e} o K, Qhat = e^{-e} o Q,  Kb = e^{e} o K,
//   A = Khat Kb^T, P = Qhat Kb^T, W = (T Khat) Diag(e^G),
//   (e^g o Q) S0 = Qhat (Diag(e^G) S0).
// With Ss = Diag(e^G) S0 (the decayed state, computed once per chunk):
//   Delta = U - (T Khat) Ss,  O = Qhat Ss + (mask o P) Delta,  S_C = Ss + Kb^T Delta.
// All exponents lie in [-|G|, |G|].  The tensor-core path takes a chunk when
// every channel has |G| <= 60 (e^60 ~ 1e26, far inside the bf16 / fp32
// range).  A chunk that decays harder than that is run token by token in fp32
// on the state held in tensor memory (exact for any log_alpha <= 0, -inf
// included); the K3-shaped inputs never need it.
//
// Work layout.  One CTA of 448 threads per (sequence, head) walks the
// sequence's chunks in order, in warp-specialised roles that form a pipeline:
//   team P (warps 0-3): decay-range check, Khat / Qhat / Kb tiles and the Gram
//      product [Khat;Qhat] Kb^T of chunk n+2,
//   team S (warps 4-7): N = Diag(beta) L(A) and the masked P, the UT solve T,
//      and W'^T = Khat^T T^T, U^T = V^T T^T of chunk n+1,
//   group B (warps 8-11): for chunk n the decayed state Ss and its bf16 copy,
//      Delta^T = U^T - Ss^T W'^T, the packed Delta, the output store (one TMA
//      store per warp) and the final state,
//   state/output issuer (warp 13): S^T += Delta^T Kb and O^T = Ss^T Qhat^T +
//      Delta^T P^T, issued while group B stores the previous chunk's output,
//   producer (warp 12): every TMA load, and L2 prefetches two chunks ahead.
// q/k, v and log_alpha have separate two-slot rings, each refilled as soon as
// its last reader is done.  Matrices that land in TMEM put a 128-wide
// dimension on the 128 lanes (M = 128 everywhere); the state lives in TMEM as
// fp32 S^T (lane = value channel, column = key channel) for the whole
// sequence, and the bf16 copies of Ss^T and Delta^T are packed into TMEM as the
// A operands of the products that read them.
//
// Diagnostic builds only: -DKDA_PHASE_TIMING adds per-role phase clock counters,
// -DKDA_TRACE_EVENTS a trace of block 0's product issues and completions, taken
// with one more warp that watches the completion barriers.  The product build
// compiles neither.
#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdint.h>

#include "kda_internal.h"
#include "sm103_primitives.cuh"

namespace kda {
namespace {

using namespace sm103;

constexpr int C = 64;          // chunk length (tokens)
constexpr int D = 128;         // dk = dv
// group A: two teams of 128 threads (P: operands and Gram, S: UT solve and W'/U), group B:
// 128 threads, then two single-thread warps: the TMA producer and the issuer of the
// state/output products
#ifdef KDA_TRACE_EVENTS
#define KDA_DIAG_TRACE 1
#endif
constexpr int kTeam = 128, kGroupA = 2 * kTeam, kGroupB = 128, kProducer = kGroupA + kGroupB,
              kIssuerOut = kProducer + 32;
#ifdef KDA_DIAG_TRACE
constexpr int kObserver = kIssuerOut + 32;   // diagnostic build: a warp that watches the products
constexpr int kThreads = kObserver + 32;
constexpr int kTraceChunks = 12, kTraceEvents = 8;   // traced chunks of block 0 (from g_trace_first)
#else
constexpr int kThreads = 448;
#endif
constexpr float kMaxExponent = 60.f;
constexpr uint64_t kWaitLimitNs = 4000000000ull;   // 4 s per bounded wait
constexpr int kBarP = 1, kBarB = 2, kBarS = 3;      // named barriers of the 128-thread groups

// ---- dynamic shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t kQK0 = 0;          // 2 x 32 KB: [k_h0 | q_h0 | k_h1 | q_h1], 64 rows x 128 B, SW128
constexpr uint32_t kV0 = 65536;       // 2 x 16 KB: [v_h0 | v_h1]
constexpr uint32_t kA0 = 98304;       // 2 x 32 KB: log_alpha fp32 [64][128]; then solve scratch + T
constexpr uint32_t kKB0 = 163840;     // 2 x 16 KB: Kb [halves]
constexpr uint32_t kPP0 = 196608;     // 2 x 8 KB: masked P, K-major
constexpr uint32_t kWT = 212992;      // 16 KB: -W'^T (MN-major), then 4 x 4 KB output staging tiles
constexpr uint32_t kSmall = 229376;   // 2 KB: barriers, flags, beta, gamma
constexpr uint32_t kSmemUsed = kSmall + 2048;
constexpr uint32_t kSmemDynamic = kSmemUsed + 1024;   // + alignment slack = 232448
// inside an A slot, after log_alpha has been consumed:
constexpr uint32_t kBlkStride = 16, kBlkBytes = 16 * kBlkStride * 4;   // 1024
constexpr uint32_t kSolveN = 0, kSolveX = 10 * kBlkBytes, kSolveY = 20 * kBlkBytes;
constexpr uint32_t kTT = 24576;                                        // T, 64 x 128 B, SW128
constexpr uint32_t kQKBytes = 32768, kVBytes = 16384, kABytes = 32768;

// ---- TMEM columns
constexpr uint32_t kTmS = 0, kTmSbf = 128, kTmDbf = 192;
// two slots (chunk parity) each for U / Delta / then the chunk's output O, and for the Gram result,
// which W' later overwrites
__device__ __forceinline__ uint32_t tm_u(int s) { return 256u + 64u * s; }
__device__ __forceinline__ uint32_t tm_apw(int s) { return 384u + 64u * s; }
constexpr uint32_t kTmCols = 512;

struct Maps {
    CUtensorMap q, k, v, a, o;
};

// Barriers and small per-slot data in the kSmall area.
struct Small {
    uint64_t qk_full[2], v_full[2], a_full[2];   // TMA completions
    uint64_t ready[2];                           // group A -> B: chunk prepared and W', U computed (2 arrivals)
    uint64_t kbp_free[2];                        // state product -> team P: Kb / P / beta / gamma slot free
    uint64_t gram_done[2];                       // team P -> team S: Gram product landed (or token chunk)
    uint64_t mma1_done, mma2_done;
    uint64_t av_free[2];                         // log_alpha / v slot free (W', U done, or token path)
    uint64_t qk_free[2];                         // q / k slot free (output product done, or token path)
    uint64_t u_free[2];                          // group B read the output held in a U slot (4 warps)
    uint64_t packed;                             // group B -> state/output issuer: Delta packed (slot in cmd_b)
    uint64_t drain, drain_p, drain_s;            // issuing threads: their products landed (at exit)
    uint32_t tmem_base;
    int mode[2];                                 // 0 tensor-core chunk, 1 token-by-token chunk
    int cmd_b;                                   // slot of the packed chunk, -1: group B is done
    int issued[3][2];                            // TMA loads issued / waited for, per
    int consumed[3][2];                          //   (kind, slot), to drain after a timeout
    __nv_bfloat16 beta[2][C];                    // bf16 inputs: exact
    float gam[2][D];
#ifdef KDA_PHASE_TIMING
    unsigned long long phase[32];                // diagnostic build only
#endif
#ifdef KDA_DIAG_TRACE
    int cmd_n;                                   // chunk index of cmd_b (diagnostic build)
    int trace_first;                             // first traced chunk (diagnostic build)
    uint32_t trace[kTraceChunks][kTraceEvents];  // block 0's product events (diagnostic build)
#endif
};
static_assert(sizeof(Small) <= 2048, "small area");
static_assert(offsetof(Small, gam) % 16 == 0, "gamma rows are read as float4");
static_assert(offsetof(Small, beta) % 16 == 0, "beta is read eight at a time");

__device__ __forceinline__ uint32_t qk_off(bool is_q, uint32_t r, uint32_t c) {
    return (c >> 6) * 16384u + (is_q ? 8192u : 0u) + sw128_offset(r, (c & 63u) * 2u);
}
__device__ __forceinline__ uint32_t half_off(uint32_t r, uint32_t c) {   // V and Kb
    return (c >> 6) * 8192u + sw128_offset(r, (c & 63u) * 2u);
}
__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ bool in_group_a() { return threadIdx.x < kGroupA; }
__device__ __forceinline__ bool in_team_p() { return threadIdx.x < kTeam; }
// Index of the thread inside its group (0..127 in teams P and S and in B, the lane in the
// single-thread warps).
__device__ __forceinline__ int lt() {
    return threadIdx.x < kProducer ? (int)(threadIdx.x & 127) : (int)(threadIdx.x & 31);
}
// First TMEM lane this warp may access (the warp's lane quarter).
__device__ __forceinline__ uint32_t lane0() { return ((threadIdx.x >> 5) & 3) * 32; }
__device__ __forceinline__ int group_count(int) { return kTeam; }

__device__ __forceinline__ void group_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(group_count(id)) : "memory");
}
// OR / AND of a predicate over the threads of a group (also a barrier).
__device__ __forceinline__ bool group_or(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(group_count(id))
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool group_and(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(group_count(id))
        : "memory");
    return r != 0;
}
// Every thread of the group waits (bounded); the group agrees on the outcome.
__device__ __forceinline__ bool group_wait(int id, uint64_t* bar, uint32_t parity) {
    return group_and(id, mbar_wait_parked(bar, parity, kWaitLimitNs));
}
// Make this thread's shared-memory and TMEM writes visible to the tensor core
// and synchronise the group.
__device__ __forceinline__ void group_publish(int id) {
    fence_proxy_async_smem();
    tc_fence_before();
    group_sync(id);
    tc_fence_after();
}

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

// ============================ group A: chunk-local stage =========================

// Operand build, team P (128 threads).
// Pass 1 (build_suffix, thread = key channel c): suffix sums of log_alpha over the
// chunk, e[r][c] = sum_{r<t<L} a[t][c]; returns false (leaving log_alpha untouched)
// when a channel's chunk total leaves +-kMaxExponent, else writes e back in place and
// returns g = e^{G_c}.  It touches only the log_alpha slot, so it runs before the
// chunk's other slots are free; the caller publishes g once they are.
// Pass 2 (build_tiles, thread = 16-byte chunk of 8 channels of one row):
// Khat = e^{-e} k, Qhat = e^{-e} q (in place), Kb = e^{e} k, all as 16-byte vector
// accesses.
__device__ bool build_suffix(float* A, int L, float& g) {
    const int c = lt();
    float e[C];
#pragma unroll
    for (int r = 0; r < C; ++r) e[r] = (r < L) ? A[r * D + c] : 0.f;
    float run = 0.f;
#pragma unroll
    for (int r = C - 1; r >= 0; --r) {
        const float ar = e[r];
        e[r] = run;
        run += ar;
    }
    if (group_or(kBarP, !(fabsf(run) <= kMaxExponent))) return false;
    g = __expf(run);
#pragma unroll
    for (int r = 0; r < C; ++r) A[r * D + c] = e[r];
    group_sync(kBarP);
    return true;
}

__device__ void build_tiles(uint8_t* qk, uint8_t* kb, const float* A, int L) {
    const int c = lt();
    // pass 2: 64 rows x 16 chunks = 1024 units, 8 per thread
#pragma unroll 2
    for (int m = 0; m < 8; ++m) {
        const int u = c + kTeam * m, r = u >> 4, j = u & 15;
        const uint32_t ko = qk_off(false, r, 8 * j), qo = qk_off(true, r, 8 * j), bo = half_off(r, 8 * j);
        uint4 kh = make_uint4(0u, 0u, 0u, 0u), qh = kh, kbv = kh;
        if (r < L) {
            const uint4 kr = *reinterpret_cast<const uint4*>(qk + ko);
            const uint4 qr = *reinterpret_cast<const uint4*>(qk + qo);
            const float4 e0 = *reinterpret_cast<const float4*>(A + r * D + 8 * j);
            const float4 e1 = *reinterpret_cast<const float4*>(A + r * D + 8 * j + 4);
            const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
            const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w}, qw[4] = {qr.x, qr.y, qr.z, qr.w};
            uint32_t o1[4], o2[4], o3[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float k0 = __uint_as_float(kw[p] << 16), k1 = __uint_as_float(kw[p] & 0xffff0000u);
                const float q0 = __uint_as_float(qw[p] << 16), q1 = __uint_as_float(qw[p] & 0xffff0000u);
                const float u0 = __expf(-ev[2 * p]), u1 = __expf(-ev[2 * p + 1]);
                const float d0 = __expf(ev[2 * p]), d1 = __expf(ev[2 * p + 1]);
                o1[p] = pack_bf16x2(k0 * u0, k1 * u1);
                o2[p] = pack_bf16x2(q0 * u0, q1 * u1);
                o3[p] = pack_bf16x2(k0 * d0, k1 * d1);
            }
            kh = make_uint4(o1[0], o1[1], o1[2], o1[3]);
            qh = make_uint4(o2[0], o2[1], o2[2], o2[3]);
            kbv = make_uint4(o3[0], o3[1], o3[2], o3[3]);
        }
        *reinterpret_cast<uint4*>(qk + ko) = kh;
        *reinterpret_cast<uint4*>(qk + qo) = qh;
        *reinterpret_cast<uint4*>(kb + bo) = kbv;
    }
}


__device__ __forceinline__ float* blk(float* base, int i, int j) {
    return base + (i * (i + 1) / 2 + j) * (kBlkBytes / 4);
}
// Element (r, c) of a 16x16 solve block sits at r * 16 + (c ^ blk_swz(r)): the swizzle
// moves 4-column groups by row so that the m16n8k8 fragment loads and the 16-byte row
// stores of a warp hit distinct banks.
__device__ __forceinline__ int blk_swz(int r) { return ((r << 2) & 8) | (r & 4); }
__device__ __forceinline__ int blk_at(int r, int c) { return r * kBlkStride + (c ^ blk_swz(r)); }

// TMEM lanes 0-63 hold A rows r: N = beta_r A_rs (s < r) as fp32
// lower-triangular 16x16 blocks in the A slot.  Lanes 64-127 hold P rows r:
// P_rs (s <= r) as the bf16 K-major operand tile.  Team S: each thread takes
// its lane's row, columns 0-31 then 32-63.
__device__ void read_gram(uint32_t tb, uint32_t col, uint8_t* aslot, uint8_t* pp, const __nv_bfloat16* beta) {
    const int row = (int)lane0() + (lt() & 31);
#pragma unroll 1
    for (int ch = 0; ch < 2; ++ch) {                 // column half
        uint32_t v[32];
        tmem_ld32(tmem_addr(tb, lane0(), col + 32 * ch), v);
        tmem_wait_ld();
        if (row < 64) {
            const int r = row, bi = r >> 4, rr = r & 15;
            const float b = bf2f(beta[r]);
            float* Nb = reinterpret_cast<float*>(aslot + kSolveN);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int bj = 2 * ch + k;
                if (bj > bi) break;
                float* dst = blk(Nb, bi, bj);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int s0 = 16 * bj + 4 * q4, i0 = 16 * k + 4 * q4;
                    float4 f;
                    f.x = (s0 + 0 < r) ? b * __uint_as_float(v[i0 + 0]) : 0.f;
                    f.y = (s0 + 1 < r) ? b * __uint_as_float(v[i0 + 1]) : 0.f;
                    f.z = (s0 + 2 < r) ? b * __uint_as_float(v[i0 + 2]) : 0.f;
                    f.w = (s0 + 3 < r) ? b * __uint_as_float(v[i0 + 3]) : 0.f;
                    *reinterpret_cast<float4*>(dst + blk_at(rr, 4 * q4)) = f;
                }
            }
        } else {
            const int r = row - 64;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int chunk = 4 * ch + k;
                uint32_t w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int s = 8 * chunk + 2 * u, i = 8 * k + 2 * u;
                    const float lo = (s <= r) ? __uint_as_float(v[i]) : 0.f;
                    const float hi = (s + 1 <= r) ? __uint_as_float(v[i + 1]) : 0.f;
                    w[u] = pack_bf16x2(lo, hi);
                }
                *reinterpret_cast<uint4*>(pp + sw128_offset(r, 16 * chunk)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// d += a(16x8, row-major fragment) * b(8x8, column fragment), TF32 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// One warp: columns [8 nt, 8 nt + 8) of C = sign * sum_p A_p B_p for 16x16 blocks (blk_at
// layout).
// With WT, the block is also written, column-scaled by beta, as bf16 into the T tile at
// rows trow0 + 0..15, columns tcol0 + 0..15.
template <int NP, bool WT = false>
__device__ __forceinline__ void blk_mma(float* Cb, const float* const (&Ab)[NP], const float* const (&Bb)[NP],
                                        int nt, float sign, uint8_t* tt = nullptr, int trow0 = 0, int tcol0 = 0,
                                        const __nv_bfloat16* beta = nullptr) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int p = 0; p < NP; ++p) {
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const float* A = Ab[p];
            const float* B = Bb[p];
            const int k0 = 8 * ks;
            const uint32_t af[4] = {to_tf32(A[blk_at(g, k0 + t)]), to_tf32(A[blk_at(g + 8, k0 + t)]),
                                    to_tf32(A[blk_at(g, k0 + t + 4)]), to_tf32(A[blk_at(g + 8, k0 + t + 4)])};
            const uint32_t bf[2] = {to_tf32(B[blk_at(k0 + t, 8 * nt + g)]), to_tf32(B[blk_at(k0 + t + 4, 8 * nt + g)])};
            mma_tf32(d, af, bf);
        }
    }
    const int c0 = 8 * nt + 2 * t;                   // a column pair stays adjacent under the swizzle
    *reinterpret_cast<float2*>(Cb + blk_at(g, c0)) = make_float2(sign * d[0], sign * d[1]);
    *reinterpret_cast<float2*>(Cb + blk_at(g + 8, c0)) = make_float2(sign * d[2], sign * d[3]);
    if constexpr (WT) {
        const float b0 = bf2f(beta[tcol0 + c0]), b1 = bf2f(beta[tcol0 + c0 + 1]);
        const uint32_t cb = 2u * (uint32_t)(tcol0 + c0);
        *reinterpret_cast<uint32_t*>(tt + sw128_offset(trow0 + g, cb)) = pack_bf16x2(sign * d[0] * b0, sign * d[1] * b1);
        *reinterpret_cast<uint32_t*>(tt + sw128_offset(trow0 + g + 8, cb)) =
            pack_bf16x2(sign * d[2] * b0, sign * d[3] * b1);
    }
}

// T = (I + N)^{-1} Diag(beta) with N strictly lower 64x64 (10 lower 16x16 blocks in the A slot):
// D_i = (I + N_ii)^{-1} by fp32 forward substitution; then the 32x32 halves
// X_10 = -D_1 N_10 D_0, X_32 = -D_3 N_32 D_2; then the lower-left 32x32 quarter
// -C^{-1} (B A^{-1}) with A^{-1}, C^{-1} the inverted halves and B = N[32:64, 0:32], using TF32
// tensor-core block products with fp32 accumulation.  Each step writes the blocks of T it
// finishes (X column-scaled by beta, bf16, into the swizzled T tile) as it stores them, and
// the idle warps of the first step write T's zero blocks.  Team S (4 warps), 4 team barriers.
__device__ void solve_T(uint8_t* aslot, const __nv_bfloat16* beta, Small* x_sw) {
#ifdef KDA_PHASE_TIMING
    long long sp_ = clock64();
#endif
    float* Nb = reinterpret_cast<float*>(aslot + kSolveN);
    float* Xb = reinterpret_cast<float*>(aslot + kSolveX);
    float* Yb = reinterpret_cast<float*>(aslot + kSolveY);   // 4 blocks
    const int t = lt(), w = t >> 5;
    if (t < 64) {
        const int i = t >> 4, jl = t & 15;
        const float* Nii = blk(Nb, i, i);
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {               // four partial sums: a short dependence chain
            float p[4] = {(r == jl) ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q = 0; q < r; ++q) p[q & 3] = fmaf(-Nii[blk_at(r, q)], x[q], p[q & 3]);
            x[r] = (p[0] + p[1]) + (p[2] + p[3]);
        }
        float* Xii = blk(Xb, i, i);
#pragma unroll
        for (int r = 0; r < 16; ++r) Xii[blk_at(r, jl)] = x[r];
        const float bj = bf2f(beta[16 * i + jl]);        // T_ii column jl = D_i column jl x beta
        uint8_t* tt = aslot + kTT;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            *reinterpret_cast<__nv_bfloat16*>(tt + sw128_offset(16 * i + r, 2 * (16 * i + jl))) =
                __float2bfloat16_rn(x[r] * bj);
    } else {                                         // the zero blocks above the diagonal of T
        const int u = t - 64;                        // 64 threads x 3 of the 6 x 16 rows x 2 16-byte pieces
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int id = u + 64 * k;               // 0 .. 191: block (6), row (16), half (2)
            const int b = id >> 5, rr = (id >> 1) & 15, hf = id & 1;
            const int bi = b < 3 ? 0 : (b < 5 ? 1 : 2), q = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
            *reinterpret_cast<uint4*>(aslot + kTT + sw128_offset(16 * bi + rr, 32 * q + 16 * hf)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    }
    group_sync(kBarS);
#ifdef KDA_PHASE_TIMING
    if (t == 0) { const long long c_ = clock64(); x_sw->phase[26 + 1] += (unsigned long long)(c_ - sp_); sp_ = c_; }
#endif
    // halves: warps 0-1 -> X_10 (n-tile w), warps 2-3 -> X_32 (n-tile w-2); Y via the block's own
    // Y slot, the chain stays inside the warp
    if (w < 4) {
        const int hb = w >> 1, nt = w & 1;                   // hb 0: blocks (1,0); hb 1: blocks (3,2)
        const int i0 = 2 * hb;                               // diagonal index of the upper block
        float* Ys = Yb + hb * (kBlkBytes / 4);
        {
            const float* A1[1] = {blk(Nb, i0 + 1, i0)};
            const float* B1[1] = {blk(Xb, i0, i0)};
            blk_mma<1>(Ys, A1, B1, nt, 1.f);
        }
        __syncwarp();
        // the second product needs both column tiles of Y; tile nt only depends on Y tile nt
        {
            const float* A1[1] = {blk(Xb, i0 + 1, i0 + 1)};
            const float* B1[1] = {Ys};
            blk_mma<1, true>(blk(Xb, i0 + 1, i0), A1, B1, nt, -1.f, aslot + kTT, 16 * (i0 + 1), 16 * i0, beta);
        }
    }
    group_sync(kBarS);
#ifdef KDA_PHASE_TIMING
    if (t == 0) { const long long c_ = clock64(); x_sw->phase[26 + 2] += (unsigned long long)(c_ - sp_); sp_ = c_; }
#endif
    // Y = B A^{-1}: Y_20 = N_20 D_0 + N_21 X_10, Y_21 = N_21 D_1, Y_30 = N_30 D_0 + N_31 X_10, Y_31 = N_31 D_1
#pragma unroll 1
    for (int it = 0; it < 2; ++it) {                 // each warp: one two-term and one one-term block
        const int ob = 2 * (w >> 1) + it, nt = w & 1;   // ob: 0 Y20, 1 Y21, 2 Y30, 3 Y31
        const int ri = 2 + (ob >> 1), cj = ob & 1;
        float* Ys = Yb + ob * (kBlkBytes / 4);
        if (cj == 0) {
            const float* A2[2] = {blk(Nb, ri, 0), blk(Nb, ri, 1)};
            const float* B2[2] = {blk(Xb, 0, 0), blk(Xb, 1, 0)};
            blk_mma<2>(Ys, A2, B2, nt, 1.f);
        } else {
            const float* A1[1] = {blk(Nb, ri, 1)};
            const float* B1[1] = {blk(Xb, 1, 1)};
            blk_mma<1>(Ys, A1, B1, nt, 1.f);
        }
    }
    group_sync(kBarS);
#ifdef KDA_PHASE_TIMING
    if (t == 0) { const long long c_ = clock64(); x_sw->phase[26 + 3] += (unsigned long long)(c_ - sp_); sp_ = c_; }
#endif
    // X_lower = -C^{-1} Y: X_20 = -D_2 Y_20, X_21 = -D_2 Y_21, X_30 = -(X_32 Y_20 + D_3 Y_30), X_31 = -(X_32 Y_21 + D_3 Y_31)
#pragma unroll 1
    for (int it = 0; it < 2; ++it) {
        const int item = w + 4 * it, ob = item >> 1, nt = item & 1;
        const int ri = 2 + (ob >> 1), cj = ob & 1;
        if (ri == 2) {
            const float* A1[1] = {blk(Xb, 2, 2)};
            const float* B1[1] = {Yb + cj * (kBlkBytes / 4)};
            blk_mma<1, true>(blk(Xb, 2, cj), A1, B1, nt, -1.f, aslot + kTT, 32, 16 * cj, beta);
        } else {
            const float* A2[2] = {blk(Xb, 3, 2), blk(Xb, 3, 3)};
            const float* B2[2] = {Yb + cj * (kBlkBytes / 4), Yb + (2 + cj) * (kBlkBytes / 4)};
            blk_mma<2, true>(blk(Xb, 3, cj), A2, B2, nt, -1.f, aslot + kTT, 48, 16 * cj, beta);
        }
    }
    group_sync(kBarS);
#ifdef KDA_PHASE_TIMING
    if (t == 0) { const long long c_ = clock64(); x_sw->phase[26 + 4] += (unsigned long long)(c_ - sp_); sp_ = c_; }
#endif
    // (every block of T was written by the step that computed it)
}

// ============================ group B: state stage ===============================

// TMEM S^T (lane j = value channel, column c = key channel): S <- S Diag(gam)
// in fp32, and the bf16 copy of the decayed state packed as an A operand.
// Works in 32-column steps to keep the register footprint small.
__device__ void decay_state(uint32_t tb, const float* gam) {
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t v[32], pk[16];
        tmem_ld32(tmem_addr(tb, lane0(), kTmS + 32 * cb), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 g = *reinterpret_cast<const float4*>(gam + 32 * cb + 4 * i);
            v[4 * i + 0] = __float_as_uint(__uint_as_float(v[4 * i + 0]) * g.x);
            v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) * g.y);
            v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) * g.z);
            v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) * g.w);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        tmem_st32(tmem_addr(tb, lane0(), kTmS + 32 * cb), v);
        tmem_st16(tmem_addr(tb, lane0(), kTmSbf + 16 * cb), pk);
    }
    tmem_wait_st();
}

// The warp's 4 KB of the W / staging area may still be read by its last output TMA store:
// wait for that read (lane 0 issued it) before the area is written again.
__device__ __forceinline__ void staging_ready() {
    if ((threadIdx.x & 31) == 0) bulk_wait_read();
    __syncwarp();
}

// Lane c holds W'^T row c (64 tokens): store -W'^T as bf16, MN-major B operand.
__device__ void read_w(uint32_t tb, uint32_t col, uint8_t* wt) {
    const int c = lt();
    staging_ready();
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[32];
        tmem_ld32(tmem_addr(tb, lane0(), col + 32 * hf), v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                w[u] = pack_bf16x2(-__uint_as_float(v[8 * k + 2 * u]), -__uint_as_float(v[8 * k + 2 * u + 1]));
            *reinterpret_cast<uint4*>(wt + sw128_offset(c, 16 * (4 * hf + k))) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// Lane j holds Delta^T row j (fp32): pack to bf16 in TMEM as an A operand.
__device__ void pack_delta(uint32_t tb, uint32_t col) {
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[32], pk[16];
        tmem_ld32(tmem_addr(tb, lane0(), col + 32 * hf), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        tmem_st16(tmem_addr(tb, lane0(), kTmDbf + 16 * hf), pk);
    }
    tmem_wait_st();
}

// Lane j holds O^T row j: read it out of TMEM, packed to bf16 pairs of rows.
__device__ __forceinline__ void o_to_regs(uint32_t tb, uint32_t col, uint32_t (&opk)[32]) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[32];
        tmem_ld32(tmem_addr(tb, lane0(), col + 32 * hf), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) opk[16 * hf + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    }
}

// (lim: floats in the state buffer, for the index checks of bounds-checked builds)
__device__ void load_state(uint32_t tb, const float* h0, size_t base, int64_t lim, unsigned int* status) {
    const int j = lt();
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const size_t e = base + (size_t)(32 * cb + i) * D + j;
            r[i] = (h0 && KDA_INDEX_OK(e, lim, status)) ? __float_as_uint(h0[e]) : 0u;
        }
        tmem_st32(tmem_addr(tb, lane0(), kTmS + 32 * cb), r);
    }
    tmem_wait_st();
}

__device__ void store_state(uint32_t tb, float* hT, size_t base, int64_t lim, unsigned int* status) {
    const int j = lt();
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tb, lane0(), kTmS + 32 * cb), r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const size_t e = base + (size_t)(32 * cb + i) * D + j;
            if (KDA_INDEX_OK(e, lim, status)) hT[e] = __uint_as_float(r[i]);
        }
    }
}

// Exact token-by-token path for a chunk whose decay leaves the factored
// range: the state row of lane j (value channel) is updated in fp32 with the
// recurrence itself (decay, erase with beta, write with beta, read after the
// write).  log_alpha in the A slot is first turned into alpha in place.
// The outputs o_r go to TMEM column ucol + r of the thread's lane (its value
// channel), where the chunk's output is stored from like any other chunk's.
// The row stays in TMEM and is walked 32 columns at a time (two passes per
// token: decay and the read under k, then the write and the read with q), so the
// path needs few registers; it is rare (only chunks with |G| > kMaxExponent).
__device__ __noinline__ void token_chunk(uint32_t tb, float* A, const uint8_t* qk, const uint8_t* vv,
                                            const __nv_bfloat16* beta, uint32_t ucol, int L) {
    const int j = lt();
#pragma unroll 1
    for (int r = 0; r < L; ++r) A[r * D + j] = expf(A[r * D + j]);
    group_sync(kBarB);
#pragma unroll 1
    for (int r = 0; r < L; ++r) {
        const float* al = A + r * D;
        float rk = 0.f;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {              // decay, and what S holds under k
            uint32_t u[32];
            tmem_ld32(tmem_addr(tb, lane0(), kTmS + 32 * cb), u);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = 32 * cb + i;
                const float sc = __uint_as_float(u[i]) * al[c];
                u[i] = __float_as_uint(sc);
                rk = fmaf(sc, bf2f(*reinterpret_cast<const __nv_bfloat16*>(qk + qk_off(false, r, c))), rk);
            }
            tmem_st32(tmem_addr(tb, lane0(), kTmS + 32 * cb), u);
            tmem_wait_st();
        }
        const float vj = bf2f(*reinterpret_cast<const __nv_bfloat16*>(vv + half_off(r, j)));
        const float d = bf2f(beta[r]) * (vj - rk);
        float y = 0.f;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {              // erase and write with the same beta, read with q
            uint32_t u[32];
            tmem_ld32(tmem_addr(tb, lane0(), kTmS + 32 * cb), u);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = 32 * cb + i;
                const float sc = fmaf(bf2f(*reinterpret_cast<const __nv_bfloat16*>(qk + qk_off(false, r, c))), d,
                                      __uint_as_float(u[i]));
                u[i] = __float_as_uint(sc);
                y = fmaf(sc, bf2f(*reinterpret_cast<const __nv_bfloat16*>(qk + qk_off(true, r, c))), y);
            }
            tmem_st32(tmem_addr(tb, lane0(), kTmS + 32 * cb), u);
            tmem_wait_st();
        }
        tmem_st1(tmem_addr(tb, lane0(), ucol + r), __float_as_uint(y));
    }
    tmem_wait_st();
}

// ---- MMA groups (each issued by one thread) --------------------------------------
// AP = [Khat; Qhat] x Kb^T : M = 128, N = 64, K = 128 (both K-major).
__device__ __forceinline__ void mma_gram(uint32_t tb, uint32_t dcol, uint32_t sQK, uint32_t sKB) {
    constexpr uint32_t id = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
    for (uint32_t ks = 0; ks < 8; ++ks) {
        const uint64_t a = smem_desc(sQK + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, kSwizzle128B);
        const uint64_t b = smem_desc(sKB + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, kSwizzle128B);
        mma_ss(tb + dcol, a, b, id, ks > 0);
    }
}

// W'^T = Khat^T T^T -> W columns; U^T = V^T T^T -> U columns.  M = 128, N = 64,
// K = 64 tokens; A operands MN-major (channel halves LBO apart), B = T K-major.
__device__ __forceinline__ void mma_wu(uint32_t tb, uint32_t wcol, uint32_t ucol, uint32_t sQK, uint32_t sV,
                                       uint32_t sTT) {
    constexpr uint32_t id = idesc_bf16_f32(128, 64, true, false);
#pragma unroll
    for (uint32_t ks = 0; ks < 4; ++ks) {
        const uint64_t b = smem_desc(sTT + ks * 32, 16, 1024, kSwizzle128B);
        mma_ss(tb + wcol, smem_desc(sQK + ks * 2048, 16384, 1024, kSwizzle128B), b, id, ks > 0);
        mma_ss(tb + ucol, smem_desc(sV + ks * 2048, 8192, 1024, kSwizzle128B), b, id, ks > 0);
    }
}

// Delta^T = U^T + Ss^T (-W'^T) in the U slot: A = Ss^T from TMEM, K = 128.
__device__ __forceinline__ void mma_delta(uint32_t tb, uint32_t ucol, uint32_t sWT) {
    constexpr uint32_t idw = idesc_bf16_f32(128, 64, false, true);
#pragma unroll
    for (uint32_t ks = 0; ks < 8; ++ks)
        mma_ts(tb + ucol, tb + kTmSbf + ks * 8, smem_desc(sWT + ks * 2048, 16384, 1024, kSwizzle128B),
               idw, 1);
}

// S^T += Delta^T Kb (N = 128, Kb MN-major); then the chunk output, in the U slot
// (Delta is already packed): O^T = Ss^T Qhat^T + Delta^T P^T.
__device__ __forceinline__ void mma_state_out(uint32_t tb, uint32_t ocol, uint32_t sKB, uint32_t sQK,
                                              uint32_t sPP) {
    constexpr uint32_t ids = idesc_bf16_f32(128, 128, false, true);
    constexpr uint32_t idq = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
    for (uint32_t ks = 0; ks < 4; ++ks)
        mma_ts(tb + kTmS, tb + kTmDbf + ks * 8, smem_desc(sKB + ks * 2048, 8192, 1024, kSwizzle128B),
               ids, 1);
#pragma unroll
    for (uint32_t ks = 0; ks < 8; ++ks)
        mma_ts(tb + ocol, tb + kTmSbf + ks * 8,
               smem_desc(sQK + 8192 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, kSwizzle128B), idq,
               ks > 0);
#pragma unroll
    for (uint32_t ks = 0; ks < 4; ++ks)
        mma_ts(tb + ocol, tb + kTmDbf + ks * 8, smem_desc(sPP + ks * 32, 16, 1024, kSwizzle128B), idq, 1);
}

#ifdef KDA_PHASE_TIMING
// Diagnostic build only: cycles per phase, summed over the blocks, as seen by
// the first thread of each group; accumulated in shared memory and added to
// the global counters when the block ends.
__device__ unsigned long long g_phase_cycles[32];
#define KDA_PHASE(i)                                                                  \
    do {                                                                              \
        if (lt() == 0) {                                                              \
            const long long t_ = clock64();                                           \
            x.sw->phase[i] += (unsigned long long)(t_ - phase_t_);                    \
            phase_t_ = t_;                                                            \
        }                                                                             \
    } while (0)
#define KDA_PHASE_INIT long long phase_t_ = clock64()
#else
#define KDA_PHASE(i) do {} while (0)
#define KDA_PHASE_INIT do {} while (0)
#endif
#ifdef KDA_DIAG_TRACE
// Event trace of block 0 (diagnostic build): the low 32 bits of the SM clock at
// the issue (events 0, 2, 4, 6) and completion (1, 3, 5, 7) of the four product
// groups of chunks g_trace_first .. g_trace_first + kTraceChunks - 1 (set by
// kda_debug_set_trace_first, 48 unless changed).  Kept in shared
// memory during the run and copied out when the block ends: stamping straight to
// global memory slowed the traced block, and so the launch, by a quarter.
__device__ uint32_t g_trace[kTraceChunks][kTraceEvents];
__device__ int g_trace_first = 48;
__device__ __forceinline__ bool trace_chunk(const Small& sw, int n) {
    return (unsigned)(n - sw.trace_first) < (unsigned)kTraceChunks;
}
#define KDA_TRACE(n, ev)                                                              \
    do {                                                                              \
        if (blockIdx.x == 0 && lt() == 0 && trace_chunk(*x.sw, (n)))                  \
            x.sw->trace[(n) - x.sw->trace_first][(ev)] = (uint32_t)clock64();         \
    } while (0)
#else
#define KDA_TRACE(n, ev) do {} while (0)
#endif

// ============================ TMA ring refills ===================================
__device__ __forceinline__ void load_qk(uint8_t* dst, const Maps& m, int h, int t0, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, kQKBytes);
    tma_load_3d(dst + 0, &m.k, 0, h, t0, bar);
    tma_load_3d(dst + 8192, &m.q, 0, h, t0, bar);
    tma_load_3d(dst + 16384, &m.k, 64, h, t0, bar);
    tma_load_3d(dst + 24576, &m.q, 64, h, t0, bar);
}
__device__ __forceinline__ void load_v(uint8_t* dst, const Maps& m, int h, int t0, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, kVBytes);
    tma_load_3d(dst, &m.v, 0, h, t0, bar);
    tma_load_3d(dst + 8192, &m.v, 64, h, t0, bar);
}
__device__ __forceinline__ void load_a(uint8_t* dst, const Maps& m, int h, int t0, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, kABytes);
    tma_load_3d(dst, &m.a, 0, h, t0, bar);
}

struct Ctx {
    uint8_t* sm;
    Small* sw;
    uint32_t tb;
    int64_t bos, eos;
    int nchunks, H, h, seq;
    int64_t T;                   // tokens of the packed batch (index checks)
    int num_seqs;
    unsigned int* status;
};

// Optional checkpoints of one sequence: the state after ck_pos[c] tokens goes to
// ck_states[c]; a position that is not a chunk end (a multiple of 64 or the
// sequence end) is skipped.
struct Ckpt {
    const int32_t* pos;
    float* states;
    int c, end;
    int64_t lim;                 // floats in the checkpoint buffer (index checks)
    unsigned int* status;
    __device__ void init(const int32_t* ck_cu, const int32_t* ck_pos, float* ck_states, int seq, int num_seqs,
                         int H, unsigned int* st) {
        pos = ck_pos;
        states = ck_states;
        status = st;
        c = end = 0;
        lim = 0;
        if (ck_states) {
            c = ck_cu[seq];
            end = ck_cu[seq + 1];
            lim = (int64_t)ck_cu[num_seqs] * H * D * D;
        }
    }
    // called by the whole group after the chunk that ends `done` tokens into the sequence
    __device__ void after_chunk(uint32_t tb, int64_t done, bool seq_end, int H, int h) {
        while (c < end) {
            const int64_t p = pos[c];
            if (p > done) break;
            if (p == done && (done % C == 0 || seq_end))
                store_state(tb, states, ((size_t)c * H + h) * D * D, lim, status);
            ++c;
        }
    }
};

enum { kLdQK = 0, kLdV = 1, kLdA = 2 };

// TMA refill of slot s with the tiles of chunk c (issued by one thread).
__device__ __forceinline__ void refill(const Ctx& x, const Maps& maps, int c, int s, bool a, bool v, bool q) {
    Small& sw = *x.sw;
    const int tc = (int)(x.bos + (int64_t)c * C);
    if (a) { load_a(x.sm + kA0 + s * kABytes, maps, x.h, tc, &sw.a_full[s]); ++sw.issued[kLdA][s]; }
    if (v) { load_v(x.sm + kV0 + s * kVBytes, maps, x.h, tc, &sw.v_full[s]); ++sw.issued[kLdV][s]; }
    if (q) { load_qk(x.sm + kQK0 + s * kQKBytes, maps, x.h, tc, &sw.qk_full[s]); ++sw.issued[kLdQK][s]; }
}

// Warm L2 with chunk c's tiles, so that its loads, issued once their ring slots
// free up, find the data close by.
__device__ __forceinline__ void prefetch_chunk(const Ctx& x, const Maps& maps, int c) {
    if (c >= x.nchunks) return;
    const int tc = (int)(x.bos + (int64_t)c * C);
    tma_prefetch_l2_3d(&maps.a, 0, x.h, tc);
    tma_prefetch_l2_3d(&maps.v, 0, x.h, tc);
    tma_prefetch_l2_3d(&maps.v, 64, x.h, tc);
    tma_prefetch_l2_3d(&maps.k, 0, x.h, tc);
    tma_prefetch_l2_3d(&maps.k, 64, x.h, tc);
    tma_prefetch_l2_3d(&maps.q, 0, x.h, tc);
    tma_prefetch_l2_3d(&maps.q, 64, x.h, tc);
}

// ============================ group A: team P loop ===============================
// Team P (warps 0-3): chunk n's beta, the decay-range check, the Khat / Qhat / Kb
// tiles and the Gram product, committed to gram_done[n % 2]; a token-by-token
// chunk arrives there directly with mode 1.  Slot reuse: the A slot waits for
// W'/U of chunk n-2 (its loads), Kb / P / beta / gamma for chunk n-2's state
// product (kbp_free), and the Gram columns for chunk n-2's W' read, which comes
// before that product.
__device__ __noinline__ bool run_team_p(const Ctx& x_in, const __nv_bfloat16* __restrict__ beta) {
    const Ctx x = x_in;
    Small& sw = *x.sw;
    const int t = lt();
    bool ok = true, issued = false;
    float braw_next = (t < C && x.bos + t < x.eos && KDA_INDEX_OK((x.bos + t) * x.H + x.h, x.T * x.H, x.status))
                          ? bf2f(beta[(x.bos + t) * x.H + x.h]) : 0.f;
    KDA_PHASE_INIT;
    for (int n = 0; n < x.nchunks; ++n) {
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        const int64_t t0 = x.bos + (int64_t)n * C;
        const int L = (int)((x.eos - t0) < C ? (x.eos - t0) : C);
        const float braw = braw_next;                    // loaded one chunk ahead
        if (n + 1 < x.nchunks) {
            const int64_t tn = t0 + C + t;
            braw_next = (t < C && tn < x.eos && KDA_INDEX_OK(tn * x.H + x.h, x.T * x.H, x.status))
                            ? bf2f(beta[tn * x.H + x.h]) : 0.f;
        }
        uint8_t* aslot = x.sm + kA0 + s * kABytes;
        uint8_t* qk = x.sm + kQK0 + s * kQKBytes;
        uint8_t* kb = x.sm + kKB0 + s * 16384;

        if (!(ok = group_wait(kBarP, &sw.a_full[s], ph))) break;
        KDA_PHASE(0);
        if (t == 0) ++sw.consumed[kLdA][s];
        float gval = 0.f;
        const bool fast = build_suffix(reinterpret_cast<float*>(aslot), L, gval);
        KDA_PHASE(4);
        // Kb / P / beta / gamma and the q/k tiles of this slot are chunk n-2's until its state product
        if (n >= 2 && !(ok = group_wait(kBarP, &sw.kbp_free[s], ((n - 2) >> 1) & 1))) break;
        KDA_PHASE(2);
        if (t < C) sw.beta[s][t] = __float2bfloat16_rn((t < L) ? braw : 0.f);
        if (fast) sw.gam[s][t] = gval;
        if (!(ok = group_wait(kBarP, &sw.qk_full[s], ph))) break;
        KDA_PHASE(3);
        if (t == 0) ++sw.consumed[kLdQK][s];
        if (fast) build_tiles(qk, kb, reinterpret_cast<const float*>(aslot), L);
        if (!fast) {                                     // token-by-token chunk: no Gram product
            if (t == 0) {
                sw.mode[s] = 1;
                mbar_arrive(&sw.gram_done[s]);
            }
            continue;
        }
        group_publish(kBarP);
        KDA_PHASE(5);
        if (t == 0) {
            sw.mode[s] = 0;
            KDA_TRACE(n, 0);
            mma_gram(x.tb, tm_apw(s), smem_u32(qk), smem_u32(kb));
            mma_commit(&sw.gram_done[s]);
            issued = true;
        }
        KDA_PHASE(25);
    }
    if (t == 0 && issued) {   // let this thread's products land before TMEM is freed (bounded)
        mma_commit(&sw.drain_p);
        mbar_wait_bounded(&sw.drain_p, 0, kWaitLimitNs);
    }
    return ok;
}

// ============================ group A: team S loop ===============================
// Team S (warps 4-7): for chunk n, N and the masked P out of the Gram columns,
// the UT solve T, then (once V has landed and chunk n-2's output has left the U
// slot) W'^T = Khat^T T^T and U^T = V^T T^T; their commit is the second arrival
// on ready.  A token-by-token chunk only waits for its V tile.
__device__ __noinline__ bool run_team_s(const Ctx& x_in) {
    const Ctx x = x_in;
    Small& sw = *x.sw;
    const int t = lt();
    bool ok = true, issued = false;
    KDA_PHASE_INIT;
    for (int n = 0; n < x.nchunks; ++n) {
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        uint8_t* aslot = x.sm + kA0 + s * kABytes;
        uint8_t* qk = x.sm + kQK0 + s * kQKBytes;
        uint8_t* pp = x.sm + kPP0 + s * 8192;

        if (!(ok = group_wait(kBarS, &sw.gram_done[s], ph))) break;
        KDA_PHASE(26);
        if (sw.mode[s]) {                                // token-by-token chunk
            if (!(ok = group_wait(kBarS, &sw.v_full[s], ph))) break;
            if (t == 0) {
                ++sw.consumed[kLdV][s];
                mbar_arrive(&sw.ready[s]);
                mbar_arrive(&sw.ready[s]);
            }
            continue;
        }
        tc_fence_after();
        read_gram(x.tb, tm_apw(s), aslot, pp, sw.beta[s]);
        // the first solve step of each warp reads only the N rows that warp wrote (warp 0:
        // blocks 0, 1; warp 1: blocks 2, 3; warps 2 and 3 wrote P and go on to T's zero
        // blocks), so a warp barrier suffices here; the solve's own barriers order the rest
        fence_proxy_async_smem();
        __syncwarp();
        KDA_PHASE(6);
        solve_T(aslot, sw.beta[s], x.sw);
        KDA_PHASE(15);
        if (!(ok = group_wait(kBarS, &sw.v_full[s], ph))) break;
        if (t == 0) ++sw.consumed[kLdV][s];
        // the U slot still holds chunk n-2's output until group B has read it (every chunk,
        // tensor-core or token-by-token, completes one phase of its slot's u_free)
        if (n >= 2 && !(ok = group_wait(kBarS, &sw.u_free[s], ((n - 2) >> 1) & 1))) break;
        group_publish(kBarS);
        KDA_PHASE(7);
        if (t == 0) {                                    // W'^T and U^T; their commit is the 2nd arrival
            KDA_TRACE(n, 2);
            mbar_arrive(&sw.ready[s]);
            mma_wu(x.tb, tm_apw(s), tm_u(s), smem_u32(qk), smem_u32(x.sm + kV0 + s * kVBytes),
                   smem_u32(aslot + kTT));
            mma_commit(&sw.ready[s]);
            mma_commit(&sw.av_free[s]);
            issued = true;
        }
        KDA_PHASE(1);
    }
    if (t == 0 && issued) {
        mma_commit(&sw.drain_s);
        mbar_wait_bounded(&sw.drain_s, 0, kWaitLimitNs);
    }
    return ok;
}

// ============================ state/output issuer ================================
// One thread: for each chunk whose Delta group B has packed (slot in cmd_b),
// S^T += Delta^T Kb and O^T = Ss^T Qhat^T + Delta^T P^T, committed to mma2_done
// and to the Kb/P and q/k slot releases.  Group B publishes the next slot only
// after mma2_done, so cmd_b is read before it changes; -1 ends the loop.
__device__ __noinline__ bool run_out_issuer(const Ctx& x_in) {
    const Ctx x = x_in;
    Small& sw = *x.sw;
    bool ok = true, issued = false;
    uint32_t ph = 0;
    for (;;) {
        if (!(ok = mbar_wait_parked(&sw.packed, ph, kWaitLimitNs))) break;
        ph ^= 1u;
        const int s = sw.cmd_b;
        if (s < 0) break;
        tc_fence_after();
#ifdef KDA_DIAG_TRACE
        KDA_TRACE(sw.cmd_n, 6);
#endif
        mma_state_out(x.tb, tm_u(s), smem_u32(x.sm + kKB0 + s * 16384), smem_u32(x.sm + kQK0 + s * kQKBytes),
                      smem_u32(x.sm + kPP0 + s * 8192));
        mma_commit(&sw.mma2_done);
        mma_commit(&sw.kbp_free[s]);
        mma_commit(&sw.qk_free[s]);                      // Qhat read by the output product
        issued = true;
    }
    if (issued) {          // let this thread's products land before TMEM is freed (bounded)
        mma_commit(&sw.drain);
        mbar_wait_bounded(&sw.drain, 0, kWaitLimitNs);
    }
    return ok;
}

// Write the held output rows straight to global memory, rows [0, L) only.
// Lane pairs swap halves so each store is a 4-byte column pair; a warp store
// covers two 64-byte row segments.
__device__ __forceinline__ void o_store_direct(const uint32_t (&opk)[32], __nv_bfloat16* __restrict__ out,
                                               int64_t t0, int H, int h, int L, int64_t T, unsigned int* status) {
    (void)T; (void)status;                    // read by the index checks of bounds-checked builds
    const int t = lt();
    const bool odd = t & 1;
    const int col = t & ~1;
    __nv_bfloat16* base = out + ((size_t)t0 * H + h) * D + col;
    const size_t rs = (size_t)H * D;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t mine = opk[i];
        const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? (mine & 0xffffu) : (mine >> 16), 1);
        const uint32_t word = odd ? (got | (mine & 0xffff0000u)) : ((mine & 0xffffu) | (got << 16));
        const int r = 2 * i + (odd ? 1 : 0);
        if (r < L && KDA_INDEX_OK(((t0 + r) * H + h) * D + col + 1, T * H * D, status))
            __stcs(reinterpret_cast<unsigned int*>(base + (size_t)r * rs), word);
    }
}

// Full 64-row tile: each warp stages its 32 value channels (64 B per row,
// row-major, no swizzle) and issues its own TMA store.  Even lanes write even
// rows, odd lanes odd rows, so a warp's 32 stores hit 32 distinct banks.
__device__ __forceinline__ void o_store_warp_tma(const uint32_t (&opk)[32], uint8_t* stg_all, const Maps& maps,
                                                 int64_t t0, int h) {
    const int t = lt();
    const int lane = t & 31, wq = t >> 5;
    const bool odd = t & 1;
    uint8_t* stg = stg_all + wq * 4096;
    const uint32_t cb = (uint32_t)(lane & ~1) * 2;
    staging_ready();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t mine = opk[i];
        const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? (mine & 0xffffu) : (mine >> 16), 1);
        const uint32_t word = odd ? (got | (mine & 0xffff0000u)) : ((mine & 0xffffu) | (got << 16));
        const int r = 2 * i + (odd ? 1 : 0);
        *reinterpret_cast<uint32_t*>(stg + r * 64 + cb) = word;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(&maps.o, 32 * wq, h, (int)t0, stg);
        bulk_commit();
    }
}

// Store the output a chunk left in its U slot, then release that U slot to
// team S (one arrival per warp, once its TMEM reads are done).
__device__ __forceinline__ void flush_prev(const Ctx& x, const Maps& maps, __nv_bfloat16* out, int prev_s,
                                           int64_t prev_t0, int prev_L) {
    uint32_t opk[32];
    o_to_regs(x.tb, tm_u(prev_s), opk);
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&x.sw->u_free[prev_s]);
    if (prev_L == C)
        o_store_warp_tma(opk, x.sm + kWT, maps, prev_t0, x.h);
    else
        o_store_direct(opk, out, prev_t0, x.H, x.h, prev_L, x.T, x.status);
}

// ============================ producer warp ======================================
// One thread issues every TMA load: chunks 0 and 1 up front, then chunk n into
// slot n % 2 as soon as that slot's last reader for chunk n-2 is done.  Each
// chunk is prefetched into L2 two chunks ahead of its loads.
__device__ __noinline__ void run_producer(const Ctx& x_in, const Maps& maps) {
    const Ctx x = x_in;
    Small& sw = *x.sw;
    for (int c = 0; c < 2 && c < x.nchunks; ++c) refill(x, maps, c, c, true, true, true);
    prefetch_chunk(x, maps, 2);
    prefetch_chunk(x, maps, 3);
    KDA_PHASE_INIT;
    for (int n = 2; n < x.nchunks; ++n) {
        const int s = n & 1;
        const uint32_t ph = ((n - 2) >> 1) & 1;
        if (!mbar_wait_parked(&sw.av_free[s], ph, kWaitLimitNs)) return;
        KDA_PHASE(18);
        refill(x, maps, n, s, true, true, false);
        KDA_PHASE(19);
        if (!mbar_wait_parked(&sw.qk_free[s], ph, kWaitLimitNs)) return;
        KDA_PHASE(20);
        refill(x, maps, n, s, false, false, true);
        prefetch_chunk(x, maps, n + 2);
        KDA_PHASE(21);
    }
}

// ============================ group B loop =======================================
__device__ __noinline__ bool run_group_b(const Ctx& x_in, const Maps& maps, __nv_bfloat16* __restrict__ out,
                            const float* __restrict__ h0, float* __restrict__ hT, size_t sbase,
                            const int32_t* ck_cu, const int32_t* ck_pos, float* ck_states) {
    const Ctx x = x_in;
    Small& sw = *x.sw;
    Ckpt ck;
    ck.init(ck_cu, ck_pos, ck_states, x.seq, x.num_seqs, x.H, x.status);
    const int t = lt();
    const bool leader = (t == 0);
    uint32_t m1_ph = 0, m2_ph = 0;
    bool mma1_pending = false;
    // the previous chunk's output waits in its U slot until the next Delta product is in flight
    bool have_prev = false;
    int prev_s = 0, prev_L = 0;
    int64_t prev_t0 = 0;
    const int64_t state_lim = (int64_t)x.num_seqs * x.H * D * D;
    load_state(x.tb, h0, sbase, state_lim, x.status);
    const uint32_t sWT = smem_u32(x.sm + kWT);
    bool ok = true;
    KDA_PHASE_INIT;
    for (int n = 0; n < x.nchunks; ++n) {
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        const int64_t t0 = x.bos + (int64_t)n * C;
        const int L = (int)((x.eos - t0) < C ? (x.eos - t0) : C);
        uint8_t* aslot = x.sm + kA0 + s * kABytes;
        uint8_t* qk = x.sm + kQK0 + s * kQKBytes;
        uint8_t* vs = x.sm + kV0 + s * kVBytes;

        if (!(ok = group_wait(kBarB, &sw.ready[s], ph))) break;
        KDA_PHASE(8);
        tc_fence_after();
        if (sw.mode[s]) {                                // token-by-token chunk (tiles already landed)
            if (have_prev) {
                flush_prev(x, maps, out, prev_s, prev_t0, prev_L);
                have_prev = false;
            }
            token_chunk(x.tb, reinterpret_cast<float*>(aslot), qk, vs, sw.beta[s], tm_u(s), L);
            tc_fence_before();
            group_sync(kBarB);
            tc_fence_after();
            ck.after_chunk(x.tb, t0 + L - x.bos, t0 + L == x.eos, x.H, x.h);
            if (leader) {                                // the U slot is released when its output is stored
                mbar_arrive(&sw.kbp_free[s]);
                mbar_arrive(&sw.av_free[s]);
                mbar_arrive(&sw.qk_free[s]);
            }
            have_prev = true; prev_s = s; prev_L = L; prev_t0 = t0;
            continue;
        }
        decay_state(x.tb, sw.gam[s]);
        KDA_PHASE(9);
        read_w(x.tb, tm_apw(s), x.sm + kWT);
        group_publish(kBarB);
        KDA_PHASE(10);
        if (leader) {
            KDA_TRACE(n, 4);
            mma_delta(x.tb, tm_u(s), sWT);
            KDA_PHASE(24);
            mma_commit(&sw.mma1_done);
        }
        mma1_pending = true;
        if (!(ok = group_wait(kBarB, &sw.mma1_done, m1_ph))) break;
        m1_ph ^= 1u; mma1_pending = false;
        KDA_PHASE(11);
        tc_fence_after();
        pack_delta(x.tb, tm_u(s));
        group_publish(kBarB);
        KDA_PHASE(12);
        if (leader) {                                    // the state/output issuer takes it from here
#ifdef KDA_DIAG_TRACE
            sw.cmd_n = n;
#endif
            sw.cmd_b = s;
            mbar_arrive(&sw.packed);
        }
        KDA_PHASE(22);
        if (have_prev) {                                 // previous output, under this chunk's MMAs
            flush_prev(x, maps, out, prev_s, prev_t0, prev_L);
            have_prev = false;
        }
        KDA_PHASE(16);
        if (!(ok = group_wait(kBarB, &sw.mma2_done, m2_ph))) break;
        m2_ph ^= 1u;
        KDA_PHASE(13);
        tc_fence_after();
        ck.after_chunk(x.tb, t0 + L - x.bos, t0 + L == x.eos, x.H, x.h);
        have_prev = true; prev_s = s; prev_L = L; prev_t0 = t0;
        tc_fence_before();
        group_sync(kBarB);
        tc_fence_after();
        KDA_PHASE(14);
    }
    if (ok) {
        if (have_prev) flush_prev(x, maps, out, prev_s, prev_t0, prev_L);
        if (hT) store_state(x.tb, hT, sbase, state_lim, x.status);
    } else if (mma1_pending) {
        mbar_wait_bounded(&sw.mma1_done, m1_ph, kWaitLimitNs);
    }
    if (leader) {                                    // end of the state/output issuer's loop
        sw.cmd_b = -1;
        mbar_arrive(&sw.packed);
    }
    if ((t & 31) == 0) bulk_wait_all();              // tile stores complete before the block exits
    return ok;
}

#ifdef KDA_DIAG_TRACE
// Diagnostic build only: lane 0 of an extra warp of block 0 probes, without
// blocking, the completion barriers of the four product groups of each chunk
// (Gram; W' and U; Delta; state and output), following every phase from chunk
// 0 on, and records the clock at which it first sees each group of a traced
// chunk complete (events 1, 3, 5, 7; the matching issue events 0, 2, 4, 6 are
// taken by the issuing threads).  It stops once the traced chunks are done,
// once group B has ended and a pass finds nothing new, or after kWaitLimitNs.
__device__ void run_observer(const Ctx& x) {
    if (blockIdx.x != 0 || (threadIdx.x & 31) != 0) return;
    Small& sw = *x.sw;
    const int last = sw.trace_first + kTraceChunks;
    const int nch = x.nchunks < last ? x.nchunks : last;
    int next[4] = {0, 0, 0, 0};
    const uint64_t t0 = globaltimer_ns();
    bool b_done = false;
    for (;;) {
        bool pending = false, progress = false;
        for (int g = 0; g < 4; ++g) {
            const int n = next[g];
            if (n >= nch) continue;
            pending = true;
            uint64_t* bar = g == 0 ? &sw.gram_done[n & 1]
                          : g == 1 ? &sw.ready[n & 1]
                          : g == 2 ? &sw.mma1_done : &sw.mma2_done;
            const uint32_t par = g < 2 ? (uint32_t)((n >> 1) & 1) : (uint32_t)(n & 1);
            if (mbar_test(bar, par)) {
                if (trace_chunk(sw, n)) sw.trace[n - sw.trace_first][2 * g + 1] = (uint32_t)clock64();
                ++next[g];
                progress = true;
            }
        }
        if (!pending || (b_done && !progress)) break;
        if (*reinterpret_cast<volatile int*>(&sw.cmd_b) == -1) b_done = true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        // sleep between passes so the watched block keeps its issue slots and shared-memory
        // pipe (a spinning watcher slowed it by 6%); a stamp can then trail its completion
        __nanosleep(32);
    }
}
#endif

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ Maps maps, const __nv_bfloat16* __restrict__ beta,
                const float* __restrict__ h0, const int32_t* __restrict__ cu,
                __nv_bfloat16* __restrict__ out, float* __restrict__ hT, int64_t T, int num_seqs,
                int H, unsigned int* status, const int32_t* __restrict__ ck_cu,
                const int32_t* __restrict__ ck_pos, float* __restrict__ ck_states) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    Small* sw = reinterpret_cast<Small*>(sm + kSmall);
    const int tid = threadIdx.x;
    Ctx x;
    x.sm = sm;
    x.sw = sw;
    x.H = H;
    x.h = blockIdx.x % H;
    const int n = blockIdx.x / H;
    x.seq = n;
    x.T = T;
    x.num_seqs = num_seqs;
    x.status = status;
    seq_bounds(cu, n, num_seqs, T, x.bos, x.eos);
    x.nchunks = (int)((x.eos - x.bos + C - 1) / C);
    const size_t sbase = ((size_t)n * H + x.h) * D * D;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sw->qk_full[s], 1);
            mbar_init(&sw->v_full[s], 1);
            mbar_init(&sw->a_full[s], 1);
            mbar_init(&sw->ready[s], 2);
            mbar_init(&sw->kbp_free[s], 1);
        }
        mbar_init(&sw->gram_done[0], 1);
        mbar_init(&sw->gram_done[1], 1);
        mbar_init(&sw->mma1_done, 1);
        mbar_init(&sw->mma2_done, 1);
        mbar_init(&sw->av_free[0], 1);
        mbar_init(&sw->av_free[1], 1);
        mbar_init(&sw->qk_free[0], 1);
        mbar_init(&sw->qk_free[1], 1);
        mbar_init(&sw->u_free[0], 4);
        mbar_init(&sw->u_free[1], 4);
        mbar_init(&sw->packed, 1);
        mbar_init(&sw->drain, 1);
        mbar_init(&sw->drain_p, 1);
        mbar_init(&sw->drain_s, 1);
        fence_mbar_init();
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
        tma_prefetch_desc(&maps.a);
        tma_prefetch_desc(&maps.o);
        for (int k = 0; k < 3; ++k)
            for (int s = 0; s < 2; ++s) sw->issued[k][s] = sw->consumed[k][s] = 0;
        sw->cmd_b = 0;
#ifdef KDA_DIAG_TRACE
        for (int i = 0; i < kTraceChunks * kTraceEvents; ++i) sw->trace[i / kTraceEvents][i % kTraceEvents] = 0u;
        sw->trace_first = g_trace_first;
#endif
#ifdef KDA_PHASE_TIMING
        for (int i = 0; i < 32; ++i) sw->phase[i] = 0;
#endif
    }
    if ((tid >> 5) == 0) {
        tmem_alloc(&sw->tmem_base, kTmCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    x.tb = sw->tmem_base;

    bool ok = true;
    if (in_team_p())
        ok = run_team_p(x, beta);
    else if (in_group_a())
        ok = run_team_s(x);
    else if (tid < kProducer)
        ok = run_group_b(x, maps, out, h0, hT, sbase, ck_cu, ck_pos, ck_states);
    else if (tid == kProducer)
        run_producer(x, maps);

    else if (tid == kIssuerOut)
        ok = run_out_issuer(x);
#ifdef KDA_DIAG_TRACE
    else if (tid >= kObserver)
        run_observer(x);
#endif
    if (!ok && lt() == 0) atomicOr(status, kStatusTimeout);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {   // let any copy still in flight land before the block exits (bounded)
        uint64_t* bars[3] = {sw->qk_full, sw->v_full, sw->a_full};
        for (int k = 0; k < 3; ++k)
            for (int s = 0; s < 2; ++s)
                if (sw->issued[k][s] > sw->consumed[k][s])
                    mbar_wait_bounded(&bars[k][s], (uint32_t)(sw->consumed[k][s] & 1), kWaitLimitNs);
    }
    __syncthreads();
#ifdef KDA_PHASE_TIMING
    if (tid < 32) atomicAdd(&g_phase_cycles[tid], sw->phase[tid]);
#endif
#ifdef KDA_DIAG_TRACE
    if (blockIdx.x == 0 && tid < kTraceChunks * kTraceEvents)
        g_trace[tid / kTraceEvents][tid % kTraceEvents] = sw->trace[tid / kTraceEvents][tid % kTraceEvents];
#endif
    if ((tid >> 5) == 0) tmem_dealloc(x.tb, kTmCols);
}

// ============================ host side ==========================================
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    // looked up once (a function-local static is initialised once, even under concurrent calls)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return nullptr;
    }();
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

#ifdef KDA_DIAG_TRACE
// Diagnostic build: copy block 0's event trace (kTraceChunks x kTraceEvents clocks).
extern "C" int kda_debug_trace(uint32_t* host_trace) {
    return cudaMemcpyFromSymbol(host_trace, g_trace, sizeof(g_trace)) == cudaSuccess ? 0 : -1;
}
// Diagnostic build: the first chunk of the traced window of later launches (>= 0).
extern "C" int kda_debug_set_trace_first(int first) {
    if (first < 0) return -1;
    return cudaMemcpyToSymbol(g_trace_first, &first, sizeof(int)) == cudaSuccess ? 0 : -1;
}
#endif
#ifdef KDA_PHASE_TIMING
extern "C" int kda_debug_phase_cycles(unsigned long long* host16, int reset) {
    if (cudaMemcpyFromSymbol(host16, g_phase_cycles, 32 * sizeof(unsigned long long)) != cudaSuccess)
        return -1;
    if (reset) {
        unsigned long long z[32] = {};
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
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&maps.o, a.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, 32,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    // the shared-memory opt-in is a per-device property of the kernel
    // (setting it twice from two host threads is harmless; the flags are atomic)
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemDynamic);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    const unsigned blocks = (unsigned)((int64_t)a.num_seqs * a.H);
    chunk_tc_kernel<<<blocks, kThreads, kSmemDynamic, s>>>(
        maps, static_cast<const __nv_bfloat16*>(a.beta), a.initial_state, a.cu_seqlens,
        static_cast<__nv_bfloat16*>(a.out), a.final_state, a.total_tokens, a.num_seqs, a.H, a.status,
        a.ckpt_cu, a.ckpt_pos, a.ckpt_states);
    return cudaGetLastError();
}

}  // namespace kda
