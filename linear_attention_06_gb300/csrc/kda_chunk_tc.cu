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
#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdint.h>

#include "kda_chunk_common.cuh"
#include "kda_internal.h"
#include "sm103_primitives.cuh"

namespace kda {
namespace {

using namespace sm103;

// group A: two teams of 128 threads (P: operands and Gram, S: UT solve and W'/U), group B:
// 128 threads, then two single-thread warps: the TMA producer and the issuer of the
// state/output products
constexpr int kTeam = 128, kGroupA = 2 * kTeam, kGroupB = 128, kProducer = kGroupA + kGroupB,
              kIssuerOut = kProducer + 32;
constexpr int kThreads = 448;
__device__ __forceinline__ bool in_group_a() { return threadIdx.x < kGroupA; }
__device__ __forceinline__ bool in_team_p() { return threadIdx.x < kTeam; }

// ---- dynamic shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t kQK0 = 0;          // 2 x 32 KB: [k_h0 | q_h0 | k_h1 | q_h1], 64 rows x 128 B, SW128
constexpr uint32_t kV0 = 65536;       // 2 x 16 KB: [v_h0 | v_h1]
constexpr uint32_t kA0 = 98304;       // 2 x 32 KB: log_alpha fp32 [64][128]; then solve scratch + T
constexpr uint32_t kKB0 = 163840;     // 2 x 16 KB: Kb [halves]
constexpr uint32_t kPP0 = 196608;     // 2 x 8 KB: masked P, K-major
constexpr uint32_t kWT = 212992;      // 16 KB: W'^T (MN-major), then 4 x 4 KB output staging tiles
constexpr uint32_t kSmall = 229376;   // 2 KB: barriers, flags, beta, gamma
constexpr uint32_t kSmemUsed = kSmall + 2048;
constexpr uint32_t kSmemDynamic = kSmemUsed + 1024;   // + alignment slack = 232448
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
    int order_seq, order_pad[3];                 // the sequence this block takes (longest first)
    int issued[3][2];                            // TMA loads issued / waited for, per
    int consumed[3][2];                          //   (kind, slot), to drain after a timeout
    __nv_bfloat16 beta[2][C];                    // bf16 inputs: exact
    float gam[2][D];
};
static_assert(sizeof(Small) <= 2048, "small area");
static_assert(offsetof(Small, gam) % 16 == 0, "gamma rows are read as float4");
static_assert(offsetof(Small, beta) % 16 == 0, "beta is read eight at a time");

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

// The layer's front end, for the instance that reads the raw projections (FRONT): the raw
// q, k, v (bf16, for the convolution's halo rows), the conv taps [H][128][W] fp32, W in
// 1..4 and the L2 norm's eps.  The TMA maps of that instance point at the raw tensors.
struct Front {
    const __nv_bfloat16* q_raw;
    const __nv_bfloat16* k_raw;
    const __nv_bfloat16* v_raw;
    const float* conv_q;
    const float* conv_k;
    const float* conv_v;
    int W;
    float eps;
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
// With FRONT, the tiles that land are the raw projections: before the build the team turns
// the decay logits into log alpha (a column per thread), the beta logits into beta, and
// q, k, v into the recurrence inputs (convolution + SiLU down a channel pair per thread,
// then the L2 norm of each q and k row), all in place.
template <bool FRONT>
__device__ __noinline__ bool run_team_p(const Ctx& x_in, const __nv_bfloat16* __restrict__ beta, const Front fe) {
    const Ctx x = x_in;
    Small& sw = *x.sw;
    const int t = lt();
    bool ok = true, issued = false;
    // front end: thread t convolves channel pair (t & 63) of k (t < 64) or q (t >= 64) down
    // all rows, then pair (t & 63) of v down rows [32 (t >> 6), 32 (t >> 6) + 32)
    const int fpair = t & 63, fc0 = 2 * fpair;
    const bool fq = t >= 64;
    ConvTaps tap_qk, tap_v;
    if constexpr (FRONT) {
        tap_qk = load_taps(fq ? fe.conv_q : fe.conv_k, x.h, D, fc0, fe.W);
        tap_v = load_taps(fe.conv_v, x.h, D, fc0, fe.W);
    }
    auto qk_pair_off = [fq, fc0](int r) { return qk_off(fq, (uint32_t)r, (uint32_t)fc0); };
    auto v_pair_off = [fc0](int r) { return half_off((uint32_t)r, (uint32_t)fc0); };
    float braw_next = (t < C && x.bos + t < x.eos && KDA_INDEX_OK((x.bos + t) * x.H + x.h, x.T * x.H, x.status))
                          ? bf2f(beta[(x.bos + t) * x.H + x.h]) : 0.f;
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
        float2 hq0, hq1, hq2, hv0, hv1, hv2;           // the convolution's halo (raw rows before its first row)
        if constexpr (FRONT) {
            conv_halo(fq ? fe.q_raw : fe.k_raw, t0, x.bos, x.H, x.h, D, fc0, hq0, hq1, hq2);
            if (!fq) conv_halo(fe.v_raw, t0, x.bos, x.H, x.h, D, fc0, hv0, hv1, hv2);
        }

        if (!(ok = group_wait(kBarP, &sw.a_full[s], ph))) break;
        if (t == 0) ++sw.consumed[kLdA][s];
        if constexpr (FRONT) {
            logsigmoid_col(reinterpret_cast<float*>(aslot), t, L);   // thread t: column t
            group_sync(kBarP);                           // build_suffix reads other threads' columns
        }
        float gval = 0.f;
        const bool fast = build_suffix(reinterpret_cast<float*>(aslot), L, gval);
        // Kb / P / beta / gamma and the q/k tiles of this slot are chunk n-2's until its state product
        if (n >= 2 && !(ok = group_wait(kBarP, &sw.kbp_free[s], ((n - 2) >> 1) & 1))) break;
        if (t < C) sw.beta[s][t] = __float2bfloat16_rn((t < L) ? (FRONT ? sigmoid_f(braw) : braw) : 0.f);
        if (fast) sw.gam[s][t] = gval;
        if (!(ok = group_wait(kBarP, &sw.qk_full[s], ph))) break;
        if (t == 0) ++sw.consumed[kLdQK][s];
        if constexpr (FRONT) {
            conv_silu_pair<C>(qk, qk_pair_off, 0, L, tap_qk, hq0, hq1, hq2);
            group_sync(kBarP);
            l2norm_row(qk + (fq ? 8192 : 0), fpair, fe.eps);   // thread t: row t & 63 of k or q
            if (!(ok = group_wait(kBarP, &sw.v_full[s], ph))) break;
            uint8_t* vt = x.sm + kV0 + s * kVBytes;
            if (fq) {                                    // rows 32-63: the halo is rows 29-31, still raw
                hv0 = unpack_bf16x2(*reinterpret_cast<const uint32_t*>(vt + v_pair_off(29)));
                hv1 = unpack_bf16x2(*reinterpret_cast<const uint32_t*>(vt + v_pair_off(30)));
                hv2 = unpack_bf16x2(*reinterpret_cast<const uint32_t*>(vt + v_pair_off(31)));
            }
            group_sync(kBarP);                           // every halo read before any row is written
            conv_silu_pair<C / 2>(vt, v_pair_off, fq ? 32 : 0, L, tap_v, hv0, hv1, hv2);
            group_sync(kBarP);
        }
        if (fast) build_tiles(qk, kb, reinterpret_cast<const float*>(aslot), L);
        if (!fast) {                                     // token-by-token chunk: no Gram product
            if (t == 0) {
                sw.mode[s] = 1;
                mbar_arrive(&sw.gram_done[s]);
            }
            continue;
        }
        group_publish(kBarP);
        if (t == 0) {
            sw.mode[s] = 0;
            mma_gram(x.tb, tm_apw(s), smem_u32(qk), smem_u32(kb));
            mma_commit(&sw.gram_done[s]);
            issued = true;
        }
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
    for (int n = 0; n < x.nchunks; ++n) {
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        uint8_t* aslot = x.sm + kA0 + s * kABytes;
        uint8_t* qk = x.sm + kQK0 + s * kQKBytes;
        uint8_t* pp = x.sm + kPP0 + s * 8192;

        if (!(ok = group_wait(kBarS, &sw.gram_done[s], ph))) break;
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
        solve_T(aslot, sw.beta[s]);
        if (!(ok = group_wait(kBarS, &sw.v_full[s], ph))) break;
        if (t == 0) ++sw.consumed[kLdV][s];
        // the U slot still holds chunk n-2's output until group B has read it (every chunk,
        // tensor-core or token-by-token, completes one phase of its slot's u_free)
        if (n >= 2 && !(ok = group_wait(kBarS, &sw.u_free[s], ((n - 2) >> 1) & 1))) break;
        group_publish(kBarS);
        if (t == 0) {                                    // W'^T and U^T; their commit is the 2nd arrival
            mbar_arrive(&sw.ready[s]);
            mma_wu(x.tb, tm_apw(s), tm_u(s), smem_u32(qk), smem_u32(x.sm + kV0 + s * kVBytes),
                   smem_u32(aslot + kTT));
            mma_commit(&sw.ready[s]);
            mma_commit(&sw.av_free[s]);
            issued = true;
        }
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
    for (int n = 2; n < x.nchunks; ++n) {
        const int s = n & 1;
        const uint32_t ph = ((n - 2) >> 1) & 1;
        if (!mbar_wait_parked(&sw.av_free[s], ph, kWaitLimitNs)) return;
        refill(x, maps, n, s, true, true, false);
        if (!mbar_wait_parked(&sw.qk_free[s], ph, kWaitLimitNs)) return;
        refill(x, maps, n, s, false, false, true);
        prefetch_chunk(x, maps, n + 2);
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
    for (int n = 0; n < x.nchunks; ++n) {
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        const int64_t t0 = x.bos + (int64_t)n * C;
        const int L = (int)((x.eos - t0) < C ? (x.eos - t0) : C);
        uint8_t* aslot = x.sm + kA0 + s * kABytes;
        uint8_t* qk = x.sm + kQK0 + s * kQKBytes;
        uint8_t* vs = x.sm + kV0 + s * kVBytes;

        if (!(ok = group_wait(kBarB, &sw.ready[s], ph))) break;
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
        read_w(x.tb, tm_apw(s), x.sm + kWT);
        group_publish(kBarB);
        if (leader) {
            mma_delta(x.tb, tm_u(s), sWT);
            mma_commit(&sw.mma1_done);
        }
        mma1_pending = true;
        if (!(ok = group_wait(kBarB, &sw.mma1_done, m1_ph))) break;
        m1_ph ^= 1u; mma1_pending = false;
        tc_fence_after();
        pack_delta(x.tb, tm_u(s));
        group_publish(kBarB);
        if (leader) {                                    // the state/output issuer takes it from here
            sw.cmd_b = s;
            mbar_arrive(&sw.packed);
        }
        if (have_prev) {                                 // previous output, under this chunk's MMAs
            flush_prev(x, maps, out, prev_s, prev_t0, prev_L);
            have_prev = false;
        }
        if (!(ok = group_wait(kBarB, &sw.mma2_done, m2_ph))) break;
        m2_ph ^= 1u;
        tc_fence_after();
        ck.after_chunk(x.tb, t0 + L - x.bos, t0 + L == x.eos, x.H, x.h);
        have_prev = true; prev_s = s; prev_L = L; prev_t0 = t0;
        tc_fence_before();
        group_sync(kBarB);
        tc_fence_after();
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


// Blocks start in index order, so with sequences of mixed lengths the block of sequence slot r
// takes the sequence of rank r by length (longest first, ties by index): the long sequences
// start in the first wave and the last wave holds short ones.  All threads; `scratch` holds
// the lengths.  Up to kOrderMax sequences (a few hundred cycles a block); beyond that the
// natural order.
constexpr int kOrderMax = 256;
__device__ int seq_by_length(const int32_t* cu, int num_seqs, int64_t T, int r, uint8_t* scratch, int* slot) {
    int64_t* len = reinterpret_cast<int64_t*>(scratch);
    for (int i = threadIdx.x; i < num_seqs; i += blockDim.x) {
        int64_t b, e;
        seq_bounds(cu, i, num_seqs, T, b, e);
        len[i] = e - b;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < num_seqs; i += blockDim.x) {
        const int64_t li = len[i];
        int rank = 0;
        for (int j = 0; j < num_seqs; ++j) {
            const int64_t lj = len[j];
            rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
        }
        if (rank == r) *slot = i;
    }
    __syncthreads();
    return *slot;
}

template <bool FRONT>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ Maps maps, const __nv_bfloat16* __restrict__ beta,
                const float* __restrict__ h0, const int32_t* __restrict__ cu,
                __nv_bfloat16* __restrict__ out, float* __restrict__ hT, int64_t T, int num_seqs,
                int H, unsigned int* status, const int32_t* __restrict__ ck_cu,
                const int32_t* __restrict__ ck_pos, float* __restrict__ ck_states, const Front fe) {
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
    const int n = (cu && num_seqs > 1 && num_seqs <= kOrderMax)
                      ? seq_by_length(cu, num_seqs, T, (int)(blockIdx.x / H), sm + kWT, &sw->order_seq)
                      : (int)(blockIdx.x / H);
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
        ok = run_team_p<FRONT>(x, beta, fe);
    else if (in_group_a())
        ok = run_team_s(x);
    else if (tid < kProducer)
        ok = run_group_b(x, maps, out, h0, hT, sbase, ck_cu, ck_pos, ck_states);
    else if (tid == kProducer)
        run_producer(x, maps);

    else if (tid == kIssuerOut)
        ok = run_out_issuer(x);
    if (!ok && (tid & 31) == 0) atomicOr(status, kStatusTimeout);

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
    if ((tid >> 5) == 0) tmem_dealloc(x.tb, kTmCols);
}

}  // namespace


bool chunk_tc_supported(const PrefillArgs& a) {
    return a.dtype == DType::BF16 && a.dk == D && a.dv == D && a.total_tokens > 0 &&
           encode_fn() != nullptr;
}

namespace {
// Maps, shared-memory opt-in and launch of one instance (q, k, v, log_alpha, beta are the
// raw projections for FRONT).
template <bool FRONT>
cudaError_t launch_instance(const PrefillArgs& a, const Front& fe, cudaStream_t s) {
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
        cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel<FRONT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemDynamic);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    const unsigned blocks = (unsigned)((int64_t)a.num_seqs * a.H);
    chunk_tc_kernel<FRONT><<<blocks, kThreads, kSmemDynamic, s>>>(
        maps, static_cast<const __nv_bfloat16*>(a.beta), a.initial_state, a.cu_seqlens,
        static_cast<__nv_bfloat16*>(a.out), a.final_state, a.total_tokens, a.num_seqs, a.H, a.status,
        a.ckpt_cu, a.ckpt_pos, a.ckpt_states, fe);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_chunk_tc_prefill(const PrefillArgs& a, cudaStream_t s) {
    return launch_instance<false>(a, Front{}, s);
}

cudaError_t launch_chunk_tc_frontend(const PrefillArgs& a, const FrontendArgs& f, cudaStream_t s) {
    const Front fe{static_cast<const __nv_bfloat16*>(f.q_raw), static_cast<const __nv_bfloat16*>(f.k_raw),
                   static_cast<const __nv_bfloat16*>(f.v_raw), f.conv_q, f.conv_k, f.conv_v, f.conv_width, f.eps};
    return launch_instance<true>(a, fe, s);
}

}  // namespace kda
