// kda_chunk_split.cu -- the chunkwise prefill split into two kernels, for inputs
// with few (sequence, head) pairs and long sequences.
//
// The fused kernel (kda_chunk_tc.cu) gives each (sequence, head) one SM, so one
// 131,072-token sequence with 32 heads keeps 32 of the 152 SMs busy.  Everything a
// chunk needs that does not depend on the state entering it (the decayed factors,
// the Gram products, the UT solve, W' and U; "Kimi K3 Architecture Teardown",
// section "Hybrid Attention for 1M Tokens": the chunk's products of
// (I - beta k k^T) Diag(alpha) folded into a WY form) is independent across chunks,
// so here it runs first, over every chunk of every head at once:
//
//   chunk_local_kernel  (one CTA per SM, each walking a share of the (head, chunk)
//                        items): team P builds Khat / Qhat / Kb and issues the Gram
//                        product, team S reads it back, solves for T and issues
//                        W'^T = Khat^T T^T and U^T = V^T T^T, team E writes the
//                        chunk's record to the workspace (TMA stores);
//   chunk_chain_kernel  (one CTA per (sequence, head)): walks the records in order
//                        and carries the fp32 state in TMEM through
//                        Delta = U - W' Ss, O = Qhat Ss + (mask o P) Delta,
//                        S <- Ss + Kb^T Delta, with Ss = Diag(e^G) S.
//
// A record (one per (head, chunk slot)) holds, in 8 KB units: Qhat (2 units, the two
// 64-channel halves), Kb (2), -W'^T as [128 key channels][64 tokens] (2), the masked P
// (1), e^G per key channel (512 B in one unit) and U^T in fp32 as two halves of
// [128 value channels][32 tokens] (4 units).  A chunk whose decay leaves the factored
// range (some |G| > 60) has no record: its mode word says so, and the chain kernel
// runs it token by token from the inputs themselves.  Records of sequence n start at
// slot floor(bos_n / 64) + n, so a head needs ceil(T / 64) + N slots whatever the
// lengths (kda_prefill_split_workspace_size).
//
// The chain kernel holds two record slots and loads each record in two parts: part A (Kb,
// -W'^T, e^G, U^T) is read up to the state update, part B (Qhat, P) by the output products,
// so part A of chunk n + 2 is loaded as soon as chunk n's state update has landed instead of
// after its output products (4.43 against 4.58 ms for one 131,072-token sequence).
#include <atomic>
#include <mutex>

#include "kda_chunk_common.cuh"

namespace kda {
namespace {

// ---- record layout
constexpr uint32_t kUnit = 8192;
constexpr int kRecUnits = 12;
constexpr uint32_t kRecBytes = kRecUnits * kUnit;           // 98304
constexpr int kUQh = 0, kUKb = 2, kUWt = 4, kUP = 6, kUSmall = 7, kUU = 8;
constexpr uint32_t kGamBytes = D * 4;
// one record's bytes moved by the chain kernel's loads, in two parts: A (Kb, -W'^T, e^G, U^T) is
// read up to the state update, B (Qhat, P) by the output products
constexpr uint32_t kRecLoadBytesA = 4 * kUnit + kGamBytes + 4 * kUnit;
constexpr uint32_t kRecLoadBytesB = 3 * kUnit;
constexpr uint32_t kRawLoadBytes = kQKBytes + kVBytes + kABytes;   // q, k, v, log_alpha tiles

struct RecMaps {
    CUtensorMap t16;   // bf16 8 KB units: {64 elements, 64 rows, unit}, 128-byte swizzle
    CUtensorMap t32;   // U^T halves: {32 floats, 128 rows, 16 KB unit}, 128-byte swizzle
};

// Workspace: H * R int32 mode words (1 = token-by-token chunk), padded to 1 KB, then
// H * R records.
struct Workspace {
    int* modes;
    uint8_t* recs;
    int R;             // record slots per head
};

// Chunk of the packed batch behind record slot r of a head (sequence n, tokens
// [t0, t0 + L)); false for a slot that holds no chunk.  The record slot of chunk k of
// sequence n is floor(bos_n / 64) + n + k, strictly increasing over (n, k).
struct Seqs {
    const int32_t* cu;
    int num_seqs;
    int64_t T;
    int R;
    __device__ __forceinline__ int rec0(int n, int64_t& bos, int64_t& eos) const {
        seq_bounds(cu, n, num_seqs, T, bos, eos);
        return (int)(bos >> 6) + n;
    }
    __device__ bool chunk_of(int r, int& n, int64_t& t0, int& L) const {
        int64_t b, e;
        if (num_seqs <= 0 || rec0(0, b, e) > r) return false;
        int lo = 0, hi = num_seqs - 1;                   // largest n with rec0(n) <= r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (rec0(mid, b, e) <= r) lo = mid; else hi = mid - 1;
        }
        n = lo;
        const int r0 = rec0(n, b, e);
        t0 = b + (int64_t)(r - r0) * C;
        if (t0 >= e) return false;
        L = (int)((e - t0) < C ? (e - t0) : C);
        return true;
    }
};

// One (head, chunk) item of the chunk-local kernel.
struct Item {
    int h;
    int64_t t0;
    int L;
    int rec;           // h * R + slot
};

// The chunk-local CTA's share of the H * R (head, slot) items, walked in order; each role
// of the CTA walks the same valid items in the same order.
struct Items {
    Seqs seqs;
    int i1;
    __device__ int next(int i, Item& it) const {
        for (; i < i1; ++i) {
            const int h = i / seqs.R, r = i - h * seqs.R;
            int n;
            if (seqs.chunk_of(r, n, it.t0, it.L)) {
                it.h = h;
                it.rec = i;
                return i;
            }
        }
        return i1;
    }
};

// ============================ chunk-local kernel =================================
// Threads: team P (warps 0-3), team S (warps 4-7), team E (warps 8-11), the TMA
// producer (warp 12, one thread); warp 13 idles (the chain kernel uses 14 warps too).
constexpr int kLocalThreads = 448;
constexpr int kLocalProducer = 384;
constexpr int kBarE = 2;   // named barrier of team E (the id the fused kernel gives group B)

// shared memory: the fused kernel's slots, with -W'^T staged in kWTl and U^T in the
// chunk's log_alpha slot once W' and U are computed
constexpr uint32_t kQKl = 0, kVl = 65536, kAl = 98304, kKBl = 163840, kPPl = 196608, kWTl = 212992,
                   kSmallL = 229376;
constexpr uint32_t kLocalSmem = kSmallL + 2048 + 1024;

struct LocalSmall {
    uint64_t qk_full[2], v_full[2], a_full[2];   // TMA completions
    uint64_t gram_done[2];                       // team P -> team S
    uint64_t ready[2];                           // team S -> team E: W', U computed (2 arrivals)
    uint64_t kbp_free[2];                        // team E -> team P: Kb / P / beta / gamma / Gram-W' slot free
    uint64_t av_free[2];                         // team E -> producer: log_alpha / v slot free
    uint64_t qk_free[2];                         // team E -> producer: q / k slot free
    uint64_t u_free[2];                          // team E -> team S: U slot of TMEM read
    uint64_t drain_p, drain_s;
    uint32_t tmem_base;
    int mode[2];
    int issued[3][2], consumed[3][2];
    alignas(16) __nv_bfloat16 beta[2][C];
    alignas(16) float gam[2][D];
};
static_assert(sizeof(LocalSmall) <= 2048, "small area");
static_assert(offsetof(LocalSmall, gam) % 16 == 0, "gamma rows are read as float4");
static_assert(offsetof(LocalSmall, beta) % 16 == 0, "beta is read eight at a time");

struct LocalCtx {
    uint8_t* sm;
    LocalSmall* sw;
    uint32_t tb;
    Items items;
    int i0;
    int H;
    int64_t T;
    unsigned int* status;
};

// Team P: as the fused kernel's team P, over the CTA's items.
__device__ __noinline__ bool run_local_p(const LocalCtx& x_in, const __nv_bfloat16* __restrict__ beta) {
    const LocalCtx x = x_in;
    LocalSmall& sw = *x.sw;
    const int t = lt();
    bool ok = true, issued = false;
    Item it, nx;
    int i = x.items.next(x.i0, it);
    float braw_next = 0.f;
    if (i < x.items.i1 && t < it.L) {
        const int64_t e = (it.t0 + t) * x.H + it.h;
        braw_next = KDA_INDEX_OK(e, x.T * x.H, x.status) ? bf2f(beta[e]) : 0.f;
    }
    for (int n = 0; i < x.items.i1; ++n) {
        const int j = x.items.next(i + 1, nx);
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        const int L = it.L;
        const float braw = braw_next;                    // loaded one item ahead
        if (j < x.items.i1) {
            braw_next = 0.f;
            if (t < nx.L) {
                const int64_t e = (nx.t0 + t) * x.H + nx.h;
                braw_next = KDA_INDEX_OK(e, x.T * x.H, x.status) ? bf2f(beta[e]) : 0.f;
            }
        }
        uint8_t* aslot = x.sm + kAl + s * kABytes;
        uint8_t* qk = x.sm + kQKl + s * kQKBytes;
        uint8_t* kb = x.sm + kKBl + s * 16384;

        if (!(ok = group_wait(kBarP, &sw.a_full[s], ph))) break;
        if (t == 0) ++sw.consumed[0][s];
        float gval = 0.f;
        const bool fast = build_suffix(reinterpret_cast<float*>(aslot), L, gval);
        if (n >= 2 && !(ok = group_wait(kBarP, &sw.kbp_free[s], ((n - 2) >> 1) & 1))) break;
        if (t < C) sw.beta[s][t] = __float2bfloat16_rn((t < L) ? braw : 0.f);
        if (fast) sw.gam[s][t] = gval;
        if (!(ok = group_wait(kBarP, &sw.qk_full[s], ph))) break;
        if (t == 0) ++sw.consumed[1][s];
        if (fast) build_tiles(qk, kb, reinterpret_cast<const float*>(aslot), L);
        if (!fast) {
            if (t == 0) {
                sw.mode[s] = 1;
                mbar_arrive(&sw.gram_done[s]);
            }
        } else {
            group_publish(kBarP);
            if (t == 0) {
                sw.mode[s] = 0;
                mma_gram(x.tb, tm_apw(s), smem_u32(qk), smem_u32(kb));
                mma_commit(&sw.gram_done[s]);
                issued = true;
            }
        }
        it = nx;
        i = j;
    }
    if (t == 0 && issued) {
        mma_commit(&sw.drain_p);
        mbar_wait_bounded(&sw.drain_p, 0, kWaitLimitNs);
    }
    return ok;
}

// Team S: as the fused kernel's team S, over the CTA's items; the U slot of TMEM is free
// again once team E has read the item two back.
__device__ __noinline__ bool run_local_s(const LocalCtx& x_in) {
    const LocalCtx x = x_in;
    LocalSmall& sw = *x.sw;
    const int t = lt();
    bool ok = true, issued = false;
    Item it;
    int i = x.items.next(x.i0, it);
    for (int n = 0; i < x.items.i1; ++n, i = x.items.next(i + 1, it)) {
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        uint8_t* aslot = x.sm + kAl + s * kABytes;
        uint8_t* qk = x.sm + kQKl + s * kQKBytes;
        uint8_t* pp = x.sm + kPPl + s * 8192;

        if (!(ok = group_wait(kBarS, &sw.gram_done[s], ph))) break;
        if (sw.mode[s]) {                                // token-by-token chunk: no products
            if (!(ok = group_wait(kBarS, &sw.v_full[s], ph))) break;
            if (t == 0) {
                ++sw.consumed[2][s];
                mbar_arrive(&sw.ready[s]);
                mbar_arrive(&sw.ready[s]);
            }
            continue;
        }
        tc_fence_after();
        read_gram(x.tb, tm_apw(s), aslot, pp, sw.beta[s]);
        fence_proxy_async_smem();
        __syncwarp();
        solve_T(aslot, sw.beta[s]);
        if (!(ok = group_wait(kBarS, &sw.v_full[s], ph))) break;
        if (t == 0) ++sw.consumed[2][s];
        if (n >= 2 && !(ok = group_wait(kBarS, &sw.u_free[s], ((n - 2) >> 1) & 1))) break;
        group_publish(kBarS);
        if (t == 0) {
            mbar_arrive(&sw.ready[s]);
            mma_wu(x.tb, tm_apw(s), tm_u(s), smem_u32(qk), smem_u32(x.sm + kVl + s * kVBytes),
                   smem_u32(aslot + kTT));
            mma_commit(&sw.ready[s]);
            issued = true;
        }
    }
    if (t == 0 && issued) {
        mma_commit(&sw.drain_s);
        mbar_wait_bounded(&sw.drain_s, 0, kWaitLimitNs);
    }
    return ok;
}

// U^T (lane j = value channel, 64 token columns, fp32 in TMEM) to shared memory as two
// halves of [128 rows][32 floats] in the 128-byte swizzle (the layout the record's TMA
// map stores and loads).
__device__ void stage_u(uint32_t tb, uint32_t col, uint8_t* dst) {
    const int j = lt();
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[32];
        tmem_ld32(tmem_addr(tb, lane0(), col + 32 * hf), v);
        tmem_wait_ld();
        uint8_t* row = dst + hf * 16384 + j * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(row + ((c ^ (j & 7)) << 4)) =
                make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    }
}

// -W'^T (lane c of the W' columns, fp32) as bf16 into the MN-major staging tile; team E's
// stores of the previous item were waited for before its slots were released, so no wait here.
__device__ void stage_w(uint32_t tb, uint32_t col, uint8_t* wt) {
    const int c = lt();
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

// Team E: writes each item's record (or marks it token-by-token), then hands the slots
// back.  Qhat, Kb and P are final in shared memory once W' and U are computed, so their
// stores go out first and overlap the read-out of W' and U from TMEM; the q/k and Kb / P
// slots are handed back as soon as those first stores have read them.
__device__ __noinline__ bool run_local_e(const LocalCtx& x_in, const RecMaps& rm, const Workspace ws) {
    const LocalCtx x = x_in;
    LocalSmall& sw = *x.sw;
    const int t = lt();
    bool ok = true;
    Item it;
    int i = x.items.next(x.i0, it);
    for (int n = 0; i < x.items.i1; ++n, i = x.items.next(i + 1, it)) {
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        uint8_t* aslot = x.sm + kAl + s * kABytes;
        uint8_t* qk = x.sm + kQKl + s * kQKBytes;
        if (!(ok = group_wait(kBarE, &sw.ready[s], ph))) break;
        tc_fence_after();
        const int mode = sw.mode[s];
        const int u0 = it.rec * kRecUnits;
        if (t == 0) {
            ws.modes[it.rec] = mode;
            if (!mode) {
                tma_store_3d(&rm.t16, 0, 0, u0 + kUQh, qk + 8192);
                tma_store_3d(&rm.t16, 0, 0, u0 + kUQh + 1, qk + 24576);
                tma_store_3d(&rm.t16, 0, 0, u0 + kUKb, x.sm + kKBl + s * 16384);
                tma_store_3d(&rm.t16, 0, 0, u0 + kUKb + 1, x.sm + kKBl + s * 16384 + 8192);
                tma_store_3d(&rm.t16, 0, 0, u0 + kUP, x.sm + kPPl + s * 8192);
                bulk_commit();
            }
        }
        if (mode) {                                      // nothing to store: the chain reads the inputs
            group_sync(kBarE);
            if (t == 0) {
                mbar_arrive(&sw.kbp_free[s]);
                mbar_arrive(&sw.av_free[s]);
                mbar_arrive(&sw.qk_free[s]);
                mbar_arrive(&sw.u_free[s]);
            }
            continue;
        }
        stage_w(x.tb, tm_apw(s), x.sm + kWTl);           // -W'^T, bf16
        stage_u(x.tb, tm_u(s), aslot);                   // U^T, fp32, over log_alpha / the solve area
        float* gdst = reinterpret_cast<float*>(ws.recs + (size_t)it.rec * kRecBytes + kUSmall * kUnit);
        gdst[t] = sw.gam[s][t];
        fence_proxy_async_smem();
        tc_fence_before();
        group_sync(kBarE);
        if (t == 0) {
            mbar_arrive(&sw.u_free[s]);                  // W' and U are out of TMEM
            tma_store_3d(&rm.t16, 0, 0, u0 + kUWt, x.sm + kWTl);
            tma_store_3d(&rm.t16, 0, 0, u0 + kUWt + 1, x.sm + kWTl + 8192);
            tma_store_3d(&rm.t32, 0, 0, it.rec * (kRecUnits / 2) + kUU / 2, aslot);
            tma_store_3d(&rm.t32, 0, 0, it.rec * (kRecUnits / 2) + kUU / 2 + 1, aslot + 16384);
            bulk_commit();
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");   // Qhat, Kb, P read
            mbar_arrive(&sw.qk_free[s]);
            mbar_arrive(&sw.kbp_free[s]);
            bulk_wait_read();                            // -W'^T and U^T read
            mbar_arrive(&sw.av_free[s]);
        }
    }
    if ((t & 31) == 0) bulk_wait_all();
    return ok;
}

// TMA loads of one item into slot s (issued by the producer thread).
__device__ __forceinline__ void local_refill(const LocalCtx& x, const Maps& maps, const Item& it, int s,
                                             bool av, bool q) {
    LocalSmall& sw = *x.sw;
    const int tc = (int)it.t0;
    if (av) {
        uint8_t* a = x.sm + kAl + s * kABytes;
        uint8_t* v = x.sm + kVl + s * kVBytes;
        mbar_arrive_expect_tx(&sw.a_full[s], kABytes);
        tma_load_3d(a, &maps.a, 0, it.h, tc, &sw.a_full[s]);
        ++sw.issued[0][s];
        mbar_arrive_expect_tx(&sw.v_full[s], kVBytes);
        tma_load_3d(v, &maps.v, 0, it.h, tc, &sw.v_full[s]);
        tma_load_3d(v + 8192, &maps.v, 64, it.h, tc, &sw.v_full[s]);
        ++sw.issued[2][s];
    }
    if (q) {
        uint8_t* d = x.sm + kQKl + s * kQKBytes;
        mbar_arrive_expect_tx(&sw.qk_full[s], kQKBytes);
        tma_load_3d(d + 0, &maps.k, 0, it.h, tc, &sw.qk_full[s]);
        tma_load_3d(d + 8192, &maps.q, 0, it.h, tc, &sw.qk_full[s]);
        tma_load_3d(d + 16384, &maps.k, 64, it.h, tc, &sw.qk_full[s]);
        tma_load_3d(d + 24576, &maps.q, 64, it.h, tc, &sw.qk_full[s]);
        ++sw.issued[1][s];
    }
}

__device__ __noinline__ void run_local_producer(const LocalCtx& x_in, const Maps& maps) {
    const LocalCtx x = x_in;
    LocalSmall& sw = *x.sw;
    Item it;
    int i = x.items.next(x.i0, it);
    for (int n = 0; i < x.items.i1; ++n, i = x.items.next(i + 1, it)) {
        const int s = n & 1;
        if (n >= 2) {
            const uint32_t ph = ((n - 2) >> 1) & 1;
            if (!mbar_wait_parked(&sw.av_free[s], ph, kWaitLimitNs)) return;
            local_refill(x, maps, it, s, true, false);
            if (!mbar_wait_parked(&sw.qk_free[s], ph, kWaitLimitNs)) return;
            local_refill(x, maps, it, s, false, true);
        } else {
            local_refill(x, maps, it, s, true, true);
        }
    }
}

__global__ void __launch_bounds__(kLocalThreads, 1)
chunk_local_kernel(const __grid_constant__ Maps maps, const __grid_constant__ RecMaps rm,
                   const __nv_bfloat16* __restrict__ beta, const int32_t* __restrict__ cu, int64_t T,
                   int num_seqs, int H, Workspace ws, int per_cta, unsigned int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    LocalSmall* sw = reinterpret_cast<LocalSmall*>(sm + kSmallL);
    const int tid = threadIdx.x;
    LocalCtx x;
    x.sm = sm;
    x.sw = sw;
    x.H = H;
    x.T = T;
    x.status = status;
    x.items.seqs = Seqs{cu, num_seqs, T, ws.R};
    const int64_t total = (int64_t)H * ws.R;
    const int64_t a = (int64_t)blockIdx.x * per_cta;
    x.i0 = (int)(a < total ? a : total);
    x.items.i1 = (int)(a + per_cta < total ? a + per_cta : total);

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sw->qk_full[s], 1);
            mbar_init(&sw->v_full[s], 1);
            mbar_init(&sw->a_full[s], 1);
            mbar_init(&sw->gram_done[s], 1);
            mbar_init(&sw->ready[s], 2);
            mbar_init(&sw->kbp_free[s], 1);
            mbar_init(&sw->av_free[s], 1);
            mbar_init(&sw->qk_free[s], 1);
            mbar_init(&sw->u_free[s], 1);
        }
        mbar_init(&sw->drain_p, 1);
        mbar_init(&sw->drain_s, 1);
        fence_mbar_init();
        for (int k = 0; k < 3; ++k)
            for (int s = 0; s < 2; ++s) sw->issued[k][s] = sw->consumed[k][s] = 0;
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
    if (tid < 128)
        ok = run_local_p(x, beta);
    else if (tid < 256)
        ok = run_local_s(x);
    else if (tid < kLocalProducer)
        ok = run_local_e(x, rm, ws);
    else if (tid == kLocalProducer)
        run_local_producer(x, maps);
    if (!ok && (tid & 31) == 0) atomicOr(status, kStatusTimeout);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {   // let any copy still in flight land before the block exits (bounded)
        uint64_t* bars[3] = {sw->a_full, sw->qk_full, sw->v_full};
        for (int k = 0; k < 3; ++k)
            for (int s = 0; s < 2; ++s)
                if (sw->issued[k][s] > sw->consumed[k][s])
                    mbar_wait_bounded(&bars[k][s], (uint32_t)(sw->consumed[k][s] & 1), kWaitLimitNs);
    }
    __syncthreads();
    if ((tid >> 5) == 0) tmem_dealloc(x.tb, kTmCols);
}

// ============================ state-chain kernel =================================
// Threads: group B (warps 0-7; warps w and w + 4 share TMEM lane quarter w % 4 and
// split the columns), team F (warps 8-11: output rows out of TMEM and to HBM), the
// record producer (warp 12, one thread) and the product issuer (warp 13, one thread).
constexpr int kChainThreads = 448;
constexpr int kChainF = 256, kChainProducer = 384, kChainIssuer = 416;
constexpr int kBarB8 = 4, kBarF = 5;   // named barriers: all of group B (256 threads); team F
constexpr int kBarB4 = 2;              // warps 0-3 of group B (the 128-thread helpers use it)

// shared memory: two record slots of 96 KB (a token-by-token chunk's q/k, v and
// log_alpha tiles land in the same slot at 0, 32 KB and 64 KB), the output staging
// tiles, the small area
constexpr uint32_t kSlot0 = 0, kStg = 2 * kRecBytes, kSmallC = kStg + 16384;
constexpr uint32_t kChainSmem = kSmallC + 2048 + 1024;
// TMEM, by chunk parity d: S^T (fp32) 0-127; bf16 Ss^T at 128 + 64 d; Delta, then O, at 256 + 64 d;
// bf16 Delta^T at 384 + 32 d.  With the bf16 operands in two copies, chunk n + 1's decay and
// pack can run while chunk n's output product still reads chunk n's copies.
__device__ __forceinline__ uint32_t tm_d(int d) { return 256u + 64u * d; }
__device__ __forceinline__ uint32_t tm_sbf(int d) { return 128u + 64u * d; }
__device__ __forceinline__ uint32_t tm_dbf(int d) { return 384u + 32u * d; }

struct ChainSmall {
    uint64_t rec_full[2];      // producer -> all: the slot's part A (or raw tiles) landed
    uint64_t rec_free[2];      // part A read by its last reader (the state update)
    uint64_t rec_full_b[2];    // producer -> issuer: part B landed (a plain arrival for raw tiles)
    uint64_t rec_free_b[2];    // part B read by its last reader (the output products)
    uint64_t decayed;          // group B -> issuer: Ss and its bf16 copy in TMEM
    uint64_t packed;           // group B -> issuer: Delta packed
    uint64_t mma1, mma2;       // issuer -> group B: Delta product; state update
    uint64_t o_ready[2];       // chunk output in TMEM slot d
    uint64_t d_free[2];        // team F read the output of slot d (4 warps)
    uint64_t drain;
    uint32_t tmem_base;
    int mode[2];
    int issued[2];             // loads the producer issued into each slot (part A / raw tiles)
    int issued_b[2];           // phases of rec_full_b the producer started
    alignas(16) __nv_bfloat16 beta[2][C];  // token-by-token chunks only
};
static_assert(sizeof(ChainSmall) <= 2048, "small area");
static_assert(offsetof(ChainSmall, beta) % 16 == 0, "beta is read eight at a time");

struct ChainCtx {
    uint8_t* sm;
    ChainSmall* sw;
    uint32_t tb;
    int64_t bos, eos;
    int nchunks, H, h, seq, rec_base;   // rec_base: h * R + first slot of the sequence
    int64_t T;
    int num_seqs, R;
    unsigned int* status;
};

__device__ __forceinline__ bool group8_and(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, 256, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(kBarB8)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void group8_sync() { asm volatile("bar.sync %0, 256;" ::"n"(kBarB8) : "memory"); }
__device__ __forceinline__ bool group8_wait(uint64_t* bar, uint32_t parity) {
    return group8_and(mbar_wait_bounded(bar, parity, kWaitLimitNs));
}
__device__ __forceinline__ void group8_publish() {
    fence_proxy_async_smem();
    tc_fence_before();
    group8_sync();
    tc_fence_after();
}

// S^T <- S^T Diag(gam) (fp32) and its bf16 copy at column sbf, for the 64 key channels of
// this warp's half (warps 0-3 channels 0-63, warps 4-7 channels 64-127), both 32-column
// blocks in flight at once.
__device__ void chain_decay(uint32_t tb, const float* gam, uint32_t sbf) {
    const int c0 = 64 * ((threadIdx.x >> 7) & 1);
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
        uint32_t v[32], pk[16];
        tmem_ld32(tmem_addr(tb, lane0(), kTmS + c0 + 32 * h), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 g = *reinterpret_cast<const float4*>(gam + c0 + 32 * h + 4 * i);
            v[4 * i + 0] = __float_as_uint(__uint_as_float(v[4 * i + 0]) * g.x);
            v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) * g.y);
            v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) * g.z);
            v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) * g.w);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        tmem_st32(tmem_addr(tb, lane0(), kTmS + c0 + 32 * h), v);
        tmem_st16(tmem_addr(tb, lane0(), sbf + c0 / 2 + 16 * h), pk);
    }
    tmem_wait_st();
}

// Delta^T (fp32, lane j = value channel) plus U^T from the record, packed to bf16 at column
// dbf as the A operand of the state and output products.  Warps 0-3 take token columns 0-31,
// warps 4-7 columns 32-63.
__device__ void pack_delta_u(uint32_t tb, uint32_t dcol, const uint8_t* ut, uint32_t dbf) {
    const int j = lt(), hf = (threadIdx.x >> 7) & 1;
    uint32_t v[32], pk[16];
    tmem_ld32(tmem_addr(tb, lane0(), dcol + 32 * hf), v);
    tmem_wait_ld();
    const uint8_t* row = ut + hf * 16384 + j * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 u = *reinterpret_cast<const float4*>(row + ((c ^ (j & 7)) << 4));
        v[4 * c + 0] = __float_as_uint(__uint_as_float(v[4 * c + 0]) + u.x);
        v[4 * c + 1] = __float_as_uint(__uint_as_float(v[4 * c + 1]) + u.y);
        v[4 * c + 2] = __float_as_uint(__uint_as_float(v[4 * c + 2]) + u.z);
        v[4 * c + 3] = __float_as_uint(__uint_as_float(v[4 * c + 3]) + u.w);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    tmem_st16(tmem_addr(tb, lane0(), dbf + 16 * hf), pk);
    tmem_wait_st();
}

// Delta^T = Ss^T (-W'^T) into TMEM slot dcol (a fresh accumulator; U is added in the pack).
__device__ __forceinline__ void mma_delta_fresh(uint32_t tb, uint32_t dcol, uint32_t sbf, uint32_t sWT) {
    constexpr uint32_t idw = idesc_bf16_f32(128, 64, false, true);
#pragma unroll
    for (uint32_t ks = 0; ks < 8; ++ks)
        mma_ts(tb + dcol, tb + sbf + ks * 8, smem_desc(sWT + ks * 2048, 16384, 1024, kSwizzle128B), idw,
               ks > 0);
}

// S^T += Delta^T Kb (the next chunk waits for this one only).
__device__ __forceinline__ void mma_state_rec(uint32_t tb, uint32_t dbf, uint32_t sKB) {
    constexpr uint32_t ids = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
    for (uint32_t ks = 0; ks < 4; ++ks)
        mma_ts(tb + kTmS, tb + dbf + ks * 8, smem_desc(sKB + ks * 2048, 8192, 1024, kSwizzle128B), ids, 1);
}

// O^T = Ss^T Qhat^T + Delta^T P^T in slot ocol.  Qhat's halves sit 8 KB apart in a record slot.
__device__ __forceinline__ void mma_out_rec(uint32_t tb, uint32_t ocol, uint32_t sbf, uint32_t dbf, uint32_t sQh,
                                            uint32_t sPP) {
    constexpr uint32_t idq = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
    for (uint32_t ks = 0; ks < 8; ++ks)
        mma_ts(tb + ocol, tb + sbf + ks * 8,
               smem_desc(sQh + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, kSwizzle128B), idq, ks > 0);
#pragma unroll
    for (uint32_t ks = 0; ks < 4; ++ks)
        mma_ts(tb + ocol, tb + dbf + ks * 8, smem_desc(sPP + ks * 32, 16, 1024, kSwizzle128B), idq, 1);
}

// Group B: the state chain.  Warps 0-3 also load the initial state, save checkpoints and
// store the final state, and run token-by-token chunks.
__device__ __noinline__ bool run_chain_b(const ChainCtx& x_in, const __nv_bfloat16* __restrict__ beta,
                                         const float* __restrict__ h0, float* __restrict__ hT, size_t sbase,
                                         const int32_t* ck_cu, const int32_t* ck_pos, float* ck_states) {
    const ChainCtx x = x_in;
    ChainSmall& sw = *x.sw;
    const int t = lt();
    const bool lower = threadIdx.x < 128;                // warps 0-3
    Ckpt ck;
    ck.init(ck_cu, ck_pos, ck_states, x.seq, x.num_seqs, x.H, x.status);
    const int64_t state_lim = (int64_t)x.num_seqs * x.H * D * D;
    if (lower) load_state(x.tb, h0, sbase, state_lim, x.status);
    tc_fence_before();
    group8_sync();
    tc_fence_after();
    uint32_t m_ph = 0;
    bool ok = true;
    for (int n = 0; n < x.nchunks; ++n) {
        const int s = n & 1, d = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        const int64_t t0 = x.bos + (int64_t)n * C;
        const int L = (int)((x.eos - t0) < C ? (x.eos - t0) : C);
        uint8_t* slot = x.sm + kSlot0 + s * kRecBytes;
        if (!(ok = group8_wait(&sw.rec_full[s], ph))) break;
        tc_fence_after();
        if (sw.mode[s]) {                                // token by token, from the input tiles
            // the output goes to TMEM slot d: team F must have read the chunk two back
            if (n >= 2 && !(ok = group8_wait(&sw.d_free[d], ((n - 2) >> 1) & 1))) break;
            tc_fence_after();
            if (lower) {
                if (t < C) {
                    const int64_t e = (t0 + t) * x.H + x.h;
                    sw.beta[s][t] = (t < L && KDA_INDEX_OK(e, x.T * x.H, x.status)) ? beta[e]
                                                                                     : __float2bfloat16_rn(0.f);
                }
                group_sync(kBarB4);
                token_chunk(x.tb, reinterpret_cast<float*>(slot + 2 * kQKBytes), slot, slot + kQKBytes,
                            sw.beta[s], tm_d(d), L);
                tc_fence_before();
                group_sync(kBarB4);
                tc_fence_after();
                ck.after_chunk(x.tb, t0 + L - x.bos, t0 + L == x.eos, x.H, x.h);
            }
            tc_fence_before();
            group8_sync();
            if (t == 0 && lower) {
                mbar_arrive(&sw.o_ready[d]);
                mbar_arrive(&sw.rec_free[s]);
                mbar_arrive(&sw.rec_free_b[s]);
            }
            continue;
        }
        chain_decay(x.tb, reinterpret_cast<const float*>(slot + kUSmall * kUnit), tm_sbf(d));
        group8_publish();
        if (t == 0 && lower) mbar_arrive(&sw.decayed);
        if (!(ok = group8_wait(&sw.mma1, m_ph))) break;
        tc_fence_after();
        pack_delta_u(x.tb, tm_d(d), slot + kUU * kUnit, tm_dbf(d));
        group8_publish();
        if (t == 0 && lower) mbar_arrive(&sw.packed);
        if (!(ok = group8_wait(&sw.mma2, m_ph))) break;
        m_ph ^= 1u;
        tc_fence_after();
        if (lower) ck.after_chunk(x.tb, t0 + L - x.bos, t0 + L == x.eos, x.H, x.h);
        tc_fence_before();
        group8_sync();
        tc_fence_after();
    }
    if (ok && hT && lower) store_state(x.tb, hT, sbase, state_lim, x.status);
    return ok;
}

// Issuer: the Delta product once the decayed state is in place, the state and output
// products once Delta is packed.
__device__ __noinline__ bool run_chain_issuer(const ChainCtx& x_in) {
    const ChainCtx x = x_in;
    ChainSmall& sw = *x.sw;
    bool ok = true, issued = false;
    uint32_t m_ph = 0;
    for (int n = 0; n < x.nchunks; ++n) {
        const int s = n & 1, d = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        if (!(ok = mbar_wait_bounded(&sw.rec_full[s], ph, kWaitLimitNs))) break;
        if (sw.mode[s]) continue;                        // group B runs it
        const uint32_t slot = smem_u32(x.sm + kSlot0 + s * kRecBytes);
        if (!(ok = mbar_wait_bounded(&sw.decayed, m_ph, kWaitLimitNs))) break;
        if (n >= 2 && !(ok = mbar_wait_bounded(&sw.d_free[d], ((n - 2) >> 1) & 1, kWaitLimitNs))) break;
        tc_fence_after();
        mma_delta_fresh(x.tb, tm_d(d), tm_sbf(d), slot + kUWt * kUnit);
        mma_commit(&sw.mma1);
        issued = true;
        if (!(ok = mbar_wait_bounded(&sw.packed, m_ph, kWaitLimitNs))) break;
        tc_fence_after();
        mma_state_rec(x.tb, tm_dbf(d), slot + kUKb * kUnit);
        mma_commit(&sw.mma2);                            // the state chain goes on from here
        mma_commit(&sw.rec_free[s]);                     // part A: Delta, the pack and the update read it
        if (!(ok = mbar_wait_bounded(&sw.rec_full_b[s], ph, kWaitLimitNs))) break;
        mma_out_rec(x.tb, tm_d(d), tm_sbf(d), tm_dbf(d), slot + kUQh * kUnit, slot + kUP * kUnit);
        mma_commit(&sw.o_ready[d]);
        mma_commit(&sw.rec_free_b[s]);
        m_ph ^= 1u;
    }
    if (issued) {
        mma_commit(&sw.drain);
        mbar_wait_bounded(&sw.drain, 0, kWaitLimitNs);
    }
    return ok;
}

// Team F: each chunk's output rows out of TMEM (slot d) and to HBM.
__device__ __noinline__ bool run_chain_f(const ChainCtx& x_in, const Maps& maps, __nv_bfloat16* __restrict__ out) {
    const ChainCtx x = x_in;
    ChainSmall& sw = *x.sw;
    bool ok = true;
    for (int n = 0; n < x.nchunks; ++n) {
        const int d = n & 1;
        const int64_t t0 = x.bos + (int64_t)n * C;
        const int L = (int)((x.eos - t0) < C ? (x.eos - t0) : C);
        if (!(ok = group_and(kBarF, mbar_wait_bounded(&sw.o_ready[d], (n >> 1) & 1, kWaitLimitNs)))) break;
        tc_fence_after();
        uint32_t opk[32];
        o_to_regs(x.tb, tm_d(d), opk);
        tc_fence_before();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&sw.d_free[d]);
        if (L == C)
            o_store_warp_tma(opk, x.sm + kStg, maps, t0, x.h);
        else
            o_store_direct(opk, out, t0, x.H, x.h, L, x.T, x.status);
    }
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    return ok;
}

// Producer: chunk n's record (or, for a token-by-token chunk, its input tiles) into slot
// n % 2 once the chunk two back has left it.
__device__ __noinline__ void run_chain_producer(const ChainCtx& x_in, const Maps& maps, const RecMaps& rm,
                                                const Workspace ws) {
    const ChainCtx x = x_in;
    ChainSmall& sw = *x.sw;
    // a record slot outside the workspace (only a malformed cu_seqlens can ask for one) is
    // read as a token-by-token chunk from the inputs
    auto mode_of = [&](int n) -> int {
        return (n < x.nchunks && (x.rec_base - x.h * x.R) + n < x.R) ? ws.modes[x.rec_base + n] : 1;
    };
    auto prefetch = [&](int n) {
        if (n < x.nchunks && (x.rec_base - x.h * x.R) + n < x.R)
            bulk_prefetch_l2(ws.recs + (size_t)(x.rec_base + n) * kRecBytes, kRecBytes);
    };
    for (int n = 0; n < 4; ++n) prefetch(n);
    int mode_next = mode_of(0), mode_next2 = mode_of(1);
    for (int n = 0; n < x.nchunks; ++n) {
        const int s = n & 1;
        const int mode = mode_next;                      // read two chunks ahead
        mode_next = mode_next2;
        mode_next2 = mode_of(n + 2);
        prefetch(n + 4);
        const uint32_t fph = ((n - 2) >> 1) & 1;
        if (n >= 2 && !mbar_wait_bounded(&sw.rec_free[s], fph, kWaitLimitNs)) return;   // part A free
        const int rec = x.rec_base + n;
        sw.mode[s] = mode;
        uint8_t* slot = x.sm + kSlot0 + s * kRecBytes;
        uint64_t* bar = &sw.rec_full[s];
        if (mode == 0) {
            ++sw.issued[s];
            mbar_arrive_expect_tx(bar, kRecLoadBytesA);
            const int u0 = rec * kRecUnits;
#pragma unroll 1
            for (int u = kUKb; u < kUP; ++u) tma_load_3d(slot + u * kUnit, &rm.t16, 0, 0, u0 + u, bar);
            bulk_load_1d(slot + kUSmall * kUnit, ws.recs + (size_t)rec * kRecBytes + kUSmall * kUnit, kGamBytes,
                         bar);
            tma_load_3d(slot + kUU * kUnit, &rm.t32, 0, 0, rec * (kRecUnits / 2) + kUU / 2, bar);
            tma_load_3d(slot + kUU * kUnit + 16384, &rm.t32, 0, 0, rec * (kRecUnits / 2) + kUU / 2 + 1, bar);
            // part B once the output products of chunk n-2 have read the slot's Qhat and P
            if (n >= 2 && !mbar_wait_bounded(&sw.rec_free_b[s], fph, kWaitLimitNs)) return;
            uint64_t* bb = &sw.rec_full_b[s];
            ++sw.issued_b[s];
            mbar_arrive_expect_tx(bb, kRecLoadBytesB);
            tma_load_3d(slot + kUQh * kUnit, &rm.t16, 0, 0, u0 + kUQh, bb);
            tma_load_3d(slot + (kUQh + 1) * kUnit, &rm.t16, 0, 0, u0 + kUQh + 1, bb);
            tma_load_3d(slot + kUP * kUnit, &rm.t16, 0, 0, u0 + kUP, bb);
        } else {
            // the raw tiles cover the whole slot: part B must be free too; rec_full_b takes a plain
            // arrival (its previous phase, a load or an arrival, completed before that release)
            if (n >= 2 && !mbar_wait_bounded(&sw.rec_free_b[s], fph, kWaitLimitNs)) return;
            ++sw.issued[s];
            const int tc = (int)(x.bos + (int64_t)n * C);
            mbar_arrive_expect_tx(bar, kRawLoadBytes);
            tma_load_3d(slot + 0, &maps.k, 0, x.h, tc, bar);
            tma_load_3d(slot + 8192, &maps.q, 0, x.h, tc, bar);
            tma_load_3d(slot + 16384, &maps.k, 64, x.h, tc, bar);
            tma_load_3d(slot + 24576, &maps.q, 64, x.h, tc, bar);
            tma_load_3d(slot + kQKBytes, &maps.v, 0, x.h, tc, bar);
            tma_load_3d(slot + kQKBytes + 8192, &maps.v, 64, x.h, tc, bar);
            tma_load_3d(slot + 2 * kQKBytes, &maps.a, 0, x.h, tc, bar);
            ++sw.issued_b[s];
            mbar_arrive(&sw.rec_full_b[s]);
        }
    }
}

__global__ void __launch_bounds__(kChainThreads, 1)
chunk_chain_kernel(const __grid_constant__ Maps maps, const __grid_constant__ RecMaps rm,
                   const __nv_bfloat16* __restrict__ beta, const float* __restrict__ h0,
                   const int32_t* __restrict__ cu, __nv_bfloat16* __restrict__ out, float* __restrict__ hT,
                   int64_t T, int num_seqs, int H, Workspace ws, unsigned int* status,
                   const int32_t* __restrict__ ck_cu, const int32_t* __restrict__ ck_pos,
                   float* __restrict__ ck_states) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    ChainSmall* sw = reinterpret_cast<ChainSmall*>(sm + kSmallC);
    const int tid = threadIdx.x;
    ChainCtx x;
    x.sm = sm;
    x.sw = sw;
    x.H = H;
    x.h = blockIdx.x % H;
    const int n = blockIdx.x / H;
    x.seq = n;
    x.T = T;
    x.num_seqs = num_seqs;
    x.R = ws.R;
    x.status = status;
    const Seqs seqs{cu, num_seqs, T, ws.R};
    const int r0 = seqs.rec0(n, x.bos, x.eos);
    x.nchunks = (int)((x.eos - x.bos + C - 1) / C);
    x.rec_base = x.h * ws.R + r0;
    const size_t sbase = ((size_t)n * H + x.h) * D * D;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sw->rec_full[s], 1);
            mbar_init(&sw->rec_free[s], 1);
            mbar_init(&sw->rec_full_b[s], 1);
            mbar_init(&sw->rec_free_b[s], 1);
            sw->issued_b[s] = 0;
            mbar_init(&sw->o_ready[s], 1);
            mbar_init(&sw->d_free[s], 4);
            sw->issued[s] = 0;
        }
        mbar_init(&sw->decayed, 1);
        mbar_init(&sw->packed, 1);
        mbar_init(&sw->mma1, 1);
        mbar_init(&sw->mma2, 1);
        mbar_init(&sw->drain, 1);
        fence_mbar_init();
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
    if (tid < kChainF)
        ok = run_chain_b(x, beta, h0, hT, sbase, ck_cu, ck_pos, ck_states);
    else if (tid < kChainProducer)
        ok = run_chain_f(x, maps, out);
    else if (tid == kChainProducer)
        run_chain_producer(x, maps, rm, ws);
    else if (tid == kChainIssuer)
        ok = run_chain_issuer(x);
    if (!ok && (tid & 31) == 0) atomicOr(status, kStatusTimeout);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {   // every load the producer issued lands before the block exits (bounded)
        for (int s = 0; s < 2; ++s)
            if (sw->issued[s] > 0) mbar_wait_bounded(&sw->rec_full[s], (uint32_t)((sw->issued[s] - 1) & 1), kWaitLimitNs);
        for (int s = 0; s < 2; ++s)
            if (sw->issued_b[s] > 0)
                mbar_wait_bounded(&sw->rec_full_b[s], (uint32_t)((sw->issued_b[s] - 1) & 1), kWaitLimitNs);
    }
    __syncthreads();
    if ((tid >> 5) == 0) tmem_dealloc(x.tb, kTmCols);
}

// ============================ host side ==========================================
bool make_rec_maps(RecMaps* m, void* recs, int64_t nrec) {
    auto enc = encode_fn();
    if (!enc) return false;
    {
        cuuint64_t dims[3] = {64, 64, (cuuint64_t)nrec * kRecUnits};
        cuuint64_t strides[2] = {128, kUnit};
        cuuint32_t box[3] = {64, 64, 1}, es[3] = {1, 1, 1};
        if (enc(&m->t16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, recs, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        cuuint64_t dims[3] = {32, 128, (cuuint64_t)nrec * (kRecUnits / 2)};
        cuuint64_t strides[2] = {128, 2 * kUnit};
        cuuint32_t box[3] = {32, 128, 1}, es[3] = {1, 1, 1};
        if (enc(&m->t32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, recs, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

bool make_input_maps(Maps* maps, const PrefillArgs& a) {
    return make_map(&maps->q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&maps->k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&maps->v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&maps->a, a.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.total_tokens, a.H, 128,
                    CU_TENSOR_MAP_SWIZZLE_NONE) &&
           make_map(&maps->o, a.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.total_tokens, a.H, 32,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
}

int record_slots(int64_t T, int num_seqs) { return (int)((T + C - 1) / C) + num_seqs; }
size_t modes_bytes(int64_t slots) { return (size_t)((slots * 4 + 1023) / 1024) * 1024; }

// A long single sequence is run in time segments of kSegTokens: the chunk-local kernel of
// segment s + 1 (on a second stream, on the SMs the chains leave free) runs while the state
// chains of segment s run, the chains carrying the fp32 state from segment to segment through
// a workspace buffer.  Records then need room for two segments only.
constexpr int64_t kSegTokens = 8192;
bool segmented(int64_t T, int num_seqs, int H) { return num_seqs == 1 && H <= 64 && T >= 2 * kSegTokens; }
size_t carry_bytes(int H) { return (size_t)H * D * D * sizeof(float); }
size_t seg_buffer_bytes(int H) {
    const int64_t slots = (int64_t)H * record_slots(kSegTokens, 1);
    return modes_bytes(slots) + (size_t)slots * kRecBytes;
}

bool configure_kernels(int* sms) {
    static std::atomic<bool> attr_set[64];
    static std::atomic<int> sm_count[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(chunk_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kLocalSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(chunk_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kChainSmem);
        int n = 0;
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return false;
        sm_count[dev].store(n > 0 ? n : 1, std::memory_order_relaxed);
        attr_set[dev].store(true, std::memory_order_release);
    }
    *sms = sm_count[dev].load(std::memory_order_relaxed);
    return true;
}

// One chunk-local pass over all (head, record slot) items of a, spread over `grid` CTAs, and
// the state chains of a (one CTA per (sequence, head)), each on its own stream.
cudaError_t enqueue_local(const PrefillArgs& a, void* buf, int grid, cudaStream_t s) {
    Maps maps;
    if (!make_input_maps(&maps, a)) return cudaErrorInvalidValue;
    const int R = record_slots(a.total_tokens, a.num_seqs);
    const int64_t slots = (int64_t)a.H * R;
    Workspace ws;
    ws.R = R;
    ws.modes = static_cast<int*>(buf);
    ws.recs = static_cast<uint8_t*>(buf) + modes_bytes(slots);
    RecMaps rm;
    if (!make_rec_maps(&rm, ws.recs, slots)) return cudaErrorInvalidValue;
    const int64_t per = (slots + grid - 1) / grid;
    const int g = (int)((slots + per - 1) / per);
    chunk_local_kernel<<<g, kLocalThreads, kLocalSmem, s>>>(maps, rm, static_cast<const __nv_bfloat16*>(a.beta),
                                                           a.cu_seqlens, a.total_tokens, a.num_seqs, a.H, ws,
                                                           (int)per, a.status);
    return cudaGetLastError();
}
cudaError_t enqueue_chain(const PrefillArgs& a, void* buf, cudaStream_t s) {
    Maps maps;
    if (!make_input_maps(&maps, a)) return cudaErrorInvalidValue;
    const int R = record_slots(a.total_tokens, a.num_seqs);
    const int64_t slots = (int64_t)a.H * R;
    Workspace ws;
    ws.R = R;
    ws.modes = static_cast<int*>(buf);
    ws.recs = static_cast<uint8_t*>(buf) + modes_bytes(slots);
    RecMaps rm;
    if (!make_rec_maps(&rm, ws.recs, slots)) return cudaErrorInvalidValue;
    chunk_chain_kernel<<<(unsigned)((int64_t)a.num_seqs * a.H), kChainThreads, kChainSmem, s>>>(
        maps, rm, static_cast<const __nv_bfloat16*>(a.beta), a.initial_state, a.cu_seqlens,
        static_cast<__nv_bfloat16*>(a.out), a.final_state, a.total_tokens, a.num_seqs, a.H, ws, a.status,
        a.ckpt_cu, a.ckpt_pos, a.ckpt_states);
    return cudaGetLastError();
}

// The second stream and the events of the segmented run, one set per device, created on
// first use and kept.  The mutex keeps one call's enqueue sequence together, so the events'
// latest records are that call's (calls from several host threads serialise on the second
// stream).
struct SegResources {
    std::mutex mu;
    bool ready = false;
    cudaStream_t aux = nullptr;
    cudaEvent_t fork = nullptr, local_done[2] = {}, chain_done[2] = {};
};
SegResources& seg_resources(int dev) {
    static SegResources r[64];
    return r[dev];
}

cudaError_t launch_segmented(const PrefillArgs& a, void* workspace, int sms, cudaStream_t s) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    SegResources& r = seg_resources(dev);
    std::lock_guard<std::mutex> lock(r.mu);
    if (!r.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&r.aux, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.fork, cudaEventDisableTiming);
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            e = cudaEventCreateWithFlags(&r.local_done[b], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.chain_done[b], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) return e;
        r.ready = true;
    }
    uint8_t* base = static_cast<uint8_t*>(workspace);
    float* carry[2] = {reinterpret_cast<float*>(base), reinterpret_cast<float*>(base + carry_bytes(a.H))};
    uint8_t* bufs[2] = {base + 2 * carry_bytes(a.H), base + 2 * carry_bytes(a.H) + seg_buffer_bytes(a.H)};
    const int pairs = a.H;                            // one sequence
    const int local_grid = sms - pairs >= sms / 2 ? sms - pairs : sms / 2;
    const int64_t nseg = (a.total_tokens + kSegTokens - 1) / kSegTokens;
    const size_t row = (size_t)a.H * D;               // elements of one token row of q, k, v, out
    cudaError_t e = cudaEventRecord(r.fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(r.aux, r.fork, 0);
    for (int64_t sg = 0; sg < nseg && e == cudaSuccess; ++sg) {
        const int b = (int)(sg & 1);
        const int64_t t0 = sg * kSegTokens;
        PrefillArgs g = a;
        g.total_tokens = (a.total_tokens - t0 < kSegTokens) ? a.total_tokens - t0 : kSegTokens;
        g.q = static_cast<const __nv_bfloat16*>(a.q) + t0 * row;
        g.k = static_cast<const __nv_bfloat16*>(a.k) + t0 * row;
        g.v = static_cast<const __nv_bfloat16*>(a.v) + t0 * row;
        g.log_alpha = a.log_alpha + t0 * row;
        g.beta = static_cast<const __nv_bfloat16*>(a.beta) + t0 * a.H;
        g.out = static_cast<__nv_bfloat16*>(a.out) + t0 * row;
        g.cu_seqlens = nullptr;
        g.initial_state = sg == 0 ? a.initial_state : carry[b ^ 1];
        g.final_state = sg == nseg - 1 ? a.final_state : carry[b];
        // the records of buffer b are free once the chains of segment sg - 2 have read them
        if (sg >= 2) e = cudaStreamWaitEvent(r.aux, r.chain_done[b], 0);
        if (e == cudaSuccess) e = enqueue_local(g, bufs[b], sg == 0 ? sms : local_grid, r.aux);
        if (e == cudaSuccess) e = cudaEventRecord(r.local_done[b], r.aux);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, r.local_done[b], 0);
        if (e == cudaSuccess) e = enqueue_chain(g, bufs[b], s);
        if (e == cudaSuccess) e = cudaEventRecord(r.chain_done[b], s);
    }
    // every operation on the second stream precedes the last chain launch on s
    return e;
}

}  // namespace

size_t split_workspace_bytes(int64_t total_tokens, int num_seqs, int H, bool segments) {
    if (segments && segmented(total_tokens, num_seqs, H)) return 2 * carry_bytes(H) + 2 * seg_buffer_bytes(H);
    const int64_t slots = (int64_t)H * record_slots(total_tokens, num_seqs);
    return modes_bytes(slots) + (size_t)slots * kRecBytes;
}

bool split_supported(const PrefillArgs& a) {
    return a.dtype == DType::BF16 && a.dk == D && a.dv == D && a.total_tokens > 0 && encode_fn() != nullptr;
}

cudaError_t launch_split_prefill(const PrefillArgs& a, void* workspace, cudaStream_t s, bool segments) {
    int sms = 1;
    if (!configure_kernels(&sms)) return cudaErrorInvalidDevice;
    if (segments && segmented(a.total_tokens, a.num_seqs, a.H) && !a.ckpt_cu)
        return launch_segmented(a, workspace, sms, s);
    cudaError_t e = enqueue_local(a, workspace, sms, s);
    if (e == cudaSuccess) e = enqueue_chain(a, workspace, s);
    return e;
}

}  // namespace kda
