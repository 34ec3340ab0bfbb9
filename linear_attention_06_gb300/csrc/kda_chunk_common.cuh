// kda_chunk_common.cuh -- device code shared by the chunkwise tensor-core prefill
// kernels of libkda (the fused per-(sequence, head) kernel in kda_chunk_tc.cu and the
// split chunk-local / state-chain kernels in kda_chunk_split.cu).
//
// The math is that of kda_chunk_tc.cu's header: per chunk of C = 64 tokens, with
// e_r = sum_{r<t<=C} a_t and G = e_0 + a_1 (the chunk's total log decay),
//   Khat = e^{-e} o K, Qhat = e^{-e} o Q, Kb = e^{e} o K,
//   A = Khat Kb^T, P = Qhat Kb^T, T = (I + Diag(beta) L(A))^{-1} Diag(beta),
//   W' = T Khat, U = T V, Ss = Diag(e^G) S0,
//   Delta = U - W' Ss, O = Qhat Ss + (mask o P) Delta, S_C = Ss + Kb^T Delta,
// an exact rewrite of the token recurrence of "Kimi K3 Architecture Teardown"
// (section "Hybrid Attention for 1M Tokens", Visual 5).  Everything here runs in
// 128-thread groups (named barriers kBarP, kBarS, kBarB) or on one issuing thread.
#pragma once

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
constexpr float kMaxExponent = 60.f;
constexpr uint64_t kWaitLimitNs = 4000000000ull;   // 4 s per bounded wait
constexpr int kBarP = 1, kBarB = 2, kBarS = 3;      // named barriers of the 128-thread groups

// ---- layout of the solve inside a log_alpha slot (after log_alpha has been consumed)
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

__device__ __forceinline__ uint32_t qk_off(bool is_q, uint32_t r, uint32_t c) {
    return (c >> 6) * 16384u + (is_q ? 8192u : 0u) + sw128_offset(r, (c & 63u) * 2u);
}
__device__ __forceinline__ uint32_t half_off(uint32_t r, uint32_t c) {   // V and Kb
    return (c >> 6) * 8192u + sw128_offset(r, (c & 63u) * 2u);
}
__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }
// Index of the thread inside its 128-thread group (the groups start at multiples of 128).
__device__ __forceinline__ int lt() { return (int)(threadIdx.x & 127); }
// First TMEM lane this warp may access (the warp's lane quarter).
__device__ __forceinline__ uint32_t lane0() { return ((threadIdx.x >> 5) & 3) * 32; }
__device__ __forceinline__ int group_count(int) { return 128; }

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
// Pass 1 (build_suffix): suffix sums of log_alpha over the chunk, e[r][c] =
// sum_{r<t<L} a[t][c].  Each warp takes a segment of 16 rows and each lane four channels
// (16-byte accesses, packed fp32x2 adds): suffix sums inside the segment, then the
// segments' totals through the slot (each segment's first row) to add the later ones.
// Returns false (leaving log_alpha as it was) when a channel's chunk total leaves
// +-kMaxExponent, else writes e * log2(e) back in place (pass 2 takes base-2
// exponentials) and returns g = e^{G_c} for the thread's own channel c.  It touches only the log_alpha slot, so it runs before the
// chunk's other slots are free; the caller publishes g once they are.
// Pass 2 (build_tiles, thread = 16-byte chunk of 8 channels of one row):
// Khat = e^{-e} k, Qhat = e^{-e} q (in place), Kb = e^{e} k, all as 16-byte vector
// accesses; the factors are 2^{-+ e log2(e)} from the SFU's base-2 exponential, the scale
// by log2(e) having been applied once per element in pass 1.
constexpr float kLog2e = 1.4426950408889634f;
// 2^x, the SFU's approximation (subnormal results flushed to zero)
__device__ __forceinline__ float ex2f_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ bool build_suffix(float* A, int L, float& g) {
    // thread (quad, seg): channels 4 quad .. +3, rows 16 seg .. +15 (a warp per row segment)
    const int t = lt(), quad = t & 31, seg = t >> 5, c4 = 4 * quad;
    float2 lo[16], hi[16];                           // rows of this segment: channels c4, c4+1 | c4+2, c4+3
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = 16 * seg + i;
        const float4 a = (r < L) ? *reinterpret_cast<const float4*>(A + r * D + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
        lo[i] = make_float2(a.x, a.y);
        hi[i] = make_float2(a.z, a.w);
    }
    const float2 raw_lo = lo[0], raw_hi = hi[0];
    float2 rl = make_float2(0.f, 0.f), rh = rl;      // suffix sums inside the segment
#pragma unroll
    for (int i = 15; i >= 0; --i) {
        const float2 al = lo[i], ah = hi[i];
        lo[i] = rl; hi[i] = rh;
        rl = add2(rl, al); rh = add2(rh, ah);
    }
    // the segment's total into its first row (each thread's own four columns), then every
    // thread reads the four totals of its columns
    *reinterpret_cast<float4*>(A + 16 * seg * D + c4) = make_float4(rl.x, rl.y, rh.x, rh.y);
    group_sync(kBarP);
    float4 tot[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) tot[u] = *reinterpret_cast<const float4*>(A + 16 * u * D + c4);
    float gt = A[t];
#pragma unroll
    for (int u = 1; u < 4; ++u) gt += A[16 * u * D + t];   // this thread's channel t, same order
    float2 later_l = make_float2(0.f, 0.f), later_h = later_l, gl = later_l, gh = later_l;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float2 tl = make_float2(tot[u].x, tot[u].y), th = make_float2(tot[u].z, tot[u].w);
        gl = add2(gl, tl); gh = add2(gh, th);
        if (u > seg) { later_l = add2(later_l, tl); later_h = add2(later_h, th); }
    }
    const bool out = !(fabsf(gl.x) <= kMaxExponent) || !(fabsf(gl.y) <= kMaxExponent) ||
                     !(fabsf(gh.x) <= kMaxExponent) || !(fabsf(gh.y) <= kMaxExponent);
    if (group_or(kBarP, out)) {                      // leave log_alpha as it was
        *reinterpret_cast<float4*>(A + 16 * seg * D + c4) = make_float4(raw_lo.x, raw_lo.y, raw_hi.x, raw_hi.y);
        group_sync(kBarP);
        return false;
    }
    g = __expf(gt);
    const float2 l2 = make_float2(kLog2e, kLog2e);
    const float2 ll = __fmul2_rn(later_l, l2), lh = __fmul2_rn(later_h, l2);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float2 el = __ffma2_rn(lo[i], l2, ll), eh = __ffma2_rn(hi[i], l2, lh);
        *reinterpret_cast<float4*>(A + (16 * seg + i) * D + c4) = make_float4(el.x, el.y, eh.x, eh.y);
    }
    group_sync(kBarP);
    return true;
}

__device__ void build_tiles(uint8_t* qk, uint8_t* kb, const float* A, int L) {
    const int c = lt();
    // pass 2: 64 rows x 16 chunks = 1024 units, 8 per thread
#pragma unroll 1
    for (int m = 0; m < 8; ++m) {
        const int u = c + 128 * m, r = u >> 4, j = u & 15;
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
                const float u0 = ex2f_approx(-ev[2 * p]), u1 = ex2f_approx(-ev[2 * p + 1]);
                const float d0 = ex2f_approx(ev[2 * p]), d1 = ex2f_approx(ev[2 * p + 1]);
                const float2 kk = make_float2(k0, k1), uu = make_float2(u0, u1);
                const float2 a1 = __fmul2_rn(kk, uu), a2 = __fmul2_rn(make_float2(q0, q1), uu),
                             a3 = __fmul2_rn(kk, make_float2(d0, d1));
                o1[p] = pack_bf16x2(a1.x, a1.y);
                o2[p] = pack_bf16x2(a2.x, a2.y);
                o3[p] = pack_bf16x2(a3.x, a3.y);
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
__device__ void solve_T(uint8_t* aslot, const __nv_bfloat16* beta) {
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
    // (every block of T was written by the step that computed it)
}

// ============================ group B: state stage ===============================

// TMEM S^T (lane j = value channel, column c = key channel): S <- S Diag(gam)
// in fp32, and the bf16 copy of the decayed state packed as an A operand.
// Works in 32-column steps to keep the register footprint small.
// [cb0, cb1): the 32-column blocks this thread's warp handles (all four by default).
__device__ void decay_state(uint32_t tb, const float* gam, int cb0 = 0, int cb1 = 4) {
#pragma unroll 1
    for (int cb = cb0; cb < cb1; ++cb) {
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

// Lane c holds W'^T row c (64 tokens): store W'^T as bf16, MN-major B operand (the Delta
// product negates it through its instruction descriptor).
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
                w[u] = pack_bf16x2(__uint_as_float(v[8 * k + 2 * u]), __uint_as_float(v[8 * k + 2 * u + 1]));
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

// ---- the layer's front end, in place on a chunk's tiles ---------------------------
// "Kimi K3 architecture: KDA, MLA and MoE", section "Scale: Total vs Active Parameters and
// Serving Economics", Visual 1 (the KDA inset): q and k pass a short convolution, SiLU and
// an L2 norm, v a short convolution and SiLU, the decay and beta a sigmoid.  The
// convolution is causal and depthwise over the tokens of one sequence with zero history
// before its start, tap W-1 on the current token (the readings of kda_frontend).  These
// helpers turn the raw projection tiles a chunk's TMA loads brought in into the recurrence
// inputs, in the same slots, before the operand build reads them.

// Conv weights of one channel pair as four taps, tap 3 on the current token (taps before
// 4 - W are zero).
struct ConvTaps {
    float2 w[4];
};
__device__ __forceinline__ ConvTaps load_taps(const float* __restrict__ conv, int h, int d, int c0, int W) {
    ConvTaps t;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = i - (4 - W);                        // the weight's own tap index
        t.w[i] = j >= 0 ? make_float2(conv[((size_t)h * d + c0) * W + j], conv[((size_t)h * d + c0 + 1) * W + j])
                        : make_float2(0.f, 0.f);
    }
    return t;
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// SiLU through one hardware tanh: y sigmoid(y) = y/2 (1 + tanh(y/2)).
__device__ __forceinline__ float silu_tanh_f(float y) {
    float th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * y));
    return 0.5f * y * (1.f + th);
}

// Convolution + SiLU of one channel pair down rows [r0, r0 + R) of a bf16 tile (row r's pair
// at byte offset off(r)), in place; rows >= L are zeroed.  h0, h1, h2: the raw pair of the
// three tokens before row r0 (zeros before the sequence start), oldest first.  Rows are
// read eight at a time before any of them is written, so the loads of a batch overlap.
template <int R, typename Off>
__device__ __forceinline__ void conv_silu_pair(uint8_t* tile, Off off, int r0, int L, const ConvTaps& tp,
                                               float2 h0, float2 h1, float2 h2) {
#pragma unroll 1
    for (int rb = 0; rb < R; rb += 8) {
        float2 x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = unpack_bf16x2(*reinterpret_cast<const uint32_t*>(tile + off(r0 + rb + i)));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = r0 + rb + i;
            float2 y = make_float2(tp.w[3].x * x[i].x, tp.w[3].y * x[i].y);
            y.x = fmaf(tp.w[0].x, h0.x, fmaf(tp.w[1].x, h1.x, fmaf(tp.w[2].x, h2.x, y.x)));
            y.y = fmaf(tp.w[0].y, h0.y, fmaf(tp.w[1].y, h1.y, fmaf(tp.w[2].y, h2.y, y.y)));
            h0 = h1; h1 = h2; h2 = x[i];
            *reinterpret_cast<uint32_t*>(tile + off(r)) = r < L ? pack_bf16x2(silu_tanh_f(y.x), silu_tanh_f(y.y)) : 0u;
        }
    }
}

// Raw pair of channels (c0, c0 + 1) of the three tokens before t0 (zero before bos).
__device__ __forceinline__ void conv_halo(const __nv_bfloat16* __restrict__ raw, int64_t t0, int64_t bos, int H,
                                          int h, int d, int c0, float2& h0, float2& h1, float2& h2) {
    float2 hv[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int64_t t = t0 - 3 + i;
        hv[i] = t >= bos ? unpack_bf16x2(*reinterpret_cast<const uint32_t*>(raw + ((size_t)t * H + h) * d + c0))
                         : make_float2(0.f, 0.f);
    }
    h0 = hv[0]; h1 = hv[1]; h2 = hv[2];
}

// L2 norm over the 128 channels of row r of a q or k tile (two 64-channel halves 16 KB
// apart, 128-byte swizzled rows): x / sqrt(sum x^2 + eps), in place, bf16.
__device__ __forceinline__ void l2norm_row(uint8_t* tile, int r, float eps) {
    float ss = 0.f;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            const uint4 u = *reinterpret_cast<const uint4*>(tile + hf * 16384 + sw128_offset(r, 16 * ch));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = unpack_bf16x2(w[i]);
                ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
            }
        }
    const float rn = rsqrtf(ss + eps);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            uint4* q = reinterpret_cast<uint4*>(tile + hf * 16384 + sw128_offset(r, 16 * ch));
            const uint4 u = *q;
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = unpack_bf16x2(w[i]);
                o[i] = pack_bf16x2(f.x * rn, f.y * rn);
            }
            *q = make_uint4(o[0], o[1], o[2], o[3]);
        }
}

// logsigmoid(x) = min(x, 0) - log(1 + e^{-|x|}); the log of a number in (1, 2] through the
// hardware log2 is accurate to a few 1e-7 absolute, far below what log alpha needs.
__device__ __forceinline__ float logsigmoid_f(float x) { return fminf(x, 0.f) - __logf(1.f + __expf(-fabsf(x))); }
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

// log alpha = logsigmoid(decay logits) over a [64][128] fp32 tile, column c = the thread's
// channel, in place (rows >= L are set to 0: no decay).
__device__ __forceinline__ void logsigmoid_col(float* A, int c, int L) {
#pragma unroll 1
    for (int rb = 0; rb < C; rb += 16) {
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = A[(rb + i) * D + c];
#pragma unroll
        for (int i = 0; i < 16; ++i) A[(rb + i) * D + c] = rb + i < L ? logsigmoid_f(x[i]) : 0.f;
    }
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

// Delta^T = U^T + Ss^T (-W'^T) in the U slot: A = Ss^T from TMEM, K = 128, B = W'^T negated
// by the instruction descriptor.
__device__ __forceinline__ void mma_delta(uint32_t tb, uint32_t ucol, uint32_t sWT) {
    constexpr uint32_t idw = idesc_bf16_f32(128, 64, false, true, false, true);   // B negated: -W'^T
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
}  // namespace kda
