/*
 * kda_oracle.c -- fp64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (one head of one sequence, tokens in order):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * written out as the three state edits and the read that the pages describe:
 *   - "Kimi K3 Architecture Teardown", section "Hybrid Attention for 1M
 *     Tokens", Visual 5 (one KDA step): first decay every key channel of the
 *     state, then erase a beta-scaled share of what the decayed state holds
 *     under the current key, then write the new key-value pair scaled by the
 *     same beta.
 *   - "Kimi K3 Architecture: KDA, MoE, and Attention", section "Memory as a
 *     First-Class Problem": alpha is a per-channel decay, the same beta drives
 *     the erase and the write, and the output is the UPDATED state queried
 *     with q (read after write).
 *   - "Kimi K3 architecture: KDA, MLA and MoE", section "KDA is a writable
 *     state, not a smaller KV cache": the delta rule first measures what the
 *     state associates with the key, then writes the correction.
 *
 * The decayed state is D S with D = Diag(alpha_t); the erase term is
 * beta k (k^T D S) and the write term beta k v^T, so
 *     S_t = D S + beta k (v - (D S)^T k)^T
 * which is exactly the matrix form above.  The loop below performs these
 * steps literally in fp64, with no blocking, chunking or reordering.
 *
 * Layouts (row-major, contiguous, all fp64):
 *   q, k, log_alpha : [total_tokens, H, dk]
 *   v, out          : [total_tokens, H, dv]
 *   beta            : [total_tokens, H]
 *   states          : [num_seqs, H, dk, dv]
 * cu_seqlens[n] .. cu_seqlens[n+1] are the tokens of sequence n.
 *
 * Parity status: pinned (unrolled-product brute force, closed forms,
 * invariants and a hand-derived example in the CPU test suite).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * Mutation hooks.  A mutant build (compiled only by the CPU test that checks
 * that the pins are discriminating) plants one plausible mistake.  The
 * default build defines none of these and computes the recurrence above.
 *   1: read before write     (o_t = (D S_{t-1})^T q_t)
 *   2: decay after the write (S_t = D (S + beta k (v - S^T k)^T))
 *   3: erase at full strength (beta scales only the write)
 *   4: transposed read       (o_t = S_t q_t; meaningful for dk == dv)
 *   5: erase measured on the undecayed state (r = S_{t-1}^T k)
 *   6: sign of the erase flipped
 */
#ifndef KDA_ORACLE_MUTATION
#define KDA_ORACLE_MUTATION 0
#endif

static void decay_rows(int64_t dk, int64_t dv, double* S, const double* log_alpha)
{
    int64_t i, j;
    for (i = 0; i < dk; ++i) {
        const double a = exp(log_alpha[i]);
        for (j = 0; j < dv; ++j) S[i * dv + j] *= a;
    }
}

/* r = S^T k */
static void read_under_key(int64_t dk, int64_t dv, const double* S,
                           const double* key, double* r)
{
    int64_t i, j;
    for (j = 0; j < dv; ++j) r[j] = 0.0;
    for (i = 0; i < dk; ++i)
        for (j = 0; j < dv; ++j) r[j] += S[i * dv + j] * key[i];
}

/* One token of one head: S (dk x dv) is updated in place, o (dv) written.
 * r is caller-provided scratch of length dv. */
static void kda_oracle_token(int64_t dk, int64_t dv, double* S,
                             const double* q, const double* k, const double* v,
                             const double* log_alpha, double beta,
                             double* o, double* r)
{
    int64_t i, j;
#if KDA_ORACLE_MUTATION == 5
    read_under_key(dk, dv, S, k, r);
#endif
#if KDA_ORACLE_MUTATION != 2
    /* step 1: decay, one factor per key channel (row of S) */
    decay_rows(dk, dv, S, log_alpha);
#endif
#if KDA_ORACLE_MUTATION == 1
    read_under_key(dk, dv, S, q, o);
#endif
#if KDA_ORACLE_MUTATION != 5
    /* what the (decayed) state stores under the key */
    read_under_key(dk, dv, S, k, r);
#endif
    /* steps 2 and 3: erase beta*k*r^T, write beta*k*v^T */
    for (i = 0; i < dk; ++i) {
        for (j = 0; j < dv; ++j) {
#if KDA_ORACLE_MUTATION == 3
            S[i * dv + j] += k[i] * (beta * v[j] - r[j]);
#elif KDA_ORACLE_MUTATION == 6
            S[i * dv + j] += beta * k[i] * (v[j] + r[j]);
#else
            S[i * dv + j] += beta * k[i] * (v[j] - r[j]);
#endif
        }
    }
#if KDA_ORACLE_MUTATION == 2
    decay_rows(dk, dv, S, log_alpha);
#endif
#if KDA_ORACLE_MUTATION == 4
    for (j = 0; j < dv; ++j) o[j] = 0.0;
    for (i = 0; i < dk; ++i)
        for (j = 0; j < dv; ++j) o[i] += S[i * dv + j] * q[j];
#elif KDA_ORACLE_MUTATION != 1
    /* read the updated state: o = S^T q */
    read_under_key(dk, dv, S, q, o);
#endif
}

/*
 * Prefill over packed variable-length sequences.
 * initial_state may be NULL (zero state); final_state may be NULL (not
 * written).  Returns 0 on success, -1 on a bad argument, -2 on allocation
 * failure.  Work is spread over (sequence, head) pairs only; each pair runs
 * its tokens strictly in order.
 */
int kda_oracle_prefill(int64_t num_seqs, const int64_t* cu_seqlens, int64_t H,
                       int64_t dk, int64_t dv,
                       const double* q, const double* k, const double* v,
                       const double* log_alpha, const double* beta,
                       const double* initial_state, double* out,
                       double* final_state, int num_threads)
{
    int64_t p, npairs;
    int failed = 0;
    if (num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
    for (p = 0; p < num_seqs; ++p)
        if (cu_seqlens[p + 1] < cu_seqlens[p]) return -1;
    npairs = num_seqs * H;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (p = 0; p < npairs; ++p) {
        const int64_t n = p / H, h = p % H;
        const int64_t sdim = dk * dv;
        double* S = (double*)malloc((size_t)sdim * sizeof(double));
        double* r = (double*)malloc((size_t)dv * sizeof(double));
        int64_t t;
        if (!S || !r) {
            free(S);
            free(r);
            failed |= 1;
            continue;
        }
        if (initial_state)
            memcpy(S, initial_state + p * sdim, (size_t)sdim * sizeof(double));
        else
            memset(S, 0, (size_t)sdim * sizeof(double));
        for (t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            const int64_t th = t * H + h;
            kda_oracle_token(dk, dv, S, q + th * dk, k + th * dk, v + th * dv,
                             log_alpha + th * dk, beta[th], out + th * dv, r);
        }
        if (final_state)
            memcpy(final_state + p * sdim, S, (size_t)sdim * sizeof(double));
        free(S);
        free(r);
    }
    return failed ? -2 : 0;
}

/*
 * One decode step for num_seqs independent sequences (one token each):
 * state [num_seqs, H, dk, dv] is updated in place, out [num_seqs, H, dv].
 * This is the same token update as the prefill loop.
 */
int kda_oracle_decode_step(int64_t num_seqs, int64_t H, int64_t dk, int64_t dv,
                           const double* q, const double* k, const double* v,
                           const double* log_alpha, const double* beta,
                           double* state, double* out, int num_threads)
{
    int64_t p, npairs;
    int failed = 0;
    if (num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    npairs = num_seqs * H;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(static) reduction(| : failed)
#endif
    for (p = 0; p < npairs; ++p) {
        double* r = (double*)malloc((size_t)dv * sizeof(double));
        if (!r) {
            failed |= 1;
            continue;
        }
        kda_oracle_token(dk, dv, state + p * dk * dv, q + p * dk, k + p * dk,
                         v + p * dv, log_alpha + p * dk, beta[p],
                         out + p * dv, r);
        free(r);
    }
    return failed ? -2 : 0;
}

int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
