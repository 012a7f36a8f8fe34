/*
 * kda_oracle.c -- fp64 CPU oracle for the Kimi Delta Attention (KDA) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct statement of what the
 * GPU path computes.  Only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark may load it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it follows (page titles and sections):
 *   - "Kimi K3: the paper and proofs side by side", section 2.1.1, Equation 1 and the
 *     `update` / `update_get2` definitions: per head the state S is a d_k x d_v matrix
 *     (rows = key channels, columns = value channels).  One token
 *       1. scales row c of S by the retention alpha_c            (decay),
 *       2. reads the decayed state with the key, r = k^T (Diag(alpha) S),
 *       3. subtracts beta * k r^T                                  (erase),
 *       4. adds beta * k v^T                                       (write),
 *     and then the query reads the *updated* state, o = S_t^T q ("step = (update, read next q)").
 *     Steps 3 and 4 are written here as one delta-rule write with u = beta (v - r), which is
 *     the same arithmetic (update_get2's coordinate form is
 *       S'[c][j] = alpha_c S[c][j] - beta k_c r_j + beta k_c v_j).
 *   - Same page, Equation 5 (`retentionReal`): g = g_min * sigmoid(exp(A_h) * z), alpha = exp(g),
 *     with one scalar A_h per head and one z per key channel; g_min = -5 in K3.
 *   - "Kimi K3: architecture, derivations and a pinned-source audit", section 4.3 and the
 *     "Worked KDA state update and limits" example (decay rows, then correct along k, then read).
 *   - Heads are independent ("updateTerm applies KDA.update per head", section 2.1.1).
 *   - Sequences are packed token-major; cu_seqlens[n]..cu_seqlens[n+1] is sequence n, and each
 *     sequence starts from its own initial state (zeros when none is given).
 *
 * Layouts (row-major):  q, k, z: [T_tot, H, d_k]; v, out: [T_tot, H, d_v]; beta: [T_tot, H];
 *                       A: [H]; states: [N, H, d_k, d_v].
 * Inputs arrive as double arrays: every fp32 or bf16 value the GPU sees is upcast exactly to
 * double by the caller.  All arithmetic is double.
 *
 * Parallelism: OpenMP over (sequence, head, block of value columns).  Column j of the state
 * evolves using column j only (r_j, u_j and o_j read column j), so splitting columns changes no
 * per-element operation and no summation order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Logistic function, written in the overflow-free form for both signs of x. */
static double oracle_sigmoid(double x)
{
    if (x >= 0.0) {
        return 1.0 / (1.0 + exp(-x));
    }
    double e = exp(x);
    return e / (1.0 + e);
}

/* Equation 5: log-decay g = g_min * sigmoid(exp(A_h) * z) for one key channel. */
static double oracle_log_decay(double z, double A_h, double g_min)
{
    return g_min * oracle_sigmoid(exp(A_h) * z);
}

/*
 * Gate over a [T_tot, H, d_k] array: g and alpha = exp(g), written as doubles.
 * Either output may be NULL.
 */
void kda_oracle_gate(int64_t T_tot, int32_t H, int32_t dk, const double* z, const double* A,
                     double g_min, double* g_out, double* alpha_out)
{
    int64_t total = T_tot * (int64_t)H * dk;
#pragma omp parallel for schedule(static)
    for (int64_t idx = 0; idx < total; ++idx) {
        int32_t h = (int32_t)((idx / dk) % H);
        double g = oracle_log_decay(z[idx], A[h], g_min);
        if (g_out) g_out[idx] = g;
        if (alpha_out) alpha_out[idx] = exp(g);
    }
}

/*
 * One token of Equation 1 on columns [j0, j1) of one head's state S (d_k x d_v, row stride dv).
 * alpha: d_k retentions; k, q: d_k; v: d_v; beta: scalar.  o receives S_t^T q on [j0, j1).
 * r and u are caller scratch of length d_v.
 */
static void oracle_token_update(double* S, int32_t dk, int32_t dv, int32_t j0, int32_t j1,
                                const double* alpha, const double* k, const double* q,
                                const double* v, double beta, double* r, double* u, double* o)
{
    /* 1. decay: S <- Diag(alpha) S */
    for (int32_t c = 0; c < dk; ++c) {
        for (int32_t j = j0; j < j1; ++j) {
            S[(int64_t)c * dv + j] *= alpha[c];
        }
    }
    /* 2. read the decayed state along the key: r = (Diag(alpha) S)^T k */
    for (int32_t j = j0; j < j1; ++j) r[j] = 0.0;
    for (int32_t c = 0; c < dk; ++c) {
        for (int32_t j = j0; j < j1; ++j) {
            r[j] += k[c] * S[(int64_t)c * dv + j];
        }
    }
    /* 3+4. delta-rule write: S <- S + beta k (v - r)^T */
    for (int32_t j = j0; j < j1; ++j) u[j] = beta * (v[j] - r[j]);
    for (int32_t c = 0; c < dk; ++c) {
        for (int32_t j = j0; j < j1; ++j) {
            S[(int64_t)c * dv + j] += k[c] * u[j];
        }
    }
    /* read-out after the update: o = S_t^T q */
    for (int32_t j = j0; j < j1; ++j) o[j] = 0.0;
    for (int32_t c = 0; c < dk; ++c) {
        for (int32_t j = j0; j < j1; ++j) {
            o[j] += q[c] * S[(int64_t)c * dv + j];
        }
    }
}

/*
 * Shared driver.  Exactly one of (alpha) or (z, A) is used:
 *   alpha != NULL : retentions given directly, [T_tot, H, d_k];
 *   alpha == NULL : retentions from the gate (z [T_tot,H,d_k], A [H], g_min).
 * cu_seqlens: N+1 offsets (int64, non-decreasing, cu_seqlens[0] = 0).
 * S0: [N,H,d_k,d_v] or NULL (zeros).  out: [T_tot,H,d_v] doubles or NULL.
 * S_final: [N,H,d_k,d_v] doubles or NULL.  col_block: value columns per parallel unit (<=0: d_v).
 * Returns 0 on success, -1 on invalid arguments, -2 on allocation failure.
 */
static int oracle_run(int32_t N, const int64_t* cu_seqlens, int32_t H, int32_t dk, int32_t dv,
                      const double* q, const double* k, const double* v, const double* alpha_in,
                      const double* z, const double* A, double g_min, const double* beta,
                      const double* S0, double* out, double* S_final, int32_t col_block,
                      int32_t nthreads)
{
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
    if (N == 0) return 0;
    if (!q || !k || !v || !beta) return -1;
    if (!alpha_in && (!z || !A)) return -1;
    for (int32_t n = 0; n < N; ++n) {
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    }
    if (col_block <= 0 || col_block > dv) col_block = dv;
    const int32_t nblk = (dv + col_block - 1) / col_block;
    const int64_t units = (int64_t)N * H * nblk;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel
    {
        double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
        double* al = (double*)malloc(sizeof(double) * (size_t)dk);
        double* kk = (double*)malloc(sizeof(double) * (size_t)dk);
        double* qq = (double*)malloc(sizeof(double) * (size_t)dk);
        double* vv = (double*)malloc(sizeof(double) * (size_t)dv);
        double* r = (double*)malloc(sizeof(double) * (size_t)dv);
        double* u = (double*)malloc(sizeof(double) * (size_t)dv);
        double* o = (double*)malloc(sizeof(double) * (size_t)dv);
        int ok = S && al && kk && qq && vv && r && u && o;
        if (!ok) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t unit = 0; unit < units; ++unit) {
            if (!ok) continue;
            const int32_t blk = (int32_t)(unit % nblk);
            const int32_t h = (int32_t)((unit / nblk) % H);
            const int32_t n = (int32_t)(unit / ((int64_t)nblk * H));
            const int32_t j0 = blk * col_block;
            const int32_t j1 = (j0 + col_block < dv) ? j0 + col_block : dv;
            const int64_t sbase = ((int64_t)n * H + h) * dk * dv;

            for (int32_t c = 0; c < dk; ++c) {
                for (int32_t j = j0; j < j1; ++j) {
                    S[(int64_t)c * dv + j] = S0 ? S0[sbase + (int64_t)c * dv + j] : 0.0;
                }
            }
            for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
                const int64_t kbase = (t * H + h) * dk;
                const int64_t vbase = (t * H + h) * dv;
                for (int32_t c = 0; c < dk; ++c) {
                    al[c] = alpha_in ? alpha_in[kbase + c]
                                     : exp(oracle_log_decay(z[kbase + c], A[h], g_min));
                    kk[c] = k[kbase + c];
                    qq[c] = q[kbase + c];
                }
                for (int32_t j = j0; j < j1; ++j) vv[j] = v[vbase + j];
                oracle_token_update(S, dk, dv, j0, j1, al, kk, qq, vv, beta[t * H + h], r, u, o);
                if (out) {
                    for (int32_t j = j0; j < j1; ++j) out[vbase + j] = o[j];
                }
            }
            if (S_final) {
                for (int32_t c = 0; c < dk; ++c) {
                    for (int32_t j = j0; j < j1; ++j) {
                        S_final[sbase + (int64_t)c * dv + j] = S[(int64_t)c * dv + j];
                    }
                }
            }
        }
        free(S); free(al); free(kk); free(qq); free(vv); free(r); free(u); free(o);
    }
    return failed ? -2 : 0;
}

/* Equation 1 with the retentions alpha [T_tot, H, d_k] given directly. */
int kda_oracle_recurrence(int32_t N, const int64_t* cu_seqlens, int32_t H, int32_t dk, int32_t dv,
                          const double* q, const double* k, const double* v, const double* alpha,
                          const double* beta, const double* S0, double* out, double* S_final,
                          int32_t col_block, int32_t nthreads)
{
    if (!alpha) return -1;
    return oracle_run(N, cu_seqlens, H, dk, dv, q, k, v, alpha, NULL, NULL, 0.0, beta, S0, out,
                      S_final, col_block, nthreads);
}

/* Equation 1 driven by the Equation 5 gate (z [T_tot, H, d_k], A [H], g_min). */
int kda_oracle_forward(int32_t N, const int64_t* cu_seqlens, int32_t H, int32_t dk, int32_t dv,
                       const double* q, const double* k, const double* v, const double* z,
                       const double* A, double g_min, const double* beta, const double* S0,
                       double* out, double* S_final, int32_t col_block, int32_t nthreads)
{
    return oracle_run(N, cu_seqlens, H, dk, dv, q, k, v, NULL, z, A, g_min, beta, S0, out, S_final,
                      col_block, nthreads);
}

/*
 * One decode step: every sequence advances by exactly one token (the `step` of section 2.1.1).
 * q, k, z: [N, H, d_k]; v: [N, H, d_v]; beta: [N, H]; S_in, S_out: [N, H, d_k, d_v] (may be the
 * same array); out: [N, H, d_v].
 */
int kda_oracle_decode_step(int32_t N, int32_t H, int32_t dk, int32_t dv, const double* q,
                           const double* k, const double* v, const double* z, const double* A,
                           double g_min, const double* beta, const double* S_in, double* S_out,
                           double* out, int32_t nthreads)
{
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (N == 0) return 0;
    if (!q || !k || !v || !z || !A || !beta || !S_in || !S_out || !out) return -1;
    const int64_t units = (int64_t)N * H;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double* al = (double*)malloc(sizeof(double) * (size_t)dk);
        double* kk = (double*)malloc(sizeof(double) * (size_t)dk);
        double* qq = (double*)malloc(sizeof(double) * (size_t)dk);
        double* vv = (double*)malloc(sizeof(double) * (size_t)dv);
        double* r = (double*)malloc(sizeof(double) * (size_t)dv);
        double* u = (double*)malloc(sizeof(double) * (size_t)dv);
        double* o = (double*)malloc(sizeof(double) * (size_t)dv);
        int ok = al && kk && qq && vv && r && u && o;
        if (!ok) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t unit = 0; unit < units; ++unit) {
            if (!ok) continue;
            const int32_t h = (int32_t)(unit % H);
            const int64_t kbase = unit * dk;
            const int64_t vbase = unit * dv;
            const int64_t sbase = unit * dk * dv;
            double* S = S_out + sbase;
            if (S_out != S_in) memcpy(S, S_in + sbase, sizeof(double) * (size_t)dk * dv);
            for (int32_t c = 0; c < dk; ++c) {
                al[c] = exp(oracle_log_decay(z[kbase + c], A[h], g_min));
                kk[c] = k[kbase + c];
                qq[c] = q[kbase + c];
            }
            for (int32_t j = 0; j < dv; ++j) vv[j] = v[vbase + j];
            oracle_token_update(S, dk, dv, 0, dv, al, kk, qq, vv, beta[unit], r, u, o);
            for (int32_t j = 0; j < dv; ++j) out[vbase + j] = o[j];
        }
        free(al); free(kk); free(qq); free(vv); free(r); free(u); free(o);
    }
    return failed ? -2 : 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
