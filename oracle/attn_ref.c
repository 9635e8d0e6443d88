/*
 * attn_ref.c -- the CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * library, and it never touches a GPU.
 *
 * Everything is IEEE double precision on plain row-major arrays
 * [heads][T][D] (heads = B*H flattened).  No blocking, fusion or
 * reordering beyond what each definition states; OpenMP only splits
 * independent rows (or columns) across threads and never changes the order
 * of any sum.
 *
 * Sources (page titles and sections):
 *  - "Lab 06 - Attention kernels: online softmax -> FlashAttention -> Triton",
 *    section 2 "Online softmax" (running max m, running sum l, rescale by
 *    e^{m-m'}, logsumexp = m + log l), section 3 "FlashAttention forward"
 *    (per query tile state (m, l, acc); O = acc/l; LSE = m + log l; causal
 *    skip/diag/full tile classes), section 4 "FlashAttention backward"
 *    (dV = P^T dO, dP = dO V^T, dS = P o (dP - D), D_i = sum_j P_ij dP_ij,
 *    dQ = dS K scale, dK = dS^T Q scale).
 *  - "Triton FlashAttention-2 forward", section "The kernel" (the same
 *    recurrence with causal mask j <= i).
 *  - "Flash Attention and Kernel Optimization", section "Causal masking"
 *    (query i may attend to key j iff i >= j).
 *
 * Readings taken where the pages leave a step open:
 *  - causal means top-left alignment, key j visible to query i iff j <= i
 *    (all three pages agree when T_q = T_k);
 *  - LSE is the natural log of sum_j exp(scale * q_i . k_j) over visible j,
 *    with no epsilon (every row sees key 0, so the sum is >= 1 term);
 *  - D_i is computed from its definition sum_j P_ij dP_ij, not from the
 *    rowsum(dO o O) shortcut, so the tests can check the identity.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Visibility of key j to query i ("Lab 06", section 3; "Flash Attention and
 * Kernel Optimization", section "Causal masking"). */
static int visible(long i, long j, int causal) { return causal ? (j <= i) : 1; }

/* One score S_ij = scale * sum_d q_id k_jd. */
static double score(const double* qi, const double* kj, long D, double scale) {
    double s = 0.0;
    for (long d = 0; d < D; ++d) s += qi[d] * kj[d];
    return scale * s;
}

/*
 * Online softmax statistics over one row x[0..n) visited in blocks of
 * `block` elements ("Lab 06", section 2): keep m (running max) and
 * l = sum exp(x - m); when a block raises the max to m', rescale
 * l <- l * e^{m - m'} + sum_block e^{x - m'}.  At the end
 * logsumexp(x) = m + log l.
 */
void oracle_online_softmax_stats(const double* x, long n, long block, double* m_out, double* l_out) {
    double m = -INFINITY, l = 0.0;
    for (long b0 = 0; b0 < n; b0 += block) {
        long b1 = b0 + block < n ? b0 + block : n;
        double mb = -INFINITY;
        for (long t = b0; t < b1; ++t) mb = x[t] > mb ? x[t] : mb;
        double m_new = m > mb ? m : mb;
        double part = 0.0;
        for (long t = b0; t < b1; ++t) part += exp(x[t] - m_new);
        /* l * e^{m - m'}; when m is still -inf, l is 0 and stays 0 */
        l = (m == -INFINITY ? 0.0 : l * exp(m - m_new)) + part;
        m = m_new;
    }
    *m_out = m;
    *l_out = l;
}

/*
 * Naive forward for `nbh` independent heads: for every row i the scores
 * S_i. are formed, masked, exponentiated against the row max and
 * normalised; O_i = sum_j P_ij V_j and LSE_i = m_i + log sum_j e^{S_ij - m_i}.
 * ("Lab 06", sections 1 and 3: this is the definition the tiled algorithm
 * reaches exactly.)
 */
void oracle_attn_fwd(const double* q, const double* k, const double* v, long nbh, long T, long D,
                     double scale, int causal, double* o, double* lse) {
    long rows = nbh * T;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)T);
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            long h = r / T, i = r % T;
            const double* qi = q + (h * T + i) * D;
            const double* kh = k + h * T * D;
            const double* vh = v + h * T * D;
            double m = -INFINITY;
            for (long j = 0; j < T; ++j) {
                s[j] = visible(i, j, causal) ? score(qi, kh + j * D, D, scale) : -INFINITY;
                if (s[j] > m) m = s[j];
            }
            double sum = 0.0;
            for (long j = 0; j < T; ++j) {
                s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
                sum += s[j];
            }
            double* oi = o + (h * T + i) * D;
            for (long d = 0; d < D; ++d) oi[d] = 0.0;
            for (long j = 0; j < T; ++j) {
                double p = s[j] / sum;
                if (p == 0.0) continue;
                const double* vj = vh + j * D;
                for (long d = 0; d < D; ++d) oi[d] += p * vj[d];
            }
            lse[h * T + i] = m + log(sum);
        }
        free(s);
    }
}

/*
 * Materialised softmax probabilities of one head, P[T][T] (row i sums to 1,
 * masked entries exactly 0).  Used by the tests to pin the oracle.
 */
void oracle_attn_probs(const double* q, const double* k, long T, long D, double scale, int causal, double* P) {
#pragma omp parallel for schedule(dynamic, 16)
    for (long i = 0; i < T; ++i) {
        double* pi = P + i * T;
        double m = -INFINITY;
        for (long j = 0; j < T; ++j) {
            pi[j] = visible(i, j, causal) ? score(q + i * D, k + j * D, D, scale) : -INFINITY;
            if (pi[j] > m) m = pi[j];
        }
        double sum = 0.0;
        for (long j = 0; j < T; ++j) {
            pi[j] = (pi[j] == -INFINITY) ? 0.0 : exp(pi[j] - m);
            sum += pi[j];
        }
        for (long j = 0; j < T; ++j) pi[j] /= sum;
    }
}

/*
 * Naive backward for `nbh` heads with the analytic gradients of "Lab 06",
 * section 4, given upstream gradient dO:
 *   P  = softmax(S)            (materialised per head)
 *   dV = P^T dO
 *   dP = dO V^T
 *   D_i = sum_j P_ij dP_ij     (the definition)
 *   dS = P o (dP - D)
 *   dQ = dS K * scale,  dK = dS^T Q * scale
 * `dvec` (optional, may be NULL) receives D_i per row.
 * Returns 0, or -1 if the T x T scratch could not be allocated.
 */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout, long nbh, long T,
                    long D, double scale, int causal, double* dq, double* dk, double* dv, double* dvec) {
    double* P = (double*)malloc(sizeof(double) * (size_t)T * (size_t)T);
    double* dS = (double*)malloc(sizeof(double) * (size_t)T * (size_t)T);
    double* Dv = (double*)malloc(sizeof(double) * (size_t)T);
    if (!P || !dS || !Dv) {
        free(P); free(dS); free(Dv);
        return -1;
    }
    for (long h = 0; h < nbh; ++h) {
        const double* qh = q + h * T * D;
        const double* kh = k + h * T * D;
        const double* vh = v + h * T * D;
        const double* doh = dout + h * T * D;
        double* dqh = dq + h * T * D;
        double* dkh = dk + h * T * D;
        double* dvh = dv + h * T * D;
        oracle_attn_probs(qh, kh, T, D, scale, causal, P);
        /* dP_ij = dO_i . V_j ; D_i = sum_j P_ij dP_ij ; dS_ij = P_ij (dP_ij - D_i) */
#pragma omp parallel for schedule(dynamic, 16)
        for (long i = 0; i < T; ++i) {
            double* dsi = dS + i * T;
            for (long j = 0; j < T; ++j) {
                double dp = 0.0;
                for (long d = 0; d < D; ++d) dp += doh[i * D + d] * vh[j * D + d];
                dsi[j] = dp; /* holds dP for now */
            }
            double di = 0.0;
            for (long j = 0; j < T; ++j) di += P[i * T + j] * dsi[j];
            Dv[i] = di;
            for (long j = 0; j < T; ++j) dsi[j] = P[i * T + j] * (dsi[j] - di);
        }
        if (dvec) memcpy(dvec + h * T, Dv, sizeof(double) * (size_t)T);
        /* dV_j = sum_i P_ij dO_i ; dK_j = scale * sum_i dS_ij Q_i (columns of P and dS) */
#pragma omp parallel for schedule(dynamic, 16)
        for (long j = 0; j < T; ++j) {
            double* dvj = dvh + j * D;
            double* dkj = dkh + j * D;
            for (long d = 0; d < D; ++d) { dvj[d] = 0.0; dkj[d] = 0.0; }
            for (long i = 0; i < T; ++i) {
                double p = P[i * T + j], ds = dS[i * T + j];
                for (long d = 0; d < D; ++d) {
                    dvj[d] += p * doh[i * D + d];
                    dkj[d] += ds * qh[i * D + d];
                }
            }
            for (long d = 0; d < D; ++d) dkj[d] *= scale;
        }
        /* dQ_i = scale * sum_j dS_ij K_j */
#pragma omp parallel for schedule(dynamic, 16)
        for (long i = 0; i < T; ++i) {
            double* dqi = dqh + i * D;
            for (long d = 0; d < D; ++d) dqi[d] = 0.0;
            for (long j = 0; j < T; ++j) {
                double ds = dS[i * T + j];
                if (ds == 0.0) continue;
                for (long d = 0; d < D; ++d) dqi[d] += ds * kh[j * D + d];
            }
            for (long d = 0; d < D; ++d) dqi[d] *= scale;
        }
    }
    free(P); free(dS); free(Dv);
    return 0;
}

/*
 * Row-sampled backward for ONE head, for sizes where T x T storage per head
 * is too large to hold for many heads.  Same definitions as
 * oracle_attn_bwd, evaluated only where asked:
 *   pass 1 (every row i): m_i, LSE_i and D_i = sum_j P_ij dP_ij;
 *   dQ_i for i in rows_q:  scale * sum_j P_ij (dP_ij - D_i) K_j;
 *   dK_j, dV_j for j in rows_k: sums over i of the column j of P and dS.
 * lse_out / dvec_out (length T) receive LSE and D for every row.
 */
int oracle_attn_bwd_rows(const double* q, const double* k, const double* v, const double* dout, long T, long D,
                         double scale, int causal, long nq, const long* rows_q, long nk, const long* rows_k,
                         double* dq_rows, double* dk_rows, double* dv_rows, double* lse_out, double* dvec_out) {
    /* pass 1: per-row statistics */
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)T);
#pragma omp for schedule(dynamic, 16)
        for (long i = 0; i < T; ++i) {
            double m = -INFINITY;
            for (long j = 0; j < T; ++j) {
                s[j] = visible(i, j, causal) ? score(q + i * D, k + j * D, D, scale) : -INFINITY;
                if (s[j] > m) m = s[j];
            }
            double sum = 0.0;
            for (long j = 0; j < T; ++j) {
                s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
                sum += s[j];
            }
            double di = 0.0;
            for (long j = 0; j < T; ++j) {
                double p = s[j] / sum;
                if (p == 0.0) continue;
                double dp = 0.0;
                for (long d = 0; d < D; ++d) dp += dout[i * D + d] * v[j * D + d];
                di += p * dp;
            }
            lse_out[i] = m + log(sum);
            dvec_out[i] = di;
        }
        free(s);
    }
    /* dQ rows */
#pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < nq; ++r) {
        long i = rows_q[r];
        double* out = dq_rows + r * D;
        for (long d = 0; d < D; ++d) out[d] = 0.0;
        for (long j = 0; j < T; ++j) {
            if (!visible(i, j, causal)) continue;
            double p = exp(score(q + i * D, k + j * D, D, scale) - lse_out[i]);
            double dp = 0.0;
            for (long d = 0; d < D; ++d) dp += dout[i * D + d] * v[j * D + d];
            double ds = p * (dp - dvec_out[i]);
            for (long d = 0; d < D; ++d) out[d] += ds * k[j * D + d];
        }
        for (long d = 0; d < D; ++d) out[d] *= scale;
    }
    /* dK and dV rows */
#pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < nk; ++r) {
        long j = rows_k[r];
        double* gk = dk_rows + r * D;
        double* gv = dv_rows + r * D;
        for (long d = 0; d < D; ++d) { gk[d] = 0.0; gv[d] = 0.0; }
        for (long i = 0; i < T; ++i) {
            if (!visible(i, j, causal)) continue;
            double p = exp(score(q + i * D, k + j * D, D, scale) - lse_out[i]);
            double dp = 0.0;
            for (long d = 0; d < D; ++d) dp += dout[i * D + d] * v[j * D + d];
            double ds = p * (dp - dvec_out[i]);
            for (long d = 0; d < D; ++d) {
                gv[d] += p * dout[i * D + d];
                gk[d] += ds * q[i * D + d];
            }
        }
        for (long d = 0; d < D; ++d) gk[d] *= scale;
    }
    return 0;
}

/*
 * Row-sampled forward for ONE head: O_i and LSE_i for i in rows only
 * (same definition as oracle_attn_fwd).
 */
void oracle_attn_fwd_rows(const double* q, const double* k, const double* v, long T, long D, double scale,
                          int causal, long nrows, const long* rows, double* o_rows, double* lse_rows) {
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)T);
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < nrows; ++r) {
            long i = rows[r];
            double m = -INFINITY;
            for (long j = 0; j < T; ++j) {
                s[j] = visible(i, j, causal) ? score(q + i * D, k + j * D, D, scale) : -INFINITY;
                if (s[j] > m) m = s[j];
            }
            double sum = 0.0;
            for (long j = 0; j < T; ++j) {
                s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
                sum += s[j];
            }
            double* oi = o_rows + r * D;
            for (long d = 0; d < D; ++d) oi[d] = 0.0;
            for (long j = 0; j < T; ++j) {
                double p = s[j] / sum;
                if (p == 0.0) continue;
                for (long d = 0; d < D; ++d) oi[d] += p * v[j * D + d];
            }
            lse_rows[r] = m + log(sum);
        }
        free(s);
    }
}

/*
 * The tiled FlashAttention forward of "Lab 06", section 3, for ONE head, in
 * double precision and in the page's order: for each query tile of `bq`
 * rows keep (m, l, acc); for each key tile of `bk` keys
 *     S  = Q_i K_j^T * scale
 *     m' = max(m, rowmax S)
 *     P~ = exp(S - m')
 *     acc <- acc * e^{m - m'} + P~ V_j
 *     l   <- l   * e^{m - m'} + rowsum P~
 * then O = acc / l and LSE = m + log l.  Under causal masking key tiles
 * wholly above the diagonal are skipped (the last tile needed is the one
 * holding the tile's last row) and the others are masked element-wise.
 * Block sizes need not divide T.
 */
void oracle_flash_fwd_tiled(const double* q, const double* k, const double* v, long T, long D, double scale,
                            int causal, long bq, long bk, double* o, double* lse) {
    for (long i0 = 0; i0 < T; i0 += bq) {
        long i1 = i0 + bq < T ? i0 + bq : T;
        long nr = i1 - i0;
        double* m = (double*)malloc(sizeof(double) * (size_t)nr);
        double* l = (double*)malloc(sizeof(double) * (size_t)nr);
        double* acc = (double*)calloc((size_t)(nr * D), sizeof(double));
        double* st = (double*)malloc(sizeof(double) * (size_t)bk);
        for (long r = 0; r < nr; ++r) { m[r] = -INFINITY; l[r] = 0.0; }
        /* last key needed by this tile is its last row i1-1 (causal) */
        long kend = causal ? i1 : T;
        for (long j0 = 0; j0 < kend; j0 += bk) {
            long j1 = j0 + bk < T ? j0 + bk : T;
            for (long r = 0; r < nr; ++r) {
                long i = i0 + r;
                double mt = -INFINITY;
                for (long j = j0; j < j1; ++j) {
                    st[j - j0] = visible(i, j, causal) ? score(q + i * D, k + j * D, D, scale) : -INFINITY;
                    if (st[j - j0] > mt) mt = st[j - j0];
                }
                double m_new = m[r] > mt ? m[r] : mt;
                if (m_new == -INFINITY) continue; /* whole tile masked for this row, nothing seen yet */
                double alpha = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - m_new);
                double rs = 0.0;
                double* ar = acc + r * D;
                for (long d = 0; d < D; ++d) ar[d] *= alpha;
                for (long j = j0; j < j1; ++j) {
                    double p = (st[j - j0] == -INFINITY) ? 0.0 : exp(st[j - j0] - m_new);
                    rs += p;
                    for (long d = 0; d < D; ++d) ar[d] += p * v[j * D + d];
                }
                l[r] = l[r] * alpha + rs;
                m[r] = m_new;
            }
        }
        for (long r = 0; r < nr; ++r) {
            for (long d = 0; d < D; ++d) o[(i0 + r) * D + d] = acc[r * D + d] / l[r];
            lse[i0 + r] = m[r] + log(l[r]);
        }
        free(m); free(l); free(acc); free(st);
    }
}

/*
 * Naive forward where the Tq queries of a head attend to all Tk keys of the
 * same head (no mask): the decoding case of "Lab 06", "Check yourself" items
 * 2 and "Stretch" (one new token against a long cache).  Same definition as
 * oracle_attn_fwd: O_i = softmax(scale * q_i . K^T) V, LSE_i = m_i + log sum.
 * q, o: [nbh][Tq][D]; k, v: [nbh][Tk][D]; lse: [nbh][Tq].
 */
void oracle_attn_fwd_cross(const double* q, const double* k, const double* v, long nbh, long Tq, long Tk, long D,
                           double scale, double* o, double* lse) {
    long rows = nbh * Tq;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Tk);
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            long h = r / Tq, i = r % Tq;
            const double* qi = q + (h * Tq + i) * D;
            const double* kh = k + h * Tk * D;
            const double* vh = v + h * Tk * D;
            double m = -INFINITY;
            for (long j = 0; j < Tk; ++j) {
                s[j] = score(qi, kh + j * D, D, scale);
                if (s[j] > m) m = s[j];
            }
            double sum = 0.0;
            for (long j = 0; j < Tk; ++j) {
                s[j] = exp(s[j] - m);
                sum += s[j];
            }
            double* oi = o + (h * Tq + i) * D;
            for (long d = 0; d < D; ++d) oi[d] = 0.0;
            for (long j = 0; j < Tk; ++j) {
                double pj = s[j] / sum;
                for (long d = 0; d < D; ++d) oi[d] += pj * vh[j * D + d];
            }
            lse[h * Tq + i] = m + log(sum);
        }
        free(s);
    }
}
