/*
 * sink_oracle.c - plain fp64 CPU oracle for softmax attention with a learnable
 * sink logit per query head (forward and analytic backward).
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT: only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load or call this code. It is
 * written straight from the definitions, with no blocking, no online softmax
 * and no fused passes, so that each step can be checked against the page by
 * eye. Citations refer to the page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、
 * 超稳定！" (nmedialink.com), abbreviated [nmedialink], by section.
 *
 * Readings taken where the page leaves a step open (each also listed with the
 * design notes of this repository):
 *   - the sink is a raw logit appended to the already-scaled scores, so it is
 *     not multiplied by the softmax scale;
 *   - there is one sink per query head (each softmax row belongs to one query
 *     head), and dL/dS_h sums over every sequence and row of that head;
 *   - the backward equations in section "反向传播的实现" write dL/dS_ij where
 *     the derivation needs the upstream gradient on the probability P_ij; the
 *     oracle applies the softmax chain rule to the combined row
 *     [scores, sink] with upstream gradient dO_i . v_j on content column j and
 *     0 on the sink column (the sink is dropped before @V);
 *   - a sliding window of W keys means keys i-W+1 .. i and is always causal.
 */
#include "sink_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int nseq;
    const int32_t* cu;
    int h_q, h_kv, d;
    double scale;
    int causal, window;
} problem_t;

static int check_problem(const problem_t* P) {
    if (P->nseq < 0 || P->cu == NULL || P->h_q <= 0 || P->h_kv <= 0 || P->d <= 0) return -1;
    if (P->h_q % P->h_kv != 0) return -1;
    if (P->window > 0 && !P->causal) return -1;
    if (P->cu[0] != 0) return -1;
    for (int s = 0; s < P->nseq; ++s)
        if (P->cu[s + 1] < P->cu[s]) return -1;
    return 0;
}

static int longest(const problem_t* P) {
    int m = 0;
    for (int s = 0; s < P->nseq; ++s) {
        int L = P->cu[s + 1] - P->cu[s];
        if (L > m) m = L;
    }
    return m;
}

/* Allowed keys of row i in a sequence of length L: positions [*j0, *j1). */
static void allowed_keys(const problem_t* P, int i, int L, int* j0, int* j1) {
    if (!P->causal) {
        *j0 = 0;
        *j1 = L;
        return;
    }
    *j1 = i + 1;
    *j0 = 0;
    if (P->window > 0 && i - P->window + 1 > 0) *j0 = i - P->window + 1;
}

/* Rows that can see key j, the same mask read from the key's side:
 * positions [*i0, *i1). Every row in the range is still checked against
 * allowed_keys before it contributes. */
static void rows_seeing(const problem_t* P, int j, int L, int* i0, int* i1) {
    *i0 = P->causal ? j : 0;
    *i1 = L;
    if (P->causal && P->window > 0 && j + P->window < L) *i1 = j + P->window;
}

static double dot(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

/*
 * The combined score row and its softmax ([nmedialink] "GPT-OSS中的带注意力槽的
 * 注意力机制" and "数学公式深入解读"): z_t = scale * q_i . k_{j0+t} for the n
 * allowed keys, z_n = S_h; p = softmax(z) computed as exp(z - max z) / sum.
 * p[0..n-1] are the content probabilities P_ij, p[n] is the sink probability
 * P_{i,h}. Returns the logsumexp of z.
 */
static double row_softmax(const problem_t* P, const double* q, const double* k,
                          const double* sinks, int base, int h, int i, int j0, int j1,
                          double* z, double* p) {
    const int g = P->h_q / P->h_kv, hk = h / g, d = P->d;
    const int n = j1 - j0;
    const double* qi = q + ((size_t)(base + i) * P->h_q + h) * d;
    for (int t = 0; t < n; ++t) {
        const double* kj = k + ((size_t)(base + j0 + t) * P->h_kv + hk) * d;
        z[t] = P->scale * dot(qi, kj, d);
    }
    z[n] = sinks[h];
    double m = z[0];
    for (int t = 1; t <= n; ++t)
        if (z[t] > m) m = z[t];
    double sum = 0.0;
    for (int t = 0; t <= n; ++t) sum += exp(z[t] - m);
    for (int t = 0; t <= n; ++t) p[t] = exp(z[t] - m) / sum;
    return m + log(sum);
}

/*
 * Chain rule through p = softmax(z) ([nmedialink] "反向传播的实现"): with upstream
 * gradient u_t = dO_i . v_{j0+t} on each content probability and u_n = 0 on the
 * dropped sink column, dz_t = p_t (u_t - sum_m p_m u_m). The last entry dz_n is
 * this row's term of dL/dS_h = -P_{i,h} sum_j P_ij u_j.
 */
static void row_backward(const problem_t* P, const double* v, const double* dout, int base,
                         int h, int i, int j0, int j1, const double* p, double* u, double* dz) {
    const int g = P->h_q / P->h_kv, hk = h / g, d = P->d;
    const int n = j1 - j0;
    const double* doi = dout + ((size_t)(base + i) * P->h_q + h) * d;
    for (int t = 0; t < n; ++t) {
        const double* vj = v + ((size_t)(base + j0 + t) * P->h_kv + hk) * d;
        u[t] = dot(doi, vj, d);
    }
    u[n] = 0.0;
    double c = 0.0;
    for (int t = 0; t <= n; ++t) c += p[t] * u[t];
    for (int t = 0; t <= n; ++t) dz[t] = p[t] * (u[t] - c);
}

/* Sequence index of every token (tokens outside [0, T) do not occur). */
static int* token_seq(const problem_t* P) {
    const int T = P->cu[P->nseq];
    int* ts = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
    if (!ts) return NULL;
    for (int s = 0; s < P->nseq; ++s)
        for (int t = P->cu[s]; t < P->cu[s + 1]; ++t) ts[t] = s;
    return ts;
}

int sink_oracle_forward(int nseq, const int32_t* cu_seqlens, int h_q, int h_kv, int d,
                        double scale, int causal, int window, int row_begin, int row_end,
                        const double* q, const double* k, const double* v, const double* sinks,
                        double* o, double* lse) {
    problem_t P = {nseq, cu_seqlens, h_q, h_kv, d, scale, causal, window};
    if (check_problem(&P)) return -1;
    if (!q || !k || !v || !sinks || !o || !lse) return -1;
    const int T = cu_seqlens[nseq];
    const int Lmax = longest(&P);
    int* ts = token_seq(&P);
    if (!ts) return -1;
    int bad = 0;
    /* rows are independent: one unit = one (token, query head) row */
    const long long nrows = (long long)T * h_q;
#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)(Lmax + 1));
        double* p = (double*)malloc(sizeof(double) * (size_t)(Lmax + 1));
        if (!z || !p) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (long long r = 0; r < nrows; ++r) {
                const int t = (int)(r / h_q), h = (int)(r % h_q);
                const int s = ts[t], base = cu_seqlens[s], L = cu_seqlens[s + 1] - base;
                const int i = t - base;
                if (i < row_begin || i >= row_end) continue;
                const int hk = h / (h_q / h_kv);
                int j0, j1;
                allowed_keys(&P, i, L, &j0, &j1);
                const double l = row_softmax(&P, q, k, sinks, base, h, i, j0, j1, z, p);
                /* output = probs_content @ V: the sink column is dropped */
                double* oi = o + ((size_t)t * h_q + h) * d;
                for (int c = 0; c < d; ++c) oi[c] = 0.0;
                for (int u = 0; u < j1 - j0; ++u) {
                    const double* vj = v + ((size_t)(base + j0 + u) * h_kv + hk) * d;
                    for (int c = 0; c < d; ++c) oi[c] += p[u] * vj[c];
                }
                lse[(size_t)h * T + t] = l;
            }
        }
        free(z);
        free(p);
    }
    free(ts);
    return bad ? -1 : 0;
}

/*
 * Backward in two passes, each a plain loop over independent outputs.
 * Pass 1, per row (i, h): the combined row's softmax p and the chain-rule
 * gradient dz = p (u - c) (row_backward). It yields dq_i = scale sum_j dz_ij k_j,
 * the row's term dz_sink of dL/dS_h, and keeps the row's logsumexp and c_i.
 * Pass 2, per key (j, key/value head): dk_j = scale sum dz_ij q_i and
 * dv_j = sum p_ij dO_i over every (query head of the group, row that sees j),
 * with p_ij = exp(z_ij - logsumexp_i) and dz_ij = p_ij (u_ij - c_i) evaluated
 * from the kept per-row quantities.
 */
int sink_oracle_backward(int nseq, const int32_t* cu_seqlens, int h_q, int h_kv, int d,
                         double scale, int causal, int window, int row_begin, int row_end,
                         const double* q, const double* k, const double* v, const double* sinks,
                         const double* dout,
                         double* dq, double* dk, double* dv, double* dsinks) {
    problem_t P = {nseq, cu_seqlens, h_q, h_kv, d, scale, causal, window};
    if (check_problem(&P)) return -1;
    if (!q || !k || !v || !sinks || !dout || !dq || !dk || !dv || !dsinks) return -1;
    const int T = cu_seqlens[nseq];
    const int g = h_q / h_kv;
    const int Lmax = longest(&P);
    int* ts = token_seq(&P);
    /* per (query head, token): logsumexp, c = sum_t p_t u_t, sink term, in-range flag */
    double* row_lse = (double*)calloc((size_t)h_q * (T > 0 ? T : 1), sizeof(double));
    double* row_c = (double*)calloc((size_t)h_q * (T > 0 ? T : 1), sizeof(double));
    double* row_sink = (double*)calloc((size_t)h_q * (T > 0 ? T : 1), sizeof(double));
    if (!ts || !row_lse || !row_c || !row_sink) {
        free(ts);
        free(row_lse);
        free(row_c);
        free(row_sink);
        return -1;
    }
    memset(dq, 0, sizeof(double) * (size_t)T * h_q * d);
    int bad = 0;
    const long long nrows = (long long)T * h_q;
#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)(Lmax + 1));
        double* p = (double*)malloc(sizeof(double) * (size_t)(Lmax + 1));
        double* u = (double*)malloc(sizeof(double) * (size_t)(Lmax + 1));
        double* dz = (double*)malloc(sizeof(double) * (size_t)(Lmax + 1));
        if (!z || !p || !u || !dz) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (long long r = 0; r < nrows; ++r) {
                const int t = (int)(r / h_q), h = (int)(r % h_q);
                const int s = ts[t], base = cu_seqlens[s], L = cu_seqlens[s + 1] - base;
                const int i = t - base;
                if (i < row_begin || i >= row_end) continue;
                const int hk = h / g;
                int j0, j1;
                allowed_keys(&P, i, L, &j0, &j1);
                const int n = j1 - j0;
                const double l = row_softmax(&P, q, k, sinks, base, h, i, j0, j1, z, p);
                row_backward(&P, v, dout, base, h, i, j0, j1, p, u, dz);
                double c = 0.0;
                for (int m = 0; m < n; ++m) c += p[m] * u[m];
                double* dqi = dq + ((size_t)t * h_q + h) * d;
                for (int m = 0; m < n; ++m) {
                    /* S_ij = scale * q_i . k_j */
                    const double* kj = k + ((size_t)(base + j0 + m) * h_kv + hk) * d;
                    for (int e = 0; e < d; ++e) dqi[e] += scale * dz[m] * kj[e];
                }
                row_lse[(size_t)h * T + t] = l;
                row_c[(size_t)h * T + t] = c;
                row_sink[(size_t)h * T + t] = dz[n];
            }
        }
        free(z);
        free(p);
        free(u);
        free(dz);
    }
    /* pass 2: one unit = one (token, key/value head) key row */
    const long long nkeys = (long long)T * h_kv;
#pragma omp parallel for schedule(dynamic, 64)
    for (long long r = 0; r < nkeys; ++r) {
        const int t = (int)(r / h_kv), hk = (int)(r % h_kv);
        const int s = ts[t], base = cu_seqlens[s], L = cu_seqlens[s + 1] - base;
        const int j = t - base;
        const size_t kv_off = ((size_t)t * h_kv + hk) * d;
        const double* kj = k + kv_off;
        const double* vj = v + kv_off;
        double* dkj = dk + kv_off;
        double* dvj = dv + kv_off;
        for (int e = 0; e < d; ++e) dkj[e] = dvj[e] = 0.0;
        int i0, i1;
        rows_seeing(&P, j, L, &i0, &i1);
        for (int h = hk * g; h < (hk + 1) * g; ++h) {
            for (int i = i0; i < i1; ++i) {
                if (i < row_begin || i >= row_end) continue;
                int j0, j1;
                allowed_keys(&P, i, L, &j0, &j1);
                if (j < j0 || j >= j1) continue;
                const size_t ri = (size_t)h * T + base + i;
                const double* qi = q + ((size_t)(base + i) * h_q + h) * d;
                const double* doi = dout + ((size_t)(base + i) * h_q + h) * d;
                const double pij = exp(scale * dot(qi, kj, d) - row_lse[ri]);
                const double dzij = pij * (dot(doi, vj, d) - row_c[ri]);
                for (int e = 0; e < d; ++e) {
                    dkj[e] += scale * dzij * qi[e];
                    dvj[e] += pij * doi[e];
                }
            }
        }
    }
    /* dL/dS_h: sum of the rows' sink terms in token order */
    for (int h = 0; h < h_q; ++h) {
        double acc = 0.0;
        for (int t = 0; t < T; ++t) acc += row_sink[(size_t)h * T + t];
        dsinks[h] = acc;
    }
    free(ts);
    free(row_lse);
    free(row_c);
    free(row_sink);
    return bad ? -1 : 0;
}

int sink_oracle_row(int nseq, const int32_t* cu_seqlens, int h_q, int h_kv, int d,
                    double scale, int causal, int window,
                    const double* q, const double* k, const double* v, const double* sinks,
                    const double* dout, int seq, int head, int row,
                    double* p, double* dz, int* first_key) {
    problem_t P = {nseq, cu_seqlens, h_q, h_kv, d, scale, causal, window};
    if (check_problem(&P)) return -1;
    if (!q || !k || !sinks || !p || !first_key) return -1;
    if (seq < 0 || seq >= nseq || head < 0 || head >= h_q) return -1;
    const int base = cu_seqlens[seq], L = cu_seqlens[seq + 1] - base;
    if (row < 0 || row >= L) return -1;
    int j0, j1;
    allowed_keys(&P, row, L, &j0, &j1);
    const int n = j1 - j0;
    double* z = (double*)malloc(sizeof(double) * (size_t)(n + 1));
    double* u = (double*)malloc(sizeof(double) * (size_t)(n + 1));
    if (!z || !u) {
        free(z);
        free(u);
        return -1;
    }
    row_softmax(&P, q, k, sinks, base, head, row, j0, j1, z, p);
    if (dout && dz && v) row_backward(&P, v, dout, base, head, row, j0, j1, p, u, dz);
    free(z);
    free(u);
    *first_key = j0;
    return n;
}

int sink_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
