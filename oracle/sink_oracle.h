/*
 * sink_oracle.h - fp64 CPU oracle for softmax attention with one learnable
 * sink logit per query head.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load or call this code. It
 * shares no code, header or table with the CUDA library.
 *
 * Sources (all on the page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！",
 * nmedialink.com, referred to below as [nmedialink]):
 *   - section "标准注意力机制回顾": scores = Q K^T / sqrt(d), softmax, @V;
 *   - section "GPT-OSS中的带注意力槽的注意力机制": the sink logit is
 *     concatenated to the scores as one extra column, softmax runs over
 *     N_k + 1 columns, the sink column is dropped before @V;
 *   - section "数学公式深入解读": the displayed equations for the content
 *     probability P_ij and the sink probability P_{i,h};
 *   - section "反向传播的实现": the two displayed equations for dL/dS_h
 *     (general form, then the form with zero upstream gradient on the sink).
 *
 * Layout (all arrays host memory, row-major, fp64 unless stated):
 *   q     [T, h_q,  d]     T = cu_seqlens[nseq]
 *   k, v  [T, h_kv, d]
 *   sinks [h_q]            raw logits S_h, not multiplied by the scale
 *   o     [T, h_q,  d]
 *   lse   [h_q, T]         natural-log logsumexp of the row including S_h
 *   dout  [T, h_q,  d]     upstream gradient dL/dO
 *   dq    [T, h_q,  d], dk/dv [T, h_kv, d], dsinks [h_q]
 * cu_seqlens is int32 [nseq + 1], non-decreasing, cu_seqlens[0] == 0.
 * Query head h reads key/value head h / (h_q / h_kv).
 *
 * Masks, per sequence, positions relative to the sequence start:
 *   causal == 0, window <= 0 : row i sees keys 0 .. L-1 (the pages' own form)
 *   causal == 1, window <= 0 : row i sees keys 0 .. i
 *   causal == 1, window  > 0 : row i sees keys max(0, i-window+1) .. i
 *
 * Row range: only rows with row_begin <= i < row_end (positions within each
 * sequence) are evaluated. The full problem is row_begin = 0, row_end >= the
 * longest sequence. With a partial range, outputs for rows in range are exact,
 * and dk/dv/dsinks hold only the contributions of the rows in range (exact for
 * a key j when every row that sees j is in range).
 *
 * Return value: 0 on success, -1 on an invalid argument.
 */
#ifndef SINK_ORACLE_H
#define SINK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int sink_oracle_forward(int nseq, const int32_t* cu_seqlens, int h_q, int h_kv, int d,
                        double scale, int causal, int window, int row_begin, int row_end,
                        const double* q, const double* k, const double* v, const double* sinks,
                        double* o, double* lse);

int sink_oracle_backward(int nseq, const int32_t* cu_seqlens, int h_q, int h_kv, int d,
                         double scale, int causal, int window, int row_begin, int row_end,
                         const double* q, const double* k, const double* v, const double* sinks,
                         const double* dout,
                         double* dq, double* dk, double* dv, double* dsinks);

/* One row in full: the combined probability vector p over the row's allowed
 * keys followed by the sink (length n+1), and the gradient dz of the loss with
 * respect to every entry of the combined score row (same length; the last entry
 * is that row's contribution to dL/dS_h). dout may be NULL, then dz is not
 * written. *first_key receives the position of the first allowed key; the
 * return value is n (number of allowed keys), or -1 on an invalid argument.
 * p and dz must hold at least (longest sequence + 1) entries. */
int sink_oracle_row(int nseq, const int32_t* cu_seqlens, int h_q, int h_kv, int d,
                    double scale, int causal, int window,
                    const double* q, const double* k, const double* v, const double* sinks,
                    const double* dout, int seq, int head, int row,
                    double* p, double* dz, int* first_key);

int sink_oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
