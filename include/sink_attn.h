/*
 * sink_attn.h - C ABI of libsinkattn: forward and backward of causal /
 * sliding-window grouped-query attention with one learnable sink logit per
 * query head, for NVIDIA GB300 (sm_103a).
 *
 * What is computed. The operation is the one defined on the page
 * "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！" (nmedialink.com):
 *   - section "GPT-OSS中的带注意力槽的注意力机制": the scaled scores of a row are
 *     concatenated with the head's sink logit, softmax runs over the N_k + 1
 *     columns, the sink column is dropped, and the remaining probabilities
 *     multiply V;
 *   - section "数学公式深入解读": P_ij = exp(S_ij) / (sum_j' exp(S_ij') + exp(S_h))
 *     with S_ij = scale * Q_i . K_j, and the sink probability
 *     P_{i,h} = exp(S_h) / (same denominator);
 *   - section "反向传播的实现": dL/dS_h = -sum_i P_{i,h} sum_j P_ij dL/dP_ij,
 *     which equals -sum_i P_{i,h} * (dO_i . O_i) because the sink column has
 *     no upstream gradient.
 * Readings where the page is silent: the sink is a raw logit (not multiplied
 * by the scale); there is one sink per query head; a window W means keys
 * i-W+1 .. i and is always causal; packed sequences are masked independently,
 * with positions counted from each sequence's start.
 *
 * Per row i of query head h (key/value head h / (h_q / h_kv)):
 *   A(i)   = allowed keys: all keys of the sequence (causal = 0), keys 0..i
 *            (causal = 1, window <= 0) or keys max(0, i-W+1)..i (window = W);
 *   M_i    = max(S_h, max_{j in A(i)} S_ij)
 *   LSE_i  = M_i + ln(exp(S_h - M_i) + sum_{j in A(i)} exp(S_ij - M_i))
 *   O_i    = sum_{j in A(i)} exp(S_ij - LSE_i) V_j
 *
 * Layouts (row-major, contiguous, device memory):
 *   padded (cu_seqlens == NULL): q/o/dout/dq [B, N, h_q, d], k/v/dk/dv [B, N, h_kv, d]
 *   packed (cu_seqlens != NULL): q/o/dout/dq [T, h_q, d],     k/v/dk/dv [T, h_kv, d]
 *   sinks, dsinks: [h_q] fp32.  lse: [h_q, T] fp32 (T = B * N when padded).
 *   cu_seqlens: int32 [batch + 1], device memory, cu_seqlens[0] = 0,
 *   non-decreasing, cu_seqlens[batch] = total_tokens.
 * Every pointer must be 16-byte aligned (cu_seqlens: 4-byte). q/k/v/o/dout/dq/dk/dv use the dtype
 * given in the params; sinks, dsinks and lse are always fp32.
 *
 * Ownership and execution. The caller allocates every buffer, including the
 * workspace (size from sink_attn_workspace_bytes). No entry point allocates,
 * frees or synchronises except sink_attn_fetch_device_error, which says so.
 * Work is enqueued on the caller's stream; outputs are valid once that stream
 * reaches the enqueued work, so every other entry point may be captured in a
 * CUDA graph and replayed. Outputs (o, lse, dq, dk, dv, dsinks) are
 * overwritten, never accumulated into. Inputs are not modified.
 *
 * Errors. Every entry point returns a status. Arguments are validated before
 * anything is enqueued; an invalid call enqueues nothing. A failed launch is
 * reported as SINK_ERR_CUDA. Conditions found on the device set a flag word at
 * the start of the workspace; sink_attn_fetch_device_error reads and clears
 * it. Its bits:
 *   SINK_FLAG_TIMEOUT      a bounded wait inside a kernel gave up (the wait
 *                          limit is sink_attn_set_wait_limit_ns); the outputs
 *                          of that call are invalid;
 *   SINK_FLAG_SEQ_TOO_LONG a sequence is longer than max_seqlen: its rows and
 *                          keys past max_seqlen were not computed (their
 *                          outputs are left as they were, except dq on the
 *                          default bf16 64-wide path, written as 0);
 *   SINK_FLAG_BAD_SEQLENS  cu_seqlens is not a valid packing: some
 *                          cu_seqlens[s] < 0, cu_seqlens[s+1] < cu_seqlens[s],
 *                          cu_seqlens[s+1] > total_tokens, or cu_seqlens[0]
 *                          != 0. cu_seqlens lives in device memory, so this is
 *                          checked by the kernels: every kernel checks the
 *                          bounds of its sequence before any load or store and
 *                          skips a sequence that fails (its rows of o and lse
 *                          and its keys' dk and dv are left as they were; its
 *                          rows of dq too, except on the default bf16 64-wide
 *                          path, which writes 0 there). Other sequences are
 *                          computed.
 * Nothing is thrown across the ABI.
 *
 * Precision of D. The backward forms D_i = dout_i . O_i from the forward's
 * output. The plain entry points (sink_attn_fwd / sink_attn_bwd) use the
 * stored O, which carries its own rounding to the output dtype; with bf16 and
 * sharp attention (dP_ij close to D_i) that rounding reaches dq, dk and dsinks
 * through dS = P (dP - D). The _ex entry points take an extra buffer o_lo
 * (same shape and dtype as o, bf16 only): the forward writes into it what the
 * rounding of O to bf16 dropped, bf16(O - bf16(O)), and the backward forms
 * D from o + o_lo, about 16 bits of O. Training code keeps o_lo with o and lse
 * between the forward and the backward.
 */
#ifndef SINK_ATTN_H
#define SINK_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SINK_API __attribute__((visibility("default")))
#else
#define SINK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Bits of the device flag word (see Errors above). */
#define SINK_FLAG_TIMEOUT 1u
#define SINK_FLAG_SEQ_TOO_LONG 2u
#define SINK_FLAG_BAD_SEQLENS 4u

typedef struct CUstream_st* sink_stream_t; /* same object as cudaStream_t; NULL = legacy default stream */

typedef enum {
    SINK_OK = 0,
    SINK_ERR_INVALID_ARG = 1,  /* a NULL/misaligned pointer, a bad size or an inconsistent field */
    SINK_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head_dim not 64 or 128) */
    SINK_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    SINK_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than sink_attn_workspace_bytes */
    SINK_ERR_TIMEOUT = 5,      /* a kernel's bounded wait gave up (reported by fetch_device_error) */
    SINK_ERR_DEVICE = 6,       /* another condition flagged on the device (see fetch_device_error) */
    SINK_ERR_SCRATCH_LIMIT = 7 /* problem too large for the fixed scratch of a _noalloc entry point */
} sink_status_t;

typedef enum { SINK_BF16 = 0, SINK_FP32 = 1 } sink_dtype_t;

typedef struct {
    int batch;            /* number of sequences: B (padded) or the length of cu_seqlens minus 1 */
    int max_seqlen;       /* N (padded) or an upper bound on every packed sequence's length */
    int total_tokens;     /* T: B * N (padded) or cu_seqlens[batch] (packed) */
    int h_q;              /* query heads; a multiple of h_kv */
    int h_kv;             /* key/value heads */
    int head_dim;         /* d: 64, or 128 (training entry points only; decode takes 64) */
    sink_dtype_t dtype;   /* dtype of q, k, v, o, dout, dq, dk, dv */
    float softmax_scale;  /* scale applied to Q.K; <= 0 selects 1/sqrt(head_dim) */
    int causal;           /* 1: causal mask; 0: every key of the sequence (window must be 0) */
    int window;           /* <= 0: no window; W > 0: keys i-W+1 .. i (requires causal = 1) */
} sink_attn_params_t;

/* Bytes of device workspace that sink_attn_fwd (is_bwd = 0) or sink_attn_bwd /
 * sink_attn_bwd_preprocess / sink_attn_bwd_main (is_bwd = 1) need for these
 * params. Returns 0 if the params are invalid. The workspace needs no
 * initialisation and may be reused across calls on the same stream. */
SINK_API size_t sink_attn_workspace_bytes(const sink_attn_params_t* params, int is_bwd);

/* Forward (sections "GPT-OSS中的带注意力槽的注意力机制" and "数学公式深入解读"):
 * writes o (input dtype) and lse (fp32 [h_q, T], natural log, sink included). */
SINK_API sink_status_t sink_attn_fwd(const sink_attn_params_t* params,
                            const void* q, const void* k, const void* v,
                            const float* sinks, const int32_t* cu_seqlens,
                            void* o, float* lse,
                            void* workspace, size_t workspace_bytes, sink_stream_t stream);

/* Forward as sink_attn_fwd, and, when o_lo is not NULL (bf16 params only;
 * NULL is required for fp32), o_lo [same shape as o] receives
 * bf16(O - bf16(O)) per element, the part of O that the bf16 output dropped
 * (see "Precision of D" above). o and lse are identical to sink_attn_fwd's. */
SINK_API sink_status_t sink_attn_fwd_ex(const sink_attn_params_t* params,
                               const void* q, const void* k, const void* v,
                               const float* sinks, const int32_t* cu_seqlens,
                               void* o, void* o_lo, float* lse,
                               void* workspace, size_t workspace_bytes, sink_stream_t stream);

/* Full backward (section "反向传播的实现"): given the forward's o and lse and the
 * upstream gradient dout, writes dq (input dtype), dk, dv (input dtype, summed
 * over the query heads of each key/value head) and dsinks (fp32 [h_q],
 * dL/dS_h summed over every sequence and row of head h, reduced in a fixed
 * order so it is bitwise reproducible). dk, dv and dsinks are bitwise
 * reproducible; dq on the bf16 d = 64 path is summed over key blocks by fp32
 * reduce-adds into the workspace in an order that varies between runs, so it
 * may differ in the last bf16 place, unless sink_attn_set_deterministic is on
 * (at d = 128 and in fp32 it is reproducible either way). Equivalent to
 * sink_attn_bwd_preprocess into workspace followed by sink_attn_bwd_main. */
SINK_API sink_status_t sink_attn_bwd(const sink_attn_params_t* params,
                            const void* q, const void* k, const void* v,
                            const float* sinks, const int32_t* cu_seqlens,
                            const void* o, const float* lse, const void* dout,
                            void* dq, void* dk, void* dv, float* dsinks,
                            void* workspace, size_t workspace_bytes, sink_stream_t stream);

/* Full backward as sink_attn_bwd, with D formed from o + o_lo (o_lo from
 * sink_attn_fwd_ex; NULL gives exactly sink_attn_bwd). dv does not depend on
 * D and equals sink_attn_bwd's. Equivalent to sink_attn_bwd_preprocess_ex
 * into workspace followed by sink_attn_bwd_main. */
SINK_API sink_status_t sink_attn_bwd_ex(const sink_attn_params_t* params,
                               const void* q, const void* k, const void* v,
                               const float* sinks, const int32_t* cu_seqlens,
                               const void* o, const void* o_lo, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, float* dsinks,
                               void* workspace, size_t workspace_bytes, sink_stream_t stream);

/* Backward step 1 (section "反向传播的实现", simplified equation): writes
 * delta[h, t] = dout_t,h . o_t,h (fp32 [h_q, T]) and
 * dsinks[h] = -sum_t exp(S_h - lse[h, t]) * delta[h, t]. Memory-bound. */
SINK_API sink_status_t sink_attn_bwd_preprocess(const sink_attn_params_t* params,
                                       const float* sinks, const void* o, const float* lse,
                                       const void* dout, float* delta, float* dsinks,
                                       void* workspace, size_t workspace_bytes,
                                       sink_stream_t stream);

/* Backward step 1 as above, with delta[h, t] = dout_t,h . (o_t,h + o_lo_t,h)
 * when o_lo is not NULL (bf16 only). */
SINK_API sink_status_t sink_attn_bwd_preprocess_ex(const sink_attn_params_t* params,
                                          const float* sinks, const void* o, const void* o_lo,
                                          const float* lse, const void* dout, float* delta,
                                          float* dsinks, void* workspace, size_t workspace_bytes,
                                          sink_stream_t stream);

/* Backward step 2 (section "反向传播的实现": the gradients of the scores and
 * through them of Q, K and V; the sink's own gradient is step 1's): recomputes
 * P = exp(S - lse), which needs no sink term because lse includes the sink,
 * and writes dq, dk, dv using delta from step 1:
 * dS_ij = P_ij (dout_i . v_j - delta_i), dq = scale dS K, dk = scale dS^T Q,
 * dv = P^T dout. */
SINK_API sink_status_t sink_attn_bwd_main(const sink_attn_params_t* params,
                                 const void* q, const void* k, const void* v,
                                 const int32_t* cu_seqlens, const float* lse,
                                 const float* delta, const void* dout,
                                 void* dq, void* dk, void* dv,
                                 void* workspace, size_t workspace_bytes, sink_stream_t stream);

/* Backward step 2 split in two, so that its memory-bound preparation can run
 * early. The preparation depends on q and k alone: on the bf16 d = 64 path it
 * writes f16 copies of q and k into the workspace and zeroes the fp32 dQ
 * accumulator there (the fused backward's reduce-adds land in it); on every
 * other path it does nothing. A caller that has q and k before the forward's
 * outputs exist can issue sink_attn_bwd_prepare on a second, lower-priority
 * stream while the forward runs (its blocks then take the SMs the forward's
 * last wave leaves idle), and later sink_attn_bwd_main_ex with
 * SINK_BWD_PREPARED, which skips the pass.
 * The caller orders the two calls (an event), passes both the same params,
 * q, k and workspace (sized by sink_attn_workspace_bytes(params, 1)), and
 * leaves q, k and the workspace unchanged in between. No call that can run at
 * the same time as the preparation may use that workspace: the forward it
 * overlaps needs a workspace of its own (a different buffer), and an earlier
 * backward on the same workspace must have finished. Arguments and error
 * behaviour as sink_attn_bwd_main. */
SINK_API sink_status_t sink_attn_bwd_prepare(const sink_attn_params_t* params,
                                    const void* q, const void* k,
                                    void* workspace, size_t workspace_bytes, sink_stream_t stream);

/* options bits of sink_attn_bwd_main_ex */
#define SINK_BWD_PREPARED 1u /* sink_attn_bwd_prepare already ran on this workspace */

/* sink_attn_bwd_main with options: options = 0 is exactly sink_attn_bwd_main;
 * SINK_BWD_PREPARED skips the preparation pass (see sink_attn_bwd_prepare).
 * Unknown option bits return SINK_ERR_INVALID_ARG. */
SINK_API sink_status_t sink_attn_bwd_main_ex(const sink_attn_params_t* params,
                                    const void* q, const void* k, const void* v,
                                    const int32_t* cu_seqlens, const float* lse,
                                    const float* delta, const void* dout,
                                    void* dq, void* dk, void* dv,
                                    void* workspace, size_t workspace_bytes,
                                    unsigned options, sink_stream_t stream);

/* Reads and clears the device flag word at the start of a workspace that was
 * passed to the calls above. SYNCHRONISES the stream (it copies 4 bytes back).
 * Returns SINK_OK, SINK_ERR_TIMEOUT (SINK_FLAG_TIMEOUT is set: outputs of that
 * call are invalid), SINK_ERR_DEVICE (another SINK_FLAG_* bit is set: a
 * sequence exceeded max_seqlen, or cu_seqlens is not a valid packing) or
 * SINK_ERR_CUDA. *flags_out (may be NULL) receives the raw flag bits. */
SINK_API sink_status_t sink_attn_fetch_device_error(void* workspace, size_t workspace_bytes,
                                           sink_stream_t stream, uint32_t* flags_out);

/* Backward step 1 without a workspace argument. No counterpart on the page:
 * this entry point exists for callers that are given their input and output
 * buffers but cannot obtain any other device memory (a plugin inside a host
 * framework that owns all device memory and offers no scratch allocator, or a
 * path where a cudaMalloc would synchronise the device or fail because a
 * caching allocator already holds the memory). It computes exactly what
 * sink_attn_bwd_preprocess computes, keeping its per-chunk dS_h partial sums
 * in a fixed device array inside the library (sink_attn_noalloc_scratch_bytes,
 * 1 MiB, held by every GPU that loads the library until the process exits).
 * It allocates and frees nothing. Limits: h_q * ceil(T / 256) partials must
 * fit the array, else SINK_ERR_SCRATCH_LIMIT is returned before anything is
 * enqueued. All calls on a device share the array, so calls whose work
 * overlaps on the GPU race; order them on one stream. The first call on each
 * device (with that device current) looks up the array's device address;
 * make that first call before any stream capture. */
SINK_API sink_status_t sink_attn_bwd_preprocess_noalloc(const sink_attn_params_t* params,
                                                        const float* sinks, const void* o,
                                                        const float* lse, const void* dout,
                                                        float* delta, float* dsinks,
                                                        sink_stream_t stream);

/* Size in bytes of the fixed scratch array used by the _noalloc entry point. */
SINK_API size_t sink_attn_noalloc_scratch_bytes(void);

/* Decode / streaming inference: one query per entry b against a key/value
 * cache. The page's sinks exist for streaming inference (section
 * "FlashAttentionV3对注意力槽的支持"), and its section "纠正训练与推理不一致问题"
 * (Fig. 4) measures the gap between the training and inference attention
 * paths; this is the inference path, and its o and lse for query b equal row
 * kv_len[b] - 1 of sink_attn_fwd on the same context (same definitions as
 * above: the sink joins the denominator once, adds no value row, and lse
 * includes it).
 * Query b is the last token of its context, cache rows kv_start[b] ..
 * kv_start[b] + kv_len[b] - 1; it sees all of them, or the last `window` of
 * them when window > 0.
 * Params: batch = number of queries; total_tokens = rows of the cache;
 * max_seqlen = an upper bound on every kv_len; h_q, h_kv, head_dim (64),
 * dtype, softmax_scale, window; causal must be 1.
 * Layouts (device memory): q, o [batch, h_q, d]; k_cache, v_cache
 * [total_tokens, h_kv, d]; sinks [h_q] fp32; lse [h_q, batch] fp32;
 * kv_start, kv_len int32 [batch] (4-byte aligned); the others 16-byte aligned.
 * The keys of each query are split into chunks whose partial results
 * (without the sink) are merged with the sink counted once; the workspace
 * (sink_attn_decode_workspace_bytes) holds the partials and one chunk counter
 * per (query, key/value head). It needs no initialisation: the call zeroes
 * the flag word and the counters on the stream first, so calls that share a
 * workspace must be ordered on one stream. The call only enqueues stream work
 * (one memset, one or two kernels), so it may be captured in a CUDA graph.
 * A query whose kv_len is < 1 or > max_seqlen, or whose
 * context runs past the end of the cache, reads no key: it gets the result
 * of an empty key set (o = 0, lse = S_h), and the flag word reports
 * SINK_ERR_DEVICE through sink_attn_fetch_device_error. */
SINK_API size_t sink_attn_decode_workspace_bytes(const sink_attn_params_t* params);
SINK_API sink_status_t sink_attn_decode(const sink_attn_params_t* params,
                                        const void* q, const void* k_cache, const void* v_cache,
                                        const float* sinks, const int32_t* kv_start,
                                        const int32_t* kv_len, void* o, float* lse,
                                        void* workspace, size_t workspace_bytes,
                                        sink_stream_t stream);

/* Static description of a status code. Never NULL. */
SINK_API const char* sink_attn_status_str(sink_status_t status);

/* Every wait inside the tensor-core kernels (on a copy or a product another
 * warp issued) gives up after a time limit, raises SINK_FLAG_TIMEOUT and lets
 * the kernel wind down, instead of hanging the GPU. Sets that limit for calls
 * made after this one, in nanoseconds, process-wide; 0 restores the default
 * (2 s). Returns the previous limit. A limit far below a kernel's normal
 * waiting time makes correct calls fail with SINK_ERR_TIMEOUT. */
SINK_API uint64_t sink_attn_set_wait_limit_ns(uint64_t limit_ns);

/* Reproducible dq (process-wide, for calls made after this one; returns the
 * previous setting). Off (0, the default): the bf16 64-wide backward sums dq
 * over key blocks by fp32 reduce-adds whose order varies between runs, so dq
 * may differ in the last bf16 place from run to run (dk, dv and dsinks are
 * always reproducible). On (1): that backward runs as two kernels instead, a
 * key-owning one for dk and dv and a query-owning one that sums each dq row in
 * a fixed order and writes it once, so dq is reproducible bit for bit; it
 * recomputes the scores for dq and takes about 1.45x as long. The workspace
 * size (sink_attn_workspace_bytes) depends on this setting. Other paths are
 * reproducible either way. */
SINK_API int sink_attn_set_deterministic(int on);

/* Number of kernels this library has enqueued in the calling process so far
 * (all entry points, all devices). Host-side counter; never synchronises. */
SINK_API uint64_t sink_attn_kernel_launches(void);

/* Library version as major * 10000 + minor * 100 + patch. */
SINK_API int sink_attn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SINK_ATTN_H */
