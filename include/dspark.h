/*
 * dspark.h -- C ABI of the batched speculative-decoding verify-and-sample epilogue
 * for one NVIDIA GB300 (sm_103a).
 *
 * One call takes, for B concurrent requests with up to K_max drafted tokens each,
 *   target logits  x [B, K_max+1, V]  (bf16 or fp32, row-major, V contiguous),
 *   draft probabilities q [B, K_max, V] (fp32),
 *   draft token ids d [B, K_max] (int32),
 * and per-request sampling parameters, and produces the accepted length, the emitted
 * tokens and (on request) their raw log-probabilities and the top log-probabilities.
 *
 * What each step computes, and the passage that defines it (mlx-dspark pages):
 *   - presence / frequency penalties on the TARGET logits; verify position j counts the
 *     request's completion history plus its own draft prefix d_0..d_{j-1}
 *     (mlx-dspark Changelog, [0.2.0] Added, "presence_penalty / frequency_penalty";
 *     v0.2.0 release notes, Highlights).  In float32: x' = x - ((f*c) + p) for c > 0,
 *     each operation rounded to nearest, no fused multiply-add;
 *   - temperature, then top-k and top-p truncation of target and draft alike
 *     (Changelog, [0.1.0] Added, "Lossless top-p / top-k sampling"), with the threshold
 *     and nucleus cutoff found by selection instead of a full vocabulary sort, giving the
 *     same truncated distribution (Changelog, [0.20.2] Changed).  The draft input holds
 *     probabilities at T=1; at temperature T the draft distribution is q^(1/T) normalised.
 *     top-k keeps every token tied with the k-th largest value; top-p acts on the
 *     renormalised top-k distribution and keeps a token iff the mass strictly above its
 *     value is < top_p;
 *   - T = 0 (greedy): accept the longest prefix where the penalised target argmax (lowest
 *     id on ties) equals the draft, then emit the argmax at the first mismatch or after
 *     the last draft (Changelog, [0.2.0] Changed, "One device sync per speculative round");
 *   - T > 0: accept draft i iff u[b][i][0] < P'(d_i)/Q'(d_i) (always when Q'(d_i) = 0 and
 *     P'(d_i) > 0); on the first rejection at a, draw from max(0, P'_a - Q'_a) normalised,
 *     or from P'_K when every draft was accepted (v0.0.2 release notes, Highlights,
 *     "Lossless temperature speculative sampling").  The draw is an inverse CDF over
 *     ascending token ids with u[b][a][1]: the smallest t whose cumulative mass exceeds
 *     u * total.  An all-zero residual draws from P'_a;
 *   - logprobs: raw (unpenalised, untempered, untruncated) target log-softmax at each
 *     emitted token, and the n largest raw logits (value descending, id ascending) with
 *     their log-softmax (Changelog, [0.2.0] Added, "logprobs / top_logprobs"); on request
 *     the same over the penalised logits x' instead (dspark_extras_t.logprob_mode);
 *   - optional (dspark_extras_t): draft rows given as m (id, probability) pairs, such as the
 *     one-hot proposal of prompt-lookup drafts (Changelog, [0.2.0] Added, "--mode lookup"),
 *     or over a reduced draft vocabulary widened through a d2t offset table, target id =
 *     draft id + d2t[draft id] (Changelog, [0.8.0] Added, reduced draft vocabularies); a
 *     per-request end-of-sequence token that ends the output at the first accepted draft
 *     equal to it (Changelog, [0.2.0] Fixed); per-position acceptance counters (Changelog,
 *     [0.9.0] Added, per-position acceptance with honest denominators).
 *
 * Conventions for every entry point:
 *   - All tensor pointers of dspark_verify_sample are DEVICE pointers owned by the caller.
 *     The library allocates nothing and keeps no state between calls.  Scratch memory is
 *     the caller's workspace (size from dspark_workspace_bytes).
 *   - Work is enqueued on params->stream and runs asynchronously; the return value covers
 *     argument validation and launch errors only.  Problems found on the device are
 *     reported per request in row_status (after the stream is synchronised); kernels never
 *     trap.  A request with a non-zero status gets accept_len = -1 and all tokens -1.
 *   - Calls that share a workspace must not overlap on the GPU.
 *   - dspark_verify_sample and dspark_verify_sample_host keep no global mutable state and may
 *     be called from several host threads at once (each with its own workspace).
 *     dspark_verify_sample_static is the exception: every call on a device shares one
 *     scratch array (see its comment).
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID_ARG = 1,   /* a null or misaligned pointer, or a size out of range */
    DSPARK_ERR_UNSUPPORTED = 2,   /* a shape or option this build does not support */
    DSPARK_ERR_WORKSPACE = 3,     /* workspace missing, too small or not 256-byte aligned */
    DSPARK_ERR_CUDA = 4           /* a CUDA runtime call or kernel launch failed */
} dspark_status_t;

typedef enum { DSPARK_BF16 = 0, DSPARK_FP32 = 1 } dspark_dtype_t;

/* Per-request status bits written to row_status[b] (0 = fine). */
#define DSPARK_ROW_BAD_PARAMS  1   /* T < 0 or not finite, top_p <= 0 or NaN, top_k < 0,
                                      num_drafts outside [0, K_max], non-finite penalty */
#define DSPARK_ROW_BAD_DRAFT   2   /* a draft id d[b][i], i < num_drafts, outside [0, V); with
                                      T > 0, a sparse draft row (i < num_drafts) with an id
                                      outside [0, V) or a repeated id, or a d2t table that maps
                                      a draft id outside [0, V) or two draft ids to one target */
#define DSPARK_ROW_NONFINITE   4   /* a non-finite target logit, a negative / non-finite
                                      draft probability, or a draft row with no mass */
#define DSPARK_ROW_BAD_HISTORY 8   /* history ids outside [0, V) / not strictly ascending,
                                      or a count <= 0 */
#define DSPARK_ROW_INTERNAL   16   /* an internal limit was hit (bounded wait expired) */

/* Largest supported sizes. */
#define DSPARK_MAX_B          2048
#define DSPARK_MAX_V          (1 << 24)
#define DSPARK_MAX_K          64
#define DSPARK_MAX_TOP_LOGPROBS 20
#define DSPARK_MAX_SPARSE_M   256  /* (id, probability) pairs per sparse draft row */

/* Sampling parameters of one request (24 bytes, device array of B). */
typedef struct {
    float   temperature;        /* 0 = greedy; > 0 = speculative sampling at T       */
    int32_t top_k;              /* 0 or >= V: off                                   */
    float   top_p;              /* in (0, 1]; >= 1: off                              */
    float   presence_penalty;   /* OpenAI presence penalty (target only)            */
    float   frequency_penalty;  /* OpenAI frequency penalty (target only)           */
    int32_t num_drafts;         /* K_b in [0, K_max]                                 */
} dspark_row_params_t;

/* Completion-count history of each request, CSR over requests (device pointers).
 * token_ids are strictly ascending within a request; counts are > 0.  A NULL
 * dspark_counts_t pointer, or row_offsets == NULL, means no history for any request. */
typedef struct {
    const int32_t* row_offsets;   /* [B+1], row_offsets[0] = 0 */
    const int32_t* token_ids;     /* [nnz] */
    const int32_t* counts;        /* [nnz] */
} dspark_counts_t;

/* Layout of the draft input q. */
typedef enum {
    DSPARK_Q_DENSE = 0,           /* q [B, K_max, V]: probabilities over the target vocabulary  */
    DSPARK_Q_SPARSE = 1,          /* q [B, K_max, m] probabilities of the ids q_ids [B, K_max, m];
                                     every other token has probability 0 (m = 1, q = 1: the
                                     one-hot proposal of a lookup draft)                         */
    DSPARK_Q_REDUCED = 2          /* q [B, K_max, Vd] over a draft vocabulary of Vd ids; draft id
                                     e stands for target id e + d2t[e], every other target id
                                     has probability 0                                           */
} dspark_q_layout_t;

typedef enum {
    DSPARK_LOGPROBS_RAW = 0,      /* log-softmax of the raw target logits x                     */
    DSPARK_LOGPROBS_PENALISED = 1 /* log-softmax of the penalised logits x' (no temperature)    */
} dspark_logprob_mode_t;

/* Options beyond the dense call (host struct; its arrays are device pointers, or host pointers
 * for dspark_verify_sample_host).  A NULL dspark_params_t.extras means: dense q, no
 * end-of-sequence tokens, no counters, raw logprobs. */
typedef struct {
    dspark_q_layout_t q_layout;
    int32_t q_row_len;            /* sparse: m in 1..DSPARK_MAX_SPARSE_M; reduced: Vd in 1..V;
                                     dense: ignored                                              */
    const int32_t* q_ids;         /* sparse: [B, K_max, m] target ids (distinct within a row)    */
    const int32_t* d2t;           /* reduced: [Vd] offsets                                       */
    const int32_t* eos_ids;       /* [B] end-of-sequence token per request (< 0: none) or NULL    */
    int32_t* out_stopped;         /* [B] or NULL: 1 when the request stopped on its eos token    */
    unsigned long long* pos_counts; /* [2, K_max] or NULL.  ADDED to, never cleared: row 0, i: the
                                     requests that verified draft i (every earlier draft accepted,
                                     no stop before it, i < num_drafts); row 1, i: those that
                                     accepted it.  Zero it once, then it accumulates over calls.  */
    dspark_logprob_mode_t logprob_mode;
} dspark_extras_t;

typedef struct {
    int32_t B;                    /* requests, 1..DSPARK_MAX_B                        */
    int32_t K_max;                /* drafted tokens at most, 0..DSPARK_MAX_K          */
    int32_t V;                    /* vocabulary, 1..DSPARK_MAX_V                      */
    dspark_dtype_t logits_dtype;  /* dtype of x; q is always fp32                     */
    const dspark_row_params_t* rows;  /* device [B]                                  */
    int32_t want_logprobs;        /* non-zero: out_logprobs is written                */
    int32_t n_top_logprobs;       /* 0..DSPARK_MAX_TOP_LOGPROBS                       */
    void*   workspace;            /* device, 256-byte aligned                         */
    size_t  workspace_bytes;      /* >= dspark_workspace_bytes(params)                */
    void*   stream;               /* cudaStream_t; NULL = legacy default stream       */
    int32_t* row_status;          /* device [B], required                             */
    void*   stage_events[2];      /* optional cudaEvent_t pair recorded on the stream
                                     right before and right after the streaming-stats
                                     kernel (for its roofline timing); NULL = none     */
    const dspark_extras_t* extras;  /* host pointer or NULL (see dspark_extras_t)      */
} dspark_params_t;

/* Scratch bytes dspark_verify_sample needs for these shapes (B, K_max, V, logits_dtype,
 * n_top_logprobs, and the draft layout of params->extras).  Returns 0 if the shapes are
 * unsupported. */
size_t dspark_workspace_bytes(const dspark_params_t* params);

/*
 * The verify-and-sample epilogue on device buffers.
 *   logits            x [B, K_max+1, V] of params->logits_dtype, 4-byte aligned
 *   q                 [B, K_max, V] fp32 (other layouts: dspark_extras_t), 4-byte aligned;
 *                     may be NULL when every request is greedy
 *   draft_ids         [B, K_max] int32 (entries past num_drafts are ignored)
 *   counts            history (may be NULL)
 *   uniforms          [B, K_max+1, 2] fp32 in [0, 1): [.., j, 0] accept draw at j,
 *                     [.., j, 1] resample / bonus draw at j
 *   out_accept_len    [B] int32: accepted drafts a (-1 for a request with an error)
 *   out_tokens        [B, K_max+1] int32: d_0..d_{a-1}, then the drawn token, then -1
 *                     (a request stopped on its eos token: d_0..d_{a-1} with d_{a-1} = eos,
 *                     then -1; nothing is drawn)
 *   out_logprobs      [B, K_max+1] fp32 or NULL; -inf past the last emitted token
 *   out_top_ids       [B, K_max+1, n_top_logprobs] int32 or NULL; -1 past the emitted token
 *   out_top_logprobs  [B, K_max+1, n_top_logprobs] fp32 or NULL; -inf past the emitted token
 */
dspark_status_t dspark_verify_sample(const void* logits, const float* q, const int32_t* draft_ids,
                                     const dspark_counts_t* counts, const dspark_params_t* params,
                                     const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                                     float* out_logprobs, int32_t* out_top_ids, float* out_top_logprobs);

/* Device bytes dspark_verify_sample_host needs: the workspace plus staging for the inputs
 * and outputs of one call with counts_nnz history entries. */
size_t dspark_host_workspace_bytes(const dspark_params_t* params, int64_t counts_nnz);

/*
 * The same epilogue from HOST buffers (same layouts as above; pinned host memory gives
 * full copy bandwidth).  params->rows, params->row_status, the dspark_counts_t arrays and the
 * arrays of params->extras are HOST pointers here (pos_counts is read, added to and written
 * back); params->workspace is a device buffer of at least
 * dspark_host_workspace_bytes.  The call copies the inputs to the device, runs the
 * epilogue, copies the outputs back and synchronises params->stream before returning.
 */
dspark_status_t dspark_verify_sample_host(const void* logits, const float* q, const int32_t* draft_ids,
                                          const dspark_counts_t* counts, const dspark_params_t* params,
                                          const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                                          float* out_logprobs, int32_t* out_top_ids, float* out_top_logprobs);

/* Size of the fixed device scratch of dspark_verify_sample_static (per device). */
#define DSPARK_STATIC_WORKSPACE_BYTES (16u << 20)

/*
 * dspark_verify_sample with no workspace argument, for callers that cannot call cudaMalloc:
 * for instance a serving loop that reserved all device memory up front and hands out no
 * allocator, or a plugin inside a host framework that owns the device memory and does not
 * expose its allocator.  The scratch is a file-scope device array of
 * DSPARK_STATIC_WORKSPACE_BYTES (16 MiB), which every device that loads the library holds
 * until the process exits; the call makes no cudaMalloc / cudaFree or other allocating call.
 * This entry point has no counterpart in the mlx-dspark pages.
 *   - Arguments, layouts and results are those of dspark_verify_sample; the caller still
 *     passes inputs and outputs.  params->workspace and params->workspace_bytes are ignored.
 *   - Shapes whose dspark_workspace_bytes exceeds DSPARK_STATIC_WORKSPACE_BYTES are rejected
 *     with DSPARK_ERR_UNSUPPORTED before any CUDA call.
 *   - Set-up: the first call on a device looks the array's address up (cudaGetSymbolAddress,
 *     with that device current) and caches it for that device; make that first call before
 *     any stream capture.  A failed lookup returns DSPARK_ERR_CUDA.  The cached address
 *     belongs to the device's primary context: after cudaDeviceReset it is stale, so do not
 *     call this entry point again in that process.
 *   - Nothing in the scratch has to start at zero: every call clears the one record it reads
 *     before writing (with cudaMemsetAsync on params->stream).  The array keeps the last
 *     call's contents.
 *   - All calls on one device share the array: calls that overlap on the GPU (other streams,
 *     other host threads) race and give undefined results.  Serialise them.
 */
dspark_status_t dspark_verify_sample_static(const void* logits, const float* q, const int32_t* draft_ids,
                                            const dspark_counts_t* counts, const dspark_params_t* params,
                                            const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                                            float* out_logprobs, int32_t* out_top_ids, float* out_top_logprobs);

/* Human-readable name of a status code. */
const char* dspark_status_string(dspark_status_t status);

/* Number of kernel launches one dspark_verify_sample call makes when it asks for logprobs
 * (want_logprobs or n_top_logprobs > 0); one fewer otherwise. */
int32_t dspark_launches_per_call(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
