/*
 * csa.h -- C ABI of the GB300 compressed sparse attention (CSA) decode step.
 *
 * One decode step of DeepSeek-V4-style compressed sparse attention, per query
 * token (hw-native-sys/pypto-lib pages):
 *   (a) indexer score of every causally visible ratio-r compressed row,
 *       score_j = sum_h w_h * ReLU(q_idx[h] . k_idx[j]), summed over h in
 *       ascending order (no atomics: "Fix: port the DeepSeek-V4 MoE, hc_pre
 *       and prefill fixes to DSpark", PR description, deterministic ordered
 *       reduction);
 *   (b) Top-K of those scores, ties to the lower index; when the visible rows
 *       fit K (vis <= K) scoring and sorting are skipped and every visible
 *       row is taken ("Perf: skip redundant CSA scoring and fuse gather
 *       unpack", PR description);
 *   (c) gather of the selected compressed rows plus the last WIN raw rows,
 *       at most WIN + min(vis, K) rows ("Fix: port the DeepSeek-V4 MoE ...",
 *       PR description, packed sparse CSA row bound);
 *   (d) attention of H heads over rows shared by all heads (row width D, the
 *       first V dims are values), one softmax stream for the window rows,
 *       one for the compressed rows (and one for heavy-compression rows when
 *       enabled), a log-sum-exp merge of the streams, then inverse RoPE on
 *       the last R = D - V output dims ("Perf: fuse HCA merge, inverse RoPE,
 *       and packing", PR description).
 *
 * Definitions used throughout (query s of request b, context length L_b
 * including the S new tokens; S = 1 is single-token decode, a few tokens are
 * multi-token decode, and a prefill chunk of T tokens is S = T, each token
 * with its own visibility and Top-K):
 *   pos  = L_b - S + s                (0-based position of the query)
 *   vis  = floor((pos + 1) / ratio)   (compressed rows whose raw span ends at or before pos)
 *   nwin = min(WIN, pos + 1)          (window = raw rows pos-nwin+1 .. pos)
 *   cnt  = min(vis, K)
 *   vis2 = floor((pos + 1) / hca_ratio) when the heavy-compression stream is on
 * Inverse RoPE: for i < R/2, output dims (V-R+2i, V-R+2i+1) are rotated by
 * -pos * base^(-2i/R).
 *
 * Conventions
 *  - Every pointer in csa_batch and every output pointer is DEVICE memory
 *    owned by the caller.  The library never frees or retains them.
 *  - Every call is asynchronous on the given CUDA stream (a cudaStream_t
 *    passed as void*; NULL = legacy default stream).  No call synchronises
 *    except csa_get_status and csa_decode_destroy.
 *  - Element types: CSA_DTYPE_BF16 (bf16 storage, fp32 arithmetic) or
 *    CSA_DTYPE_F32.  Strides are in ELEMENTS; every row must start on a
 *    16-byte boundary (pointer and stride*element_size multiples of 16).
 *  - Row r of pool X for request b is at X + (X_off[b] + r) * X_stride, or
 *    where the pool's block table puts it (paged pools, see csa_batch).
 *    X_rows is the number of rows the pool holds; a row index outside
 *    [0, X_rows) is never dereferenced: it sets CSA_ERR_BAD_INDEX in the
 *    handle's status word and the row is skipped.
 *  - Errors found on the host return a non-zero code before any launch and
 *    leave the outputs untouched; csa_last_error() describes the last one
 *    on the calling thread.  Errors found on the device (bad lengths or row
 *    indices in device memory) are recorded in the status word, the affected
 *    query's output is written as zeros, and csa_get_status reports them.
 *  - A handle may be used from one host thread at a time.  Calls that share
 *    a handle must be ordered on the GPU (same stream, or the caller orders
 *    them): they share the handle's workspace.
 *  - Several devices in one process: a handle belongs to the device that was
 *    current at csa_decode_create and must be used with that device current.
 *    Handles of different devices may be used from different host threads
 *    at the same time; the library's per-device set-up (kernel shared-memory
 *    opt-ins) is done once per device, under a lock.
 *  - Value range: the kernels accumulate in fp32, so products and sums of
 *    the inputs (q . row over D dims, softmax-weighted sums of rows, indexer
 *    dot products) must stay within the fp32 range; any bf16 magnitude is
 *    otherwise accepted (intermediate attention partials are bf16).
 */
#ifndef CSA_H
#define CSA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSA_ABI_VERSION 3

#if defined(__GNUC__)
#define CSA_API __attribute__((visibility("default")))
#else
#define CSA_API
#endif

/* return codes */
enum {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer or stride  */
    CSA_ERR_UNSUPPORTED = 2, /* shape or dtype outside the compiled set               */
    CSA_ERR_WORKSPACE = 3,   /* B, S or a length above the create-time maxima         */
    CSA_ERR_CUDA = 4,        /* a CUDA runtime call failed (message in last_error)    */
    CSA_ERR_BAD_INDEX = 5,   /* device-side: a length or row index out of range       */
    CSA_ERR_TIMEOUT = 6      /* device-side: a bounded wait gave up                   */
};

enum { CSA_DTYPE_F32 = 0, CSA_DTYPE_BF16 = 1, CSA_DTYPE_FP8_E4M3 = 2 };

/* Static shape of one attention layer; fixed at csa_decode_create. */
typedef struct {
    int32_t heads;     /* H: attention heads                                   */
    int32_t row_dim;   /* D: width of a KV row (values + rope dims)            */
    int32_t v_dim;     /* V: value / output dims, V < D, R = D - V even        */
    int32_t idx_heads; /* Hi: indexer heads                                    */
    int32_t idx_dim;   /* Di: indexer dim                                      */
    int32_t ratio;     /* compression ratio of the CSA rows (4)                */
    int32_t topk;      /* K                                                    */
    int32_t win;       /* WIN: sliding window, >= 1                            */
    int32_t hca_ratio; /* ratio of the heavy-compression stream; 0 = off       */
    int32_t dtype;     /* CSA_DTYPE_BF16 or CSA_DTYPE_F32                      */
    float softmax_scale; /* <= 0 selects 1/sqrt(D)                             */
    float rope_base;     /* RoPE base (10000)                                  */
    int32_t max_batch;   /* workspace bound on B                               */
    int32_t max_queries_per_req; /* workspace bound on S                       */
    int32_t max_context; /* workspace bound on every L_b                       */
    /* Storage of the indexer key pool (idx_k): 0 = the layer dtype, or
     * CSA_DTYPE_FP8_E4M3 = one byte per key element (OCP FP8 E4M3: 1 sign,
     * 4 exponent bits with bias 7, 3 mantissa bits, subnormals, no
     * infinities, NaN = S.1111.111) with one fp32 scale per pool row, the
     * key being idx_scale[row] * e4m3(byte).  The pages pass the indexer
     * cache as a key pool plus a per-row scale pool ("Fix: complete DeepSeek
     * V4 TP CSA decode", PR description: idx_kv_cache and idx_kv_scale); the
     * element format is this library's choice.  FP8 keys need dtype bf16,
     * idx_heads 64 and idx_dim 128 (the tcgen05 indexer), else
     * CSA_ERR_UNSUPPORTED.  The score is unchanged:
     * score_j = sum_h w_h * ReLU(q_idx[h] . key_j). */
    int32_t idx_dtype;
} csa_config;

/* One batch.  All pointers: caller-owned device memory. */
typedef struct {
    int32_t B, S;             /* requests, queries per request (B = 0: no-op)   */
    const int32_t *ctx_len;   /* [B] L_b, including the S new tokens; S <= L_b <= max_context */
    const int32_t *ctx_len_host; /* optional HOST copy of ctx_len (same values):
                                    lets the host size grids exactly and skip
                                    launches with no work; NULL = size for the
                                    create-time maxima                          */
    const void *q;            /* [B,S,H,D]                                      */
    const void *q_idx;        /* [B,S,Hi,Di]                                    */
    const float *w;           /* [B,S,Hi] fp32 indexer head weights             */
    const void *raw_kv;  const int64_t *raw_off; int64_t raw_stride; int64_t raw_rows; /* raw rows, width D */
    const void *cmp_kv;  const int64_t *cmp_off; int64_t cmp_stride; int64_t cmp_rows; /* ratio rows, width D */
    const void *idx_k;   const int64_t *idx_off; int64_t idx_stride; int64_t idx_rows; /* indexer keys, width Di */
    const void *hca_kv;  const int64_t *hca_off; int64_t hca_stride; int64_t hca_rows; /* heavy rows, width D; NULL if off */
    const float *idx_scale;   /* [idx_rows] per-row scale of FP8 indexer keys (16-byte
                                 aligned); required with idx_dtype FP8, else ignored.
                                 idx_stride is then in bytes (a multiple of 16). */
    /* Paged pools (optional; NULL tables = the contiguous layout above).  With
     * X_table given, logical row r of request b in pool X is pool row
     * X_table[b * table_stride + r / X_block] * X_block + r % X_block, and
     * X_off is not read (it may be NULL).  A negative table entry is an
     * unmapped block: a row the step needs there is skipped and reported as
     * CSA_ERR_BAD_INDEX.  Raw rows are indexed by position (r in [0, L_b));
     * compressed, indexer-key and heavy rows by their index in the request.
     * idx_block must be a multiple of 128 (the indexer reads 128 keys at a
     * time); FP8 key scales follow the key rows.  Tables are device int32
     * arrays of B * table_stride entries. */
    const int32_t *raw_table, *cmp_table, *idx_table, *hca_table;
    int32_t raw_block, cmp_block, idx_block, hca_block;
    int32_t table_stride;
} csa_batch;

typedef struct csa_handle csa_handle;

/* Validates cfg and allocates the handle's device workspace on the current
 * device (scores [B*S, max_context/ratio] fp32, plan and status words).
 * Returns CSA_ERR_INVALID_ARG / CSA_ERR_UNSUPPORTED for a bad cfg,
 * CSA_ERR_CUDA if allocation fails.  *out is set only on success. */
CSA_API int csa_decode_create(const csa_config *cfg, csa_handle **out);

/* Synchronises the device, frees the workspace and the handle.  NULL is a no-op. */
CSA_API void csa_decode_destroy(csa_handle *h);

/* Steps (a)+(b).  topk_idx [B,S,K] int32: the selected compressed-row
 * indices of each query in ascending order, slots >= count set to -1;
 * topk_cnt [B,S] int32: count = min(vis, K).  ("Perf: skip redundant CSA
 * scoring and fuse gather unpack": bounded Top-K indices, bypass.) */
CSA_API int csa_indexer_topk(csa_handle *h, const csa_batch *b, int32_t *topk_idx,
                     int32_t *topk_cnt, void *stream);

/* Steps (c)+(d) with caller-supplied indices (layout as csa_indexer_topk
 * writes them; every index must lie in [0, vis) and count <= min(vis, K),
 * else CSA_ERR_BAD_INDEX is recorded and the bad entries are skipped).
 * out [B,S,H,V] in the config dtype; lse_out [B,S,H] fp32 natural-log
 * log-sum-exp of the merged streams, may be NULL.  Accuracy of lse_out on the
 * bf16 tensor-core path: the softmax weights are rounded to bf16 (the tensor
 * cores' operand type) before they are summed, so ln(sum) may differ from the
 * exact value by up to -ln(1-u) ~ 3.91e-3 with u = 2^-8 (bf16's unit
 * roundoff); this bound comes from that operand choice, not from the method,
 * and (with fp32 noise, 4e-3) is the tolerance the parity tests apply to
 * lse_out (the fp32 path: 1e-5). */
CSA_API int csa_sparse_attn(csa_handle *h, const csa_batch *b, const int32_t *topk_idx,
                    const int32_t *topk_cnt, void *out, float *lse_out, void *stream);

/* The whole step (a)-(d).  topk_idx_out / topk_cnt_out may be NULL (the
 * handle's workspace holds them); when given they receive what
 * csa_indexer_topk would write. */
CSA_API int csa_decode_step(csa_handle *h, const csa_batch *b, void *out, float *lse_out,
                    int32_t *topk_idx_out, int32_t *topk_cnt_out, void *stream);

/* Step (a) alone, for inspection: scores [B*S, ld] fp32, row j < vis of each
 * query.  score_all = 0 scores only queries with vis > K (as the step does);
 * 1 scores every query.  Entries j >= vis are not written. */
CSA_API int csa_indexer_scores(csa_handle *h, const csa_batch *b, float *scores, int64_t ld,
                       int32_t score_all, void *stream);

/* Step (b) alone on caller scores: for each of nq queries, the K best of
 * scores[q*ld + 0 .. n[q]) (ties to the lower index, -0.0 == +0.0), written
 * like csa_indexer_topk.  n: [nq] int32 device, 0 <= n[q] <= ld, and
 * n[q] <= max_context/ratio.  Uses the handle's K. */
CSA_API int csa_topk_select(csa_handle *h, int32_t nq, const float *scores, int64_t ld,
                    const int32_t *n, int32_t *topk_idx, int32_t *topk_cnt, void *stream);

/* Steps (a)+(b) like csa_indexer_topk, without a handle and without
 * allocating device memory.  The published method has no counterpart of this
 * entry point: it serves callers that may not allocate during a decode step, such
 * as a serving loop whose device memory is planned up front (a library
 * allocation would go around its pool) or whose step must not block (cudaMalloc
 * and cudaFree may synchronise the device).
 *
 * Scratch (a status word, the indexer work list and the fp32 score matrix
 * [B*S, max_context/ratio]) is an 8 MiB array of this library's device
 * module; a batch needing more is rejected with CSA_ERR_WORKSPACE and a
 * message giving the size (csa_indexer_topk has no such limit).  cfg's
 * max_batch / max_queries_per_req bound B and S as for a handle.
 *
 * The first call in each CUDA context (normally one per device, its primary
 * context) looks up the array's address and the SM count and keeps them,
 * keyed by the context's unique id: a context created later on the same
 * device (after cudaDeviceReset, which unloads the module, or a driver-API
 * context made current) gets a lookup of its own.  Make that first call, for
 * example with B = 0, outside stream capture.  Each call clears the status
 * word on `stream` before its kernels run.  The array is shared by every
 * call in the process on that device: calls whose execution overlaps (other
 * streams or host threads) race on it and must be ordered by the caller.
 *
 * topk_idx / topk_cnt as csa_indexer_topk.  status_out: NULL or a device
 * int32 that receives the status word after the kernels (with B = 0, a 0
 * written on `stream`): 0, or an OR of the value 1 (bit 0: a length or row
 * index out of range, what csa_get_status reports as CSA_ERR_BAD_INDEX) and
 * the value 2 (bit 1: a device wait gave up, CSA_ERR_TIMEOUT).
 * Launches on `stream`; does not synchronise. */
CSA_API int csa_indexer_topk_static(const csa_config *cfg, const csa_batch *b, int32_t *topk_idx,
                            int32_t *topk_cnt, int32_t *status_out, void *stream);

/* The cache update that precedes a step: pool row slot[t] receives row t of
 * `rows` for t < n, each row_bytes bytes (any element type: bf16 KV rows,
 * FP8 key rows, fp32 scale rows).  rows_stride / pool_stride are in BYTES
 * (>= row_bytes); rows, slot and pool are device memory.  slot [n] int64:
 * a negative slot is a padding token and is skipped; a slot >= pool_rows is
 * skipped and sets bit 1 in *status (a device int32, may be NULL).  Slots
 * are expected to be collision-free (each pool row written by at most one
 * token, as an allocator hands them out); with a repeated slot the row holds
 * one of the rows written to it.  ("Perf: parallelize the DSpark TP-4 SWA
 * decode hot tasks", PR description: the SWA KV scatter by slot mapping
 * must commit every mapping entry, whatever the row count.)  n = 0 is a
 * no-op.  Returns CSA_ERR_INVALID_ARG for a NULL pointer with n > 0, n < 0,
 * a stride below row_bytes or negative sizes; launches on `stream`, does
 * not synchronise. */
CSA_API int csa_cache_writeback(const void *rows, int64_t rows_stride, const int64_t *slot,
                                int32_t n, void *pool, int64_t pool_stride, int64_t pool_rows,
                                int64_t row_bytes, int32_t *status, void *stream);

/* Host-side checks of a batch against a config, exactly those every entry
 * point runs before launching (null / misaligned pointers, strides, sizes
 * against the maxima, ctx_len_host values).  Touches no device memory and
 * needs no GPU.  Returns CSA_OK or the code the entry point would return. */
CSA_API int csa_check_batch(const csa_config *cfg, const csa_batch *b);

/* Synchronises `stream`, then returns and clears the handle's device status:
 * CSA_OK, CSA_ERR_BAD_INDEX or CSA_ERR_TIMEOUT (or CSA_ERR_CUDA). */
CSA_API int csa_get_status(csa_handle *h, void *stream);

/* Per-stage timing.  While enabled, every kernel launch of the handle is
 * bracketed by CUDA events recorded on its stream (stages, in order: plan,
 * indexer, Top-K, attention).  csa_profile_read waits for the recorded
 * events, writes the summed milliseconds ms[4] and launch counts
 * launches[4] since the last read, and resets them.  Timing adds two event
 * records per launch; leave it off for end-to-end timing. */
CSA_API int csa_profile_enable(csa_handle *h, int32_t enable);
CSA_API int csa_profile_read(csa_handle *h, float *ms, int32_t *launches);

/* Test hook for the device-side timeout path.  Every wait of this library's
 * kernels on another thread's progress (an mbarrier phase) is bounded: after
 * about a second it gives up, the block winds down (copies and tensor-core
 * operations already started are waited for, tensor memory is freed) and the
 * status word records CSA_ERR_TIMEOUT, so a stalled pipeline returns an error
 * instead of hanging the GPU.  With polls >= 0, the consumer waits of the
 * attention tile kernel launched by later calls on this handle give up after
 * `polls` polls (0: at their first wait, whatever the data), which drives that
 * path on purpose; the outputs of such a call are then undefined.  polls < 0
 * restores the default.  Returns CSA_ERR_INVALID_ARG for a NULL handle. */
CSA_API int csa_debug_set_wait_polls(csa_handle *h, int32_t polls);

/* Message for the last error on this host thread ("" if none). */
CSA_API const char *csa_last_error(void);

/* Number of kernel launches the last call on this handle made. */
CSA_API int32_t csa_last_launch_count(const csa_handle *h);

/* CSA_ABI_VERSION of the built library. */
CSA_API int32_t csa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H */
