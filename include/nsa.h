/*
 * nsa.h -- C ABI of the DeepSeek sparse-attention (NSA / DSA) decode and
 * extend hot path on one GPU:
 *
 *   nsa_metadata        per-step sequence-length and page-table metadata
 *   nsa_local_virtual_batches   chunk-local attention virtual batches (host)
 *   nsa_indexer_logits  lightning-indexer scores  sum_h w * ReLU(q . k)
 *   nsa_topk_transform  per-row top-k of the scores, mapped to KV slots
 *   nsa_sparse_mla      MLA attention over only the selected KV rows
 *
 * Sources, cited by page title and the function shown on the page:
 *   [NSA-diff] "sglang 0.5.3rc2 -> 0.5.4 diff: sglang/srt/layers/attention/nsa_backend.py"
 *   [FA3-diff] "sglang 0.4.4.post3 -> 0.4.5 diff: sglang/srt/layers/attention/flashattention_backend.py"
 *   [NSA]      "sglang/python/sglang/srt/layers/attention/nsa_backend.py"
 *   [DSA]      "sgl-project--sglang/python/sglang/srt/layers/attention/dsa_backend.py"
 *
 * General rules
 *  - Ownership: the caller allocates every buffer.  The library never
 *    allocates device or host memory, keeps no state between calls and holds
 *    no pointer after a call returns.
 *  - Pointers named *_dev (or documented "device") are device pointers; all
 *    work is enqueued asynchronously on `stream` (NULL = the legacy default
 *    stream).  Host pointers are read before the call returns.
 *  - Errors: arguments are validated on the host before any launch; a bad
 *    argument returns NSA_ERR_INVALID_ARG / NSA_ERR_UNSUPPORTED and nothing is
 *    launched.  A failed launch returns NSA_ERR_CUDA.  Problems that only the
 *    device can see (a page id or slot outside the cache, a length beyond the
 *    table) are recorded in the optional device status word `status_dev`
 *    (int32, caller-zeroed; the first error code written wins) and the
 *    offending element is skipped -- kernels never trap.  Read it with
 *    nsa_status_read() when convenient.
 *  - Integers are int32 unless stated; leading dimensions (`*_ld`) count
 *    elements, not bytes.
 *  - -1 is the "no index" sentinel in index rows ([DSA] _pad_topk_indices).
 */
#ifndef NSA_H
#define NSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *nsa_stream_t; /* same type as cudaStream_t */

typedef enum nsa_status {
    NSA_OK = 0,
    NSA_ERR_INVALID_ARG = 1, /* host-detected bad argument; nothing launched */
    NSA_ERR_UNSUPPORTED = 2, /* valid but not supported (dtype / shape combination) */
    NSA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    NSA_ERR_BOUNDS = 4,      /* device-detected index, page id or length out of range */
    NSA_ERR_TIMEOUT = 5      /* a bounded device wait gave up */
} nsa_status;

typedef enum nsa_mode {
    NSA_MODE_DECODE = 0,        /* one query row per request */
    NSA_MODE_EXTEND = 1,        /* extend_lens[b] new query rows per request (chunked prefill) */
    NSA_MODE_TARGET_VERIFY = 2  /* n_draft query rows per request (speculative verify) */
} nsa_mode;

typedef enum nsa_dtype {
    NSA_DT_F32 = 0,
    NSA_DT_BF16 = 1,
    NSA_DT_E4M3 = 2 /* OCP float8 e4m3fn */
} nsa_dtype;

/* Human-readable name of a status code (static storage). */
const char *nsa_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int nsa_abi_version(void);

/* Copy the device status word to *host_value after synchronizing `stream`.
 * Returns NSA_OK if the copy worked, NSA_ERR_CUDA otherwise. */
nsa_status nsa_status_read(const int32_t *status_dev, int32_t *host_value, nsa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* nsa_metadata                                                             */
/* ------------------------------------------------------------------------ */

/* Output arrays of nsa_metadata: device pointers, all caller-allocated.
 * R = number of query rows (decode: B; target-verify: B * n_draft;
 * extend: sum(extend_lens)). */
typedef struct nsa_metadata_out {
    int32_t *cache_seqlens;     /* [B]    seq_lens (+ n_draft in target-verify) */
    int32_t *cu_seqlens_k;      /* [B+1]  [0, cumsum(cache_seqlens)] */
    int32_t *cu_seqlens_q;      /* decode [B+1] arange; extend [B+1] [0, cumsum(extend_lens)];
                                   target-verify [R+1] arange */
    int32_t *seqlens_expanded;  /* [R]    tokens visible to each row (unclipped) */
    int32_t *nsa_cache_seqlens; /* [R]    min(seqlens_expanded, topk) */
    int32_t *nsa_cu_seqlens_k;  /* [R+1]  [0, cumsum(nsa_cache_seqlens)] */
    int32_t *nsa_cu_seqlens_q;  /* [R+1]  arange(R+1) */
    int32_t *row_to_req;        /* [R]    request of each row */
    int32_t *page_table_1;      /* [B, page_table_1_ld]; columns 0..W-1 written.  May be NULL:
                                   then not written (the top-k can read the slots from
                                   req_to_token through req_rows instead) */
    int64_t page_table_1_ld;    /* >= W (ignored when page_table_1 is NULL) */
    int32_t *real_page_table;   /* [B, real_page_table_ld]; columns 0..ceil(W/ps)-1 written */
    int64_t real_page_table_ld; /* >= ceil(W / page_size) */
    int32_t *indexer_ks;        /* [R] extend only (may be NULL): first key of the row's request
                                   in the ragged key space */
    int32_t *indexer_ke;        /* [R] extend only (may be NULL): indexer_ks + seqlens_expanded */
    int32_t *req_rows;          /* [B] (may be NULL): req_pool_indices as this call read them, the
                                   row of req_to_token holding each request's token slots */
} nsa_metadata_out;

/*
 * Per-step metadata of the sparse-attention backend, in one launch.
 * [DSA] DeepseekSparseAttnBackend.init_forward_metadata (decode, target-verify
 * and extend branches) and _cal_indexer_k_start_end; [NSA] NSAMetadata,
 * compute_cu_seqlens; [NSA-diff] the target-verify branch.
 *
 *   mode               decode / extend / target-verify
 *   B                  requests in the step (>= 0)
 *   R                  query rows (must equal the value implied by mode; host-known)
 *   W                  page-table width = max_seqlen_k (host-known, >= every cache_seqlens)
 *   n_draft            draft tokens per request (target-verify; else ignored)
 *   topk               top-k of the indexer (clips nsa_cache_seqlens)
 *   page_size          tokens per KV page (>= 1)
 *   seq_lens_dev       [B] committed tokens per request (extend: including new tokens)
 *   extend_lens_dev    [B] new tokens per request (extend only; else may be NULL)
 *   req_to_token_dev   [pool_rows, req_to_token_ld] token slot of each request position
 *   req_pool_indices_dev [B] row of each request in req_to_token
 *   out                host struct of device output pointers
 *
 * Differences from the pages: the page table is kept per request in every
 * mode (target-verify rows reach it through row_to_req instead of an n-times
 * repeated copy), and row_to_req is always produced.
 * Device errors: a cache length outside [0, W] or a pool index outside
 * [0, pool_rows) sets NSA_ERR_BOUNDS in *status_dev (that request's table
 * row is skipped).
 */
nsa_status nsa_metadata(nsa_mode mode, int B, int R, int W, int n_draft, int topk, int page_size,
                        const int32_t *seq_lens_dev, const int32_t *extend_lens_dev,
                        const int32_t *req_to_token_dev, int64_t req_to_token_ld,
                        int64_t pool_rows, const int32_t *req_pool_indices_dev,
                        const nsa_metadata_out *out, int32_t *status_dev, nsa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* nsa_local_virtual_batches (host)                                         */
/* ------------------------------------------------------------------------ */

/* Effective local-attention chunk: min(chunk, max_seq_len) floored to a
 * multiple of page_size, and at least page_size.  [FA3-diff]
 * FlashAttentionBackend.init_forward_metadata.  Returns -1 on bad input. */
int nsa_effective_chunk_size(int attn_chunk_size, int max_seq_len, int page_size);

/*
 * Chunk-local attention as independent "virtual" requests.
 * [FA3-diff] make_local_attention_virtual_batches: every request's query
 * rows are cut where the key axis crosses a multiple of attn_chunk_size, and
 * each piece attends (causally, bottom-right aligned) to the keys of its own
 * chunk only.
 *
 * All pointers are HOST pointers (the pages build this on the host too).
 *   cu_seqlens_q   [B+1] query start of each request (every request has >= 1 query)
 *   seq_lens       [B]   key length of each request
 *   block_table    [B, block_table_ld] page ids of each request
 *   block_table_cols  valid columns of block_table (bounds check)
 * Outputs (V = number of virtual batches, P = attn_chunk_size / page_size):
 *   seqlens_q_local [V], cu_seqlens_q_local [V+1], seqlens_k_local [V],
 *   k_seqstarts_absolute [V], block_table_local [V, P]
 * With any output pointer NULL the call only counts: *num_virtual_batches = V.
 * Returns NSA_ERR_INVALID_ARG if attn_chunk_size is not a positive multiple of
 * page_size, V exceeds max_virtual_batches, or a block_table read would fall
 * outside block_table_cols.
 */
nsa_status nsa_local_virtual_batches(int attn_chunk_size, int page_size, int B,
                                     const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                     const int32_t *block_table, int64_t block_table_ld,
                                     int64_t block_table_cols, int max_virtual_batches,
                                     int *num_virtual_batches, int32_t *seqlens_q_local,
                                     int32_t *cu_seqlens_q_local, int32_t *seqlens_k_local,
                                     int32_t *k_seqstarts_absolute, int32_t *block_table_local);

/* ------------------------------------------------------------------------ */
/* nsa_indexer_logits                                                       */
/* ------------------------------------------------------------------------ */

/*
 * Lightning-indexer scores over the paged indexer-key cache:
 *   logits[r, s] = k_scale[slot] * sum_h w[r, h] * ReLU(sum_d q[r, h, d] * k[slot, d])
 *   slot        = real_page_table[row_to_req[r], s / page_size] * page_size + s % page_size
 * for 0 <= s < row_len[r].  This is the score the pages hand to top-k
 * ([NSA] NSAIndexerMetadata: get_page_table_64, get_seqlens_int32; [DSA]
 * the paged MQA logits call); with k_scale >= 0 it equals
 * sum_h w * ReLU(q . (k * k_scale)).  Entries at s >= row_len[r] are not written.
 *
 *   dtype              NSA_DT_E4M3 (q and k e4m3) or NSA_DT_F32 (q and k float32)
 *   q_dev              [R, Hi, Di] row-major
 *   weights_dev        [R, Hi] float32
 *   k_cache_dev        [num_pages, page_size, Di] (slot-major rows of Di)
 *   k_scale_dev        [num_pages, page_size] float32, >= 0 (one scale per key row)
 *   real_page_table_dev [*, rpt_ld] page ids per request (from nsa_metadata)
 *   row_to_req_dev     [R], row_len_dev [R] (seqlens_expanded)
 *   rows_per_group     >= 1: up to this many (at most 4) consecutive rows are
 *                      scored together so that rows of one request share each
 *                      K tile: 1 for decode, n_draft for target-verify, 4 for
 *                      extend.  Rows of a group that belong to different
 *                      requests are handled separately, so any value is correct.
 *   max_row_len        host-known upper bound of row_len (sizes the grid)
 *   logits_dev         [R, logits_ld] float32, logits_ld >= max_row_len
 *   score_hist_dev     optional (NULL: none) [R, 2048] uint32, caller-owned: the
 *                      call adds, for every logit it writes, 1 to bin
 *                      key >> 21 of its row, where key is the score's order-
 *                      preserving 32-bit key (the top-k's first 11-bit radix
 *                      digit; see nsa_topk_transform).  Allocate it zeroed once;
 *                      nsa_topk_transform given the same buffer clears every row it
 *                      reads, so the next step starts from zero.  This is the
 *                      indexer-to-top-k fusion of the pages' fused top-k switch
 *                      ([DSA] SGLANG_DSA_FUSE_TOPK / the top-k v2 plan): the top-k
 *                      starts from these counts instead of a pass over the scores.
 * Supported: Hi*Di <= 8192, Di % 16 == 0.  e4m3 with Hi == 64, Di == 128 and
 * page_size % 64 == 0 runs on the tensor cores (tcgen05, fp8); every other
 * shape runs on the CUDA cores.
 * Device errors: a page id outside [0, num_pages) sets NSA_ERR_BOUNDS and the
 * affected logits are written as -inf.  rpt_ld < ceil(max_row_len / page_size)
 * or logits_ld < max_row_len returns NSA_ERR_INVALID_ARG.  Not checked (the
 * arrays from nsa_metadata always satisfy it): row_to_req[r] names a row of
 * real_page_table.
 */
nsa_status nsa_indexer_logits(nsa_dtype dtype, const void *q_dev, const float *weights_dev,
                              const void *k_cache_dev, const float *k_scale_dev, int64_t num_pages,
                              int page_size, int Hi, int Di, const int32_t *real_page_table_dev,
                              int64_t rpt_ld, const int32_t *row_to_req_dev,
                              const int32_t *row_len_dev, int R, int rows_per_group, int max_row_len,
                              float *logits_dev, int64_t logits_ld, uint32_t *score_hist_dev,
                              int32_t *status_dev, nsa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* nsa_topk_transform                                                       */
/* ------------------------------------------------------------------------ */

/*
 * Per-row top-k of the indexer scores, transformed to KV slots
 * ([NSA] NSAIndexerMetadata.topk_transform, fused variant that "returns a
 * transformed page table directly"; [DSA] transform_index_page_table_decode /
 * _prefill with page size 1 and _pad_topk_indices; rows split over several
 * CTAs as in [DSA]'s top-k v2 plan):
 *   row r with L = row_len[r]:
 *     L <= topk : every position 0..L-1
 *     L >  topk : the topk positions with the largest logits; equal logits
 *                 prefer the lower position; -0 equals +0; NaN ranks lowest
 *   the chosen positions are listed in ascending order, each replaced by
 *   page_table_1[row_to_req[r], s], and the row is padded with -1.
 *
 *   logits_dev       [R, logits_ld] float32 (only s < row_len[r] is read)
 *   row_len_dev      [R] (seqlens_expanded), row_to_req_dev [R]
 *   page_table_1_dev [*, pt_ld] token slots per request (from nsa_metadata)
 *   pt_rows_dev      optional (NULL: request b is row b): request b's slots are row
 *                    pt_rows_dev[b] of page_table_1_dev, which may then be req_to_token
 *                    itself with nsa_metadata's req_rows (the same positions map to the
 *                    same slots, with no copied table).  A row outside [0, pt_rows_limit)
 *                    sets NSA_ERR_BOUNDS and that request's rows get -1 slots.
 *   max_row_len      host-known upper bound of row_len (at most 2,097,152)
 *   indices_dev      [R, indices_ld] int32, indices_ld >= topk
 *   score_hist_dev   optional (NULL: none) [R, 2048] uint32 digit counts from
 *                    nsa_indexer_logits (its score_hist_dev).  The counts are a
 *                    hint: a row whose counts disagree with its scores (the
 *                    numbers of keys above and in the chosen digit) is selected
 *                    from the scores directly, so the indices never depend on the
 *                    buffer's contents.  Every row r < R is left zero.  NULL: the
 *                    call counts the digits itself (one more kernel) into ws.
 *   ws, ws_bytes     caller-owned device workspace of at least
 *                    nsa_topk_workspace_bytes(R, max_row_len, score_hist_dev != NULL)
 *                    bytes, 256-byte aligned (0 bytes, and ws may be NULL, when
 *                    every row is selected by one CTA in shared memory:
 *                    max_row_len <= 16384, or <= 40960 with R no larger than the
 *                    device's SM count).  Longer rows go through per-chunk lists in
 *                    ws.  Without score_hist_dev the workspace also holds the call's
 *                    own digit counts, which must be ZERO before the first call;
 *                    every call leaves them zero again.  A workspace serves calls of
 *                    one (R, max_row_len, with/without score_hist) shape; zero it
 *                    again before using it for another.  Calls sharing a workspace
 *                    or a score_hist buffer must not overlap on the GPU.
 * Supported: 1 <= topk <= 4096.
 * Device errors: row_len[r] < 0 or > max_row_len sets NSA_ERR_BOUNDS and that
 * row is written as all -1.  Not checked on the device (nsa_metadata's arrays
 * always satisfy it): row_to_req[r] names a row of page_table_1.
 */
nsa_status nsa_topk_transform(const float *logits_dev, int64_t logits_ld, const int32_t *row_len_dev,
                              const int32_t *row_to_req_dev, const int32_t *page_table_1_dev,
                              int64_t pt_ld, const int32_t *pt_rows_dev, int64_t pt_rows_limit, int R,
                              int topk, int max_row_len, int32_t *indices_dev,
                              int64_t indices_ld, uint32_t *score_hist_dev, void *ws, size_t ws_bytes,
                              int32_t *status_dev, nsa_stream_t stream);

/* Workspace bytes nsa_topk_transform / nsa_topk_transform_ragged need for R rows
 * of at most max_row_len scores; with_score_hist != 0 when the caller passes the
 * indexer's digit counts (the workspace then holds none of its own).  0 for R <= 0. */
size_t nsa_topk_workspace_bytes(int R, int max_row_len, int with_score_hist);

/* Kernel launches one nsa_topk_transform / nsa_topk_transform_ragged call makes
 * for that shape: 0 for R <= 0; 1 when every row fits one CTA's shared memory;
 * otherwise 2 with the indexer's digit counts (per-chunk candidates, then one
 * assembly per row) or 3 without them (the call counts the digits first). */
int nsa_topk_launches(int R, int max_row_len, int with_score_hist);

/* ------------------------------------------------------------------------ */
/* nsa_sparse_mla                                                           */
/* ------------------------------------------------------------------------ */

/*
 * Sparse MLA attention over only the selected KV rows ([DSA]
 * _forward_flashmla_sparse / _forward_flashmla_kv call contract; [NSA]
 * "here, we use page size = 1": indices are rows of the flat KV view).
 * Keys and values share the latent: K_j = KV[idx_j, 0:d_latent+d_rope],
 * V_j = KV[idx_j, 0:d_latent].  For each row r and head h:
 *   s_j      = sm_scale * (q_nope[r,h] . K_j[0:d_latent] + q_rope[r,h] . K_j[d_latent:])
 *   lse[r,h] = ln sum_j exp(s_j)        (natural log; -inf if no valid index)
 *   out[r,h] = sum_j exp(s_j - lse) V_j (0 if no valid index)
 * over the valid entries j of indices[r, 0:topk] (-1 entries are skipped).
 *
 *   q_dtype           NSA_DT_BF16 or NSA_DT_F32; `out` has the same dtype
 *   kv_dtype          NSA_DT_BF16 rows of d_latent+d_rope bf16,
 *                     NSA_DT_F32 rows of d_latent+d_rope float32, or
 *                     NSA_DT_E4M3 rows of d_latent e4m3 codes, then one float32
 *                     scale per 128 latent elements, then d_rope bf16
 *                     (656 bytes for 512 + 64); requires d_latent % 128 == 0
 *   q_nope_dev        element (r, h, d) at r*nope_ld_r + h*nope_ld_h + d
 *   q_rope_dev        element (r, h, d) at r*rope_ld_r + rope_ld_h*h + d
 *   kv_dev            [num_slots, row] as above
 *   indices_dev       [R, indices_ld] int32 slots or -1
 *   out_dev           [R, H, d_latent] contiguous, dtype = q_dtype
 *   lse_dev           [R, H] float32
 *                     (out and lse are only written, once each: they may also be
 *                     pinned host memory mapped into the device's address space,
 *                     which then receives the result without a separate copy)
 *   workspace_dev     scratch of nsa_sparse_mla_workspace_bytes(...) bytes
 *                     (16-byte aligned; may be NULL if that size is 0)
 * q_dtype F32 requires kv_dtype F32; BF16 q takes BF16 or E4M3 KV.
 * Device errors: an index outside [-1, num_slots) sets NSA_ERR_BOUNDS and is
 * treated as -1.
 */
nsa_status nsa_sparse_mla(nsa_dtype q_dtype, nsa_dtype kv_dtype, const void *q_nope_dev,
                          int64_t nope_ld_r, int64_t nope_ld_h, const void *q_rope_dev,
                          int64_t rope_ld_r, int64_t rope_ld_h, const void *kv_dev,
                          int64_t num_slots, const int32_t *indices_dev, int64_t indices_ld, int R,
                          int H, int d_latent, int d_rope, int topk, float sm_scale, void *out_dev,
                          float *lse_dev, void *workspace_dev, size_t workspace_bytes,
                          int32_t *status_dev, nsa_stream_t stream);

/* Scratch bytes nsa_sparse_mla needs for this problem (0 if none). */
size_t nsa_sparse_mla_workspace_bytes(nsa_dtype q_dtype, nsa_dtype kv_dtype, int R, int H,
                                      int d_latent, int d_rope, int topk);

/*
 * How nsa_sparse_mla runs a problem of this shape (a runtime aid; the pages
 * have no counterpart): *nsplit receives the number of parts each top-k list
 * is split into (1 = none), *launches the number of kernel launches one call
 * makes (0 when R = 0).  Assumes the tensor-core path's alignment (q and KV
 * 16-byte aligned, q strides multiples of 8 elements); calls without it run
 * one CUDA-core launch.  Returns NSA_ERR_INVALID_ARG for NULL outputs or a
 * shape nsa_sparse_mla rejects with that code, NSA_ERR_UNSUPPORTED for a
 * dtype combination it does not support.
 */
nsa_status nsa_sparse_mla_plan(nsa_dtype q_dtype, nsa_dtype kv_dtype, int R, int H, int d_latent,
                               int d_rope, int topk, int *nsplit, int *launches);

/*
 * Self-test of the library's bounded device waits (a test aid; the pages have
 * no counterpart): one block waits for `budget_cycles` SM clocks on an
 * mbarrier that nothing arrives on, gives up and writes NSA_ERR_TIMEOUT into
 * the caller-zeroed status word, the way every tensor-core kernel here reports
 * a wait that ran out instead of hanging.  budget_cycles in [1, 4e9].
 */
nsa_status nsa_check_bounded_wait(int32_t *status_dev, long long budget_cycles, nsa_stream_t stream);

/*
 * Up to 16 copies in one kernel launch (a runtime aid; the pages have no
 * counterpart): bytes[i] bytes from src[i] to dst[i], asynchronously on
 * `stream`.  The pointer arrays are read on the host during the call; the
 * buffers may be device memory or pinned host memory that the device can
 * address (cudaHostAlloc / a pinned torch tensor), so a step's host inputs and
 * outputs can move without one memcpy per buffer.  Buffers must not overlap.
 * Returns NSA_ERR_INVALID_ARG for n outside [0, 16] or a NULL pointer with a
 * non-zero size.
 */
nsa_status nsa_copy_buffers(int n, const void *const *src, void *const *dst, const int64_t *bytes,
                            nsa_stream_t stream);

/* ------------------------------------------------------------------------
 * RAGGED extend ([DSA] TopkTransformMethod.RAGGED): the KV of each request is
 * laid out contiguously (request b from offset cu_seqlens_k[b]), gathered by
 * nsa_dequantize_kv_paged through page_table_1_flattened, and the top-k
 * indices are token positions shifted by the row's request offset
 * (topk_indices_offset = repeat_interleave(cu_seqlens_k[:-1], extend_lens)).
 * ------------------------------------------------------------------------ */

/* As nsa_topk_transform (same workspace), but row r's selected positions s become
 * s + req_offset_dev[row_to_req[r]] instead of page-table slots (-1 padding
 * kept).  req_offset_dev is typically the metadata's cu_seqlens_k; the sums
 * must fit int32. */
nsa_status nsa_topk_transform_ragged(const float *logits_dev, int64_t logits_ld, const int32_t *row_len_dev,
                                     const int32_t *row_to_req_dev, const int32_t *req_offset_dev, int R,
                                     int topk, int max_row_len, int32_t *indices_dev, int64_t indices_ld,
                                     uint32_t *score_hist_dev, void *ws, size_t ws_bytes, int32_t *status_dev,
                                     nsa_stream_t stream);

/* page_table_1_flattened: out_dev[kv_start_dev[b] + t] = page_table_1_dev[b *
 * pt_ld + t] for t < kv_len_dev[b] (typically cache_seqlens and cu_seqlens_k of
 * the metadata).  A request whose range leaves [0, out_len) or whose length
 * exceeds pt_ld sets NSA_ERR_BOUNDS and is skipped. */
nsa_status nsa_flatten_page_table(int B, const int32_t *page_table_1_dev, int64_t pt_ld,
                                  const int32_t *kv_len_dev, const int32_t *kv_start_dev, int32_t *out_dev,
                                  int64_t out_len, int32_t *status_dev, nsa_stream_t stream);

/* ------------------------------------------------------------------------
 * KV-cache write side: the rows the attention and the indexer read.
 *
 * [NSA] / [DSA] set_mla_kv_buffer(layer, loc, k, k_rope) stores the new tokens'
 * latent (k, 512 values) and rope (k_rope, 64 values) parts at their KV slots;
 * quantize_k_cache turns a bf16 cache into the fp8 row layout; [DSA]
 * dequantize_k_cache_paged gathers fp8 rows back to bf16 through the flattened
 * page table.  The pages only name these conversions; the rule used for a
 * block of values: scale = (largest magnitude) / 448 in fp32 (1 for an
 * all-zero block), code = e4m3(value / scale) rounded to nearest, ties to even,
 * saturating at +-448.  fp8 row (656 bytes): 512 e4m3 latent codes | 4 fp32
 * scales (one per 128 latent values) | 64 bf16 rope values.  bf16 row: 576
 * bf16 values (1152 bytes).  Dequantised value: code x scale rounded to fp32,
 * then to bf16 (nearest even).
 *
 * All calls are asynchronous on `stream`, allocate nothing, and return
 * NSA_ERR_UNSUPPORTED for other dims (d_latent 512, d_rope 64, Di 128 only)
 * and NSA_ERR_INVALID_ARG for NULL or misaligned buffers (16-byte aligned KV
 * caches and rope rows, 8-byte aligned bf16 rows) before any launch.
 * A slot outside [0, num_slots) sets NSA_ERR_BOUNDS in the optional status word
 * and its row is skipped (written as zeros by the dequantiser; a negative slot
 * there is padding and gives a zero row without error).
 * ------------------------------------------------------------------------ */

/* New tokens into the MLA KV cache: row i (k_nope_dev + i * nope_ld, k_rope_dev +
 * i * rope_ld, both bf16) goes to slot loc_dev[i] of kv_dev, a [num_slots] array
 * of fp8 rows (kv_dtype NSA_DT_E4M3) or bf16 rows (NSA_DT_BF16).  Slots of one
 * call must be distinct. */
nsa_status nsa_set_mla_kv(nsa_dtype kv_dtype, const void *k_nope_dev, int64_t nope_ld,
                          const void *k_rope_dev, int64_t rope_ld, const int32_t *loc_dev, int n,
                          int d_latent, int d_rope, void *kv_dev, int64_t num_slots,
                          int32_t *status_dev, nsa_stream_t stream);

/* The whole bf16 cache [num_slots][576] to fp8 rows [num_slots][656]. */
nsa_status nsa_quantize_kv_cache(const void *kv_bf16_dev, int64_t num_slots, int d_latent, int d_rope,
                                 void *kv_fp8_dev, nsa_stream_t stream);

/* out_bf16_dev[i] = dequantised fp8 row slots_dev[i] of kv_fp8_dev, i < m
 * (bf16 rows of 576). */
nsa_status nsa_dequantize_kv_paged(const void *kv_fp8_dev, int64_t num_slots, int d_latent, int d_rope,
                                   const int32_t *slots_dev, int64_t m, void *out_bf16_dev,
                                   int32_t *status_dev, nsa_stream_t stream);

/* Indexer keys of new tokens: row i of k_dev (bf16, Di = 128 values, row stride
 * k_ld) -> e4m3 codes at k_cache_dev[loc_dev[i] * 128 ..] and one fp32 scale at
 * k_scale_dev[loc_dev[i]] (the [pages][page_size] arrays nsa_indexer_logits reads,
 * indexed by slot = page * page_size + offset). */
nsa_status nsa_set_index_k(const void *k_dev, int64_t k_ld, const int32_t *loc_dev, int n, int Di,
                           void *k_cache_dev, float *k_scale_dev, int64_t num_slots, int32_t *status_dev,
                           nsa_stream_t stream);

/*
 * nsa_sparse_mla without a caller workspace, for callers that cannot allocate
 * device memory when they call in -- for example a plug-in inside a host
 * framework that owns all device memory and gives the plug-in no allocator,
 * or a serving loop that allows no allocation after start-up so that its
 * memory footprint stays fixed.  The pages have no counterpart: they always
 * run with framework-allocated buffers.
 *
 * Same arguments, semantics and results as nsa_sparse_mla, minus the
 * workspace.  The split-KV scratch is one fixed 32 MiB device array inside
 * this library (every GPU that loads the library holds it until the process
 * exits); this call allocates nothing.  The first call on a device looks up
 * that array's device address (cudaGetSymbolAddress) and caches it, so make
 * the first call on each device before any stream capture.  All calls share
 * the array: calls that may overlap on the GPU (other streams, other host
 * threads) race on it and must be serialised by the caller.  Nothing in the
 * array needs to start at zero.
 * Returns NSA_ERR_UNSUPPORTED when nsa_sparse_mla_workspace_bytes() for the
 * problem exceeds 32 MiB (use nsa_sparse_mla with a workspace instead);
 * otherwise the same status codes as nsa_sparse_mla.
 */
nsa_status nsa_sparse_mla_noalloc(nsa_dtype q_dtype, nsa_dtype kv_dtype, const void *q_nope_dev,
                                  int64_t nope_ld_r, int64_t nope_ld_h, const void *q_rope_dev,
                                  int64_t rope_ld_r, int64_t rope_ld_h, const void *kv_dev,
                                  int64_t num_slots, const int32_t *indices_dev, int64_t indices_ld,
                                  int R, int H, int d_latent, int d_rope, int topk, float sm_scale,
                                  void *out_dev, float *lse_dev, int32_t *status_dev,
                                  nsa_stream_t stream);

/* ------------------------------------------------------------------------
 * nsa_local_attention: dense attention inside attention chunks
 * ------------------------------------------------------------------------ */

/*
 * Chunk-local attention over the virtual batches that
 * nsa_local_virtual_batches builds.  [FA3-diff] FlashAttentionBackend, local
 * attention: the attention call over local_query_start_loc, local_seqused_k
 * and local_block_table, causal.  Virtual batch b holds the query rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and the first seqused_k[b] keys of
 * its chunk; the queries are the last n_q positions of those keys, so query i
 * (of n_q) sees keys 0 .. seqused_k[b] - n_q + i.  Query head h reads key/value
 * head h / (Hq / Hkv).  For each query row t and head h:
 *   out[t, h, :] = sum_j p_j v_j,  p = softmax_j(sm_scale * q[t, h] . k_j)
 *   lse[t, h]    = ln sum_j exp(sm_scale * q[t, h] . k_j)   (natural log)
 * over the visible keys j; a row that sees no key gets out 0 and lse -inf.
 *
 *   q_dev            [total_q, q_ld] bf16; head h of row t at t*q_ld + h*D
 *                    (q_ld >= Hq*D, even; 4-byte aligned)
 *   k_cache_dev, v_cache_dev  [num_pages, page_size, Hkv, D] bf16, 16-byte aligned
 *   block_table_dev  [nvb, bt_ld] int32 page ids (the local block table); bt_ld is
 *                    the row stride and also the row's capacity: a row holds
 *                    page ids for bt_ld * page_size keys
 *   cu_seqlens_q_dev [nvb + 1], seqused_k_dev [nvb]  int32
 *   out_dev          [total_q, Hq, D] bf16 (written), lse_dev [total_q, Hq] float32
 *                    (only written, once each: they may be pinned host memory mapped
 *                    into the device's address space, which then receives the result
 *                    without a separate copy)
 * D is 64 or 128 and Hq / Hkv at most 16 (else NSA_ERR_UNSUPPORTED).  Asynchronous
 * on `stream`; allocates nothing.  Returns NSA_ERR_INVALID_ARG for NULL or
 * misaligned buffers, Hq not a multiple of Hkv, num_pages < 1 or a bad size,
 * before any launch.  Device errors (NSA_ERR_BOUNDS in the optional status
 * word; the result is then invalid): a page id outside [0, num_pages) (slot 0
 * is read instead), and a virtual batch whose seqused_k is negative or above
 * bt_ld * page_size or whose query range does not hold a row it is asked for
 * (cu_seqlens_q must be non-decreasing with cu_seqlens_q[nvb] == total_q); such
 * a batch is treated as having no keys.
 */
nsa_status nsa_local_attention(const void *q_dev, int64_t q_ld, const void *k_cache_dev,
                               const void *v_cache_dev, int64_t num_pages, int page_size,
                               const int32_t *block_table_dev, int64_t bt_ld,
                               const int32_t *cu_seqlens_q_dev, const int32_t *seqused_k_dev, int nvb,
                               int total_q, int Hq, int Hkv, int D, float sm_scale, void *out_dev,
                               float *lse_dev, int32_t *status_dev, nsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NSA_H */
