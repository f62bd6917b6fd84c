/*
 * nsa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded C99 statement of what the sparse-attention
 * decode/extend path computes.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load it; the product library never does, and
 * this file shares no code, header, table or constant with the CUDA sources.
 *
 * Sources (web pages, cited by title and the function shown on them):
 *   [NSA-diff]  "sglang 0.5.3rc2 -> 0.5.4 diff: sglang/srt/layers/attention/nsa_backend.py"
 *   [FA3-diff]  "sglang 0.4.4.post3 -> 0.4.5 diff: sglang/srt/layers/attention/flashattention_backend.py"
 *   [NSA]       "sglang/python/sglang/srt/layers/attention/nsa_backend.py"
 *   [DSA]       "sgl-project--sglang/python/sglang/srt/layers/attention/dsa_backend.py"
 *
 * All floating point is carried in double.  Every function is pinned by the
 * tests under tests/test_oracle_*.py against worked examples printed on the
 * pages, closed forms, brute force and library routines.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EARG (-1)
#define ORC_EBOUNDS (-2)

#define ORC_MODE_DECODE 0
#define ORC_MODE_EXTEND 1
#define ORC_MODE_VERIFY 2

#define ORC_DT_F32 0
#define ORC_DT_BF16 1
#define ORC_DT_E4M3 2

/* ------------------------------------------------------------------------ */
/* Number formats, decoded from their bit fields.                           */
/* ------------------------------------------------------------------------ */

/* OCP 8-bit E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 encodes subnormals m * 2^-9; S.1111.111 is NaN; there
 * is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_to_f64(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9); /* m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static double load_elem(const void *base, int64_t i, int dtype)
{
    switch (dtype) {
    case ORC_DT_F32: return (double)((const float *)base)[i];
    case ORC_DT_BF16: return orc_bf16_to_f64(((const uint16_t *)base)[i]);
    default: return orc_e4m3_to_f64(((const uint8_t *)base)[i]);
    }
}

/* Python's floor division and modulo (the pages' numpy code relies on them
 * for negative divisors, e.g. `seq_lens % -attn_chunk_size`). */
static int64_t py_floordiv(int64_t a, int64_t b)
{
    int64_t q = a / b, r = a % b;
    if (r != 0 && ((r < 0) != (b < 0)))
        q -= 1;
    return q;
}
static int64_t py_mod(int64_t a, int64_t b) { return a - b * py_floordiv(a, b); }

/* ------------------------------------------------------------------------ */
/* Stage 0: per-step metadata.                                              */
/* ------------------------------------------------------------------------ */

/*
 * Number of query rows R of a step: decode -> B; target-verify -> B * n_draft;
 * extend -> sum(extend_lens).  [NSA] init_forward_metadata, [NSA-diff]
 * target-verify branch, [DSA] init_forward_metadata.
 */
int64_t orc_num_rows(int mode, int B, const int32_t *extend_lens, int n_draft)
{
    int64_t R = 0;
    if (mode == ORC_MODE_DECODE) return B;
    if (mode == ORC_MODE_VERIFY) return (int64_t)B * n_draft;
    for (int b = 0; b < B; ++b) R += extend_lens[b];
    return R;
}

/*
 * The metadata of one step ([DSA] DeepseekSparseAttnBackend.init_forward_metadata
 * and _cal_indexer_k_start_end; [NSA] NSAMetadata and compute_cu_seqlens;
 * [NSA-diff] the target-verify branch):
 *   cache_seqlens[b]  = seq_lens[b] (+ n_draft in target-verify)
 *   cu_seqlens_k      = [0, cumsum(cache_seqlens)]
 *   cu_seqlens_q      = decode: arange(B+1); verify: arange(B*n+1);
 *                       extend: [0, cumsum(extend_lens)]
 *   seqlens_expanded  = decode: cache_seqlens; otherwise, per request,
 *                       arange(kv - q + 1, kv + 1) with q = extend_lens[b] or n
 *   nsa_cache_seqlens = seqlens_expanded clipped to topk (the field comment
 *                       "clipped to `topk`"; the clipping body is not shown)
 *   nsa_cu_seqlens_k  = [0, cumsum(nsa_cache_seqlens)]
 *   nsa_cu_seqlens_q  = arange(R+1)
 *   row_to_req[r]     = the request of row r (token_to_batch_idx)
 *   page_table_1[b,:] = req_to_token[req_pool_indices[b], 0:W]
 *   real_page_table   = page_table_1[:, ::page_size] // page_size
 *   ks, ke (extend)   = ks: sum of seq_lens of earlier requests,
 *                       ke = ks + seqlens_expanded
 * The page table is kept per request; target-verify rows reach their
 * request's row through row_to_req instead of a repeated copy.
 * Returns R, or ORC_EARG if a length exceeds W or an input is malformed.
 */
int64_t orc_metadata(int mode, int B, int W, int n_draft, int topk, int page_size,
                     const int32_t *seq_lens, const int32_t *extend_lens,
                     const int32_t *req_to_token, int64_t r2t_ld,
                     const int32_t *req_pool_indices,
                     int32_t *cache_seqlens, int32_t *cu_seqlens_k, int32_t *cu_seqlens_q,
                     int32_t *seqlens_expanded, int32_t *nsa_cache_seqlens,
                     int32_t *nsa_cu_seqlens_k, int32_t *nsa_cu_seqlens_q,
                     int32_t *row_to_req, int32_t *page_table_1, int64_t pt_ld,
                     int32_t *real_page_table, int64_t rpt_ld, int32_t *ks, int32_t *ke)
{
    int64_t R = orc_num_rows(mode, B, extend_lens, n_draft);
    int64_t r = 0, k_offset = 0;
    int draft = (mode == ORC_MODE_VERIFY) ? n_draft : 0;
    int npages = (W + page_size - 1) / page_size;
    if (page_size <= 0 || topk <= 0 || W < 0) return ORC_EARG;

    cu_seqlens_k[0] = 0;
    for (int b = 0; b < B; ++b) {
        cache_seqlens[b] = seq_lens[b] + draft;
        if (cache_seqlens[b] > W || cache_seqlens[b] < 0) return ORC_EARG;
        cu_seqlens_k[b + 1] = cu_seqlens_k[b] + cache_seqlens[b];
    }

    if (mode == ORC_MODE_DECODE) {
        for (int b = 0; b <= B; ++b) cu_seqlens_q[b] = b;
    } else if (mode == ORC_MODE_VERIFY) {
        for (int64_t i = 0; i <= R; ++i) cu_seqlens_q[i] = (int32_t)i;
    } else {
        cu_seqlens_q[0] = 0;
        for (int b = 0; b < B; ++b) cu_seqlens_q[b + 1] = cu_seqlens_q[b] + extend_lens[b];
    }

    for (int b = 0; b < B; ++b) {
        int kv = cache_seqlens[b];
        int q = (mode == ORC_MODE_DECODE) ? 1 : (mode == ORC_MODE_VERIFY ? n_draft : extend_lens[b]);
        for (int i = 0; i < q; ++i, ++r) {
            /* arange(kv - q + 1, kv + 1); decode reduces to kv itself */
            seqlens_expanded[r] = kv - q + 1 + i;
            row_to_req[r] = b;
            if (mode == ORC_MODE_EXTEND && ks && ke) {
                ks[r] = (int32_t)k_offset;
                ke[r] = (int32_t)(k_offset + seqlens_expanded[r]);
            }
        }
        k_offset += seq_lens[b];
    }

    nsa_cu_seqlens_k[0] = 0;
    for (int64_t i = 0; i < R; ++i) {
        int L = seqlens_expanded[i];
        nsa_cache_seqlens[i] = L < topk ? L : topk;
        nsa_cu_seqlens_k[i + 1] = nsa_cu_seqlens_k[i] + nsa_cache_seqlens[i];
    }
    for (int64_t i = 0; i <= R; ++i) nsa_cu_seqlens_q[i] = (int32_t)i;

    for (int b = 0; b < B; ++b) {
        const int32_t *src = req_to_token + (int64_t)req_pool_indices[b] * r2t_ld;
        for (int t = 0; t < W; ++t) page_table_1[(int64_t)b * pt_ld + t] = src[t];
        for (int p = 0; p < npages; ++p)
            real_page_table[(int64_t)b * rpt_ld + p] =
                (int32_t)py_floordiv(src[p * page_size], page_size);
    }
    return R;
}

/*
 * Effective local-attention chunk: min(chunk, max_seq_len) rounded down to a
 * multiple of page_size, and at least page_size.  [FA3-diff]
 * FlashAttentionBackend.init_forward_metadata, local-attention set-up.
 */
int orc_effective_chunk_size(int chunk, int max_seq_len, int page_size)
{
    int c = chunk < max_seq_len ? chunk : max_seq_len;
    c = (c / page_size) * page_size;
    if (c < page_size) c = page_size;
    return c;
}

/*
 * make_local_attention_virtual_batches ([FA3-diff], with its worked example):
 * each request's queries are cut at attention-chunk boundaries of the key
 * axis; every piece becomes a "virtual" request that attends only to the keys
 * of its own chunk.  Steps, in the pages' order and names:
 *   q_tokens_in_first_block = min(c - ((kv - q) mod c), q)
 *   tokens_in_last_block    = c + (kv mod -c)                (Python mod)
 *   local_blocks            = 1 + cdiv(q - q_tokens_in_first_block, c)
 *   per virtual batch j of a request (arange j, rarange = blocks - j - 1):
 *     seqlens_q_local  = first block: q_tokens_in_first_block;
 *                        later: min(q - q_first - c*(j-1), c)
 *     seqlens_k_local  = c, except the last block: tokens_in_last_block
 *     k_seqstarts_abs  = kv - (rarange*c + tokens_in_last_block)
 *     block_table_local[j, i] = block_table[b, k_seqstarts_abs // ps + i],
 *                               i < c / ps
 * Returns the number of virtual batches; with null outputs it only counts.
 * ORC_EARG if c is not a multiple of ps or a virtual batch would exceed
 * max_vb.
 */
int orc_local_virtual_batches(int c, int ps, int B, const int32_t *cu_seqlens_q,
                              const int32_t *seq_lens, const int32_t *block_table,
                              int64_t bt_ld, int max_vb, int32_t *seqlens_q_local,
                              int32_t *cu_seqlens_q_local, int32_t *seqlens_k_local,
                              int32_t *k_seqstarts_abs, int32_t *block_table_local)
{
    int vb = 0;
    int ppl;
    if (c <= 0 || ps <= 0 || c % ps != 0) return ORC_EARG;
    ppl = c / ps;
    if (cu_seqlens_q_local) cu_seqlens_q_local[0] = 0;
    for (int b = 0; b < B; ++b) {
        int64_t q = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        int64_t kv = seq_lens[b];
        int64_t q_first = c - py_mod(kv - q, c);
        int64_t last = c + py_mod(kv, -(int64_t)c);
        int64_t blocks;
        if (q_first > q) q_first = q;
        /* cdiv(a, b) = -(a // -b) */
        blocks = 1 + (-py_floordiv(q - q_first, -(int64_t)c));
        for (int64_t j = 0; j < blocks; ++j, ++vb) {
            int64_t rj = blocks - j - 1;
            int64_t sq, sk, start;
            if (!seqlens_q_local) continue;
            if (vb >= max_vb) return ORC_EARG;
            if (j == 0) {
                sq = q_first;
            } else {
                sq = (q - q_first) - (int64_t)c * (j - 1);
                if (sq > c) sq = c;
            }
            sk = (j == blocks - 1) ? last : c;
            start = kv - (rj * c + last);
            seqlens_q_local[vb] = (int32_t)sq;
            cu_seqlens_q_local[vb + 1] = cu_seqlens_q_local[vb] + (int32_t)sq;
            seqlens_k_local[vb] = (int32_t)sk;
            k_seqstarts_abs[vb] = (int32_t)start;
            for (int i = 0; i < ppl; ++i)
                block_table_local[(int64_t)vb * ppl + i] =
                    block_table[(int64_t)b * bt_ld + py_floordiv(start, ps) + i];
        }
    }
    return vb;
}

/* ------------------------------------------------------------------------ */
/* Stage 1: lightning-indexer logits.                                       */
/* ------------------------------------------------------------------------ */

/*
 * One row r of the indexer scores over its first L cached tokens:
 *   k[s]        = k_cache[slot(s)] * k_scale[slot(s)]   (dequantised key)
 *   logits[s]   = sum_h w[h] * max(0, sum_d q[h,d] * k[s][d])
 *   slot(s)     = real_page_table[b, s / ps] * ps + s % ps
 * The sum over heads of weighted ReLU'd dot products is the indexer score the
 * DeepSeek sparse attention pages feed to top-k ([NSA] NSAIndexerMetadata,
 * get_page_table_64 / get_seqlens_int32); the pages only call the kernel, so
 * the formula is the method's stated definition.  Accumulated in double,
 * rounded once to float.  Returns ORC_EBOUNDS on a page id outside the cache.
 */
int orc_indexer_row(int dtype, int Hi, int Di, int ps, int64_t num_pages,
                    const void *q_row, const float *w_row, const void *k_cache,
                    const float *k_scale, const int32_t *rpt_row, int L, float *logits_row)
{
    for (int s = 0; s < L; ++s) {
        int64_t page = rpt_row[s / ps];
        int64_t slot;
        double scale, acc = 0.0;
        if (page < 0 || page >= num_pages) return ORC_EBOUNDS;
        slot = page * ps + s % ps;
        scale = (double)k_scale[slot];
        for (int h = 0; h < Hi; ++h) {
            double dot = 0.0;
            for (int d = 0; d < Di; ++d)
                dot += load_elem(q_row, (int64_t)h * Di + d, dtype) *
                       (load_elem(k_cache, slot * Di + d, dtype) * scale);
            acc += (double)w_row[h] * (dot > 0.0 ? dot : 0.0);
        }
        logits_row[s] = (float)acc;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Stage 2: top-k of the logits, transformed to KV slots.                   */
/* ------------------------------------------------------------------------ */

typedef struct { float v; int32_t s; } orc_cand;

/* Order: larger logit first; NaN below everything; -0 equals +0; equal
 * logits keep the lower token position first. */
static int orc_cand_cmp(const void *pa, const void *pb)
{
    const orc_cand *a = (const orc_cand *)pa, *b = (const orc_cand *)pb;
    int an = isnan(a->v), bn = isnan(b->v);
    if (an != bn) return an ? 1 : -1;
    if (!an && a->v != b->v) return a->v > b->v ? -1 : 1;
    return (a->s > b->s) - (a->s < b->s);
}
static int orc_int_cmp(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/*
 * One row of top-k + transform ([NSA] NSAIndexerMetadata.topk_transform, the
 * fused branch that emits page-table slots instead of positions; [DSA]
 * _pad_topk_indices for the -1 sentinel):
 *   the positions s in [0, L) of the topk largest logits (all of [0, L) when
 *   L <= topk), listed in ascending s, each mapped to page_table_1[b, s],
 *   and the rest of the row filled with -1.
 * Returns the number of valid entries.
 */
int orc_topk_row(const float *logits_row, int L, int topk, const int32_t *pt_row,
                 int32_t *out_row)
{
    int n = 0;
    if (L < 0) L = 0;
    if (L <= topk) {
        for (int s = 0; s < L; ++s) out_row[n++] = pt_row[s];
    } else {
        orc_cand *c = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)L);
        int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)topk);
        for (int s = 0; s < L; ++s) { c[s].v = logits_row[s]; c[s].s = s; }
        qsort(c, (size_t)L, sizeof(orc_cand), orc_cand_cmp);
        for (int i = 0; i < topk; ++i) pos[i] = c[i].s;
        qsort(pos, (size_t)topk, sizeof(int32_t), orc_int_cmp);
        for (int i = 0; i < topk; ++i) out_row[n++] = pt_row[pos[i]];
        free(pos);
        free(c);
    }
    for (int i = n; i < topk; ++i) out_row[i] = -1;
    return n;
}

/* ------------------------------------------------------------------------ */
/* Stage 3: sparse MLA over the selected KV rows.                           */
/* ------------------------------------------------------------------------ */

/* Bytes of one fp8 MLA KV row: d_latent e4m3 codes, one float32 scale per
 * 128 latent elements, then d_rope bfloat16 values. */
int64_t orc_fp8_row_bytes(int d_latent, int d_rope)
{
    return (int64_t)d_latent + 4 * (int64_t)(d_latent / 128) + 2 * (int64_t)d_rope;
}

/* Element d (0 <= d < d_latent + d_rope) of KV row `slot`, exactly. */
static double kv_elem(const void *kv, int kv_dtype, int d_latent, int d_rope, int64_t slot, int d)
{
    int dq = d_latent + d_rope;
    if (kv_dtype == ORC_DT_F32) return (double)((const float *)kv)[slot * dq + d];
    if (kv_dtype == ORC_DT_BF16) return orc_bf16_to_f64(((const uint16_t *)kv)[slot * dq + d]);
    {
        const uint8_t *row = (const uint8_t *)kv + slot * orc_fp8_row_bytes(d_latent, d_rope);
        if (d < d_latent) {
            float sc;
            memcpy(&sc, row + d_latent + 4 * (d / 128), 4);
            return orc_e4m3_to_f64(row[d]) * (double)sc;
        } else {
            uint16_t h;
            memcpy(&h, row + d_latent + 4 * (d_latent / 128) + 2 * (d - d_latent), 2);
            return orc_bf16_to_f64(h);
        }
    }
}

/*
 * One query row of sparse MLA ([DSA] _forward_flashmla_sparse /
 * _forward_flashmla_kv call contract; [NSA] "NOTE(dark): here, we use page
 * size = 1" -- indices are rows of the flat KV view):
 *   K_j = KV[idx_j, 0 : d_latent + d_rope],  V_j = KV[idx_j, 0 : d_latent]
 *   s_j = sm_scale * q_h . K_j  over the valid (non -1) entries j
 *   lse_h = ln sum_j exp(s_j);  out_h = sum_j exp(s_j - lse_h) V_j
 * q is given as its latent ("nope") and rope halves, which concatenate to
 * the 576-wide absorbed query.  No valid entry: out = 0, lse = -inf.
 * Returns ORC_EBOUNDS for an index outside [-1, num_slots).
 */
int orc_sparse_mla_row(int q_dtype, int kv_dtype, int H, int d_latent, int d_rope, int topk,
                       const void *q_nope, int64_t nope_ld_h, const void *q_rope,
                       int64_t rope_ld_h, const void *kv, int64_t num_slots,
                       const int32_t *idx_row, double sm_scale, double *out, double *lse)
{
    int nvalid = 0;
    double *s = (double *)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
    for (int j = 0; j < topk; ++j) {
        if (idx_row[j] == -1) continue;
        if (idx_row[j] < -1 || idx_row[j] >= num_slots) { free(s); return ORC_EBOUNDS; }
    }
    for (int h = 0; h < H; ++h) {
        double m = -INFINITY, sum = 0.0, l;
        for (int j = 0; j < topk; ++j) {
            int64_t slot = idx_row[j];
            double dot = 0.0;
            if (slot < 0) continue;
            for (int d = 0; d < d_latent; ++d)
                dot += load_elem(q_nope, (int64_t)h * nope_ld_h + d, q_dtype) *
                       kv_elem(kv, kv_dtype, d_latent, d_rope, slot, d);
            for (int d = 0; d < d_rope; ++d)
                dot += load_elem(q_rope, (int64_t)h * rope_ld_h + d, q_dtype) *
                       kv_elem(kv, kv_dtype, d_latent, d_rope, slot, d_latent + d);
            s[j] = sm_scale * dot;
            if (s[j] > m) m = s[j];
        }
        for (int d = 0; d < d_latent; ++d) out[(int64_t)h * d_latent + d] = 0.0;
        nvalid = 0;
        for (int j = 0; j < topk; ++j)
            if (idx_row[j] >= 0) { sum += exp(s[j] - m); ++nvalid; }
        if (nvalid == 0) { lse[h] = -INFINITY; continue; }
        l = m + log(sum);
        lse[h] = l;
        for (int j = 0; j < topk; ++j) {
            int64_t slot = idx_row[j];
            double p;
            if (slot < 0) continue;
            p = exp(s[j] - l);
            for (int d = 0; d < d_latent; ++d)
                out[(int64_t)h * d_latent + d] += p * kv_elem(kv, kv_dtype, d_latent, d_rope, slot, d);
        }
    }
    free(s);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* KV-cache write side: the rows the attention reads, written from bf16.    */
/* ------------------------------------------------------------------------ */

/* The pages name the conversions only ([NSA] set_mla_kv_buffer(layer, loc, k,
 * k_rope) and quantize_k_cache(kv_cache), which turns a bf16 cache into the
 * fp8 layout; [DSA] the same plus dequantize_k_cache_paged(kv_cache,
 * page_table_1_flattened)).  The rule written out here: a block of values gets
 * one fp32 scale, its largest magnitude divided by 448 (1 for an all-zero
 * block); each value divided by the scale (fp32) is rounded to the nearest
 * e4m3 value, ties to even mantissa, magnitudes beyond 448 saturating. */

/* x -> e4m3 code (round to nearest, ties to even; saturating; NaN -> 0x7F). */
uint8_t orc_e4m3_encode(float x)
{
    double a = fabs((double)x);
    uint8_t sign = (uint8_t)(signbit(x) ? 0x80 : 0x00);
    if (x != x) return 0x7F;
    if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* largest finite */
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; a mantissa of 8 is the smallest normal */
        double m = nearbyint(a * 512.0); /* exact scaling; ties to even */
        return (uint8_t)(sign | (uint8_t)m);
    }
    {
        int e;
        double fr = frexp(a, &e);           /* a = fr * 2^e, fr in [0.5, 1) */
        double m = nearbyint((fr * 2.0 - 1.0) * 8.0); /* 3 mantissa bits, ties to even */
        int ef = (e - 1) + 7;               /* biased exponent of 2^(e-1) */
        if (m >= 8.0) {
            m = 0.0;
            ef += 1;
        }
        if (ef > 15 || (ef == 15 && m > 6.0)) return (uint8_t)(sign | 0x7E);
        return (uint8_t)(sign | (uint8_t)(ef << 3) | (uint8_t)m);
    }
}

/* fp32 -> bf16 bits, round to nearest even (NaN stays a quiet NaN). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* One block of n bf16 values -> n codes and the block's scale. */
static float quantize_block(const uint16_t *x, int n, uint8_t *codes)
{
    float amax = 0.0f, scale;
    for (int i = 0; i < n; ++i) {
        float v = fabsf(bf16_to_f32(x[i]));
        if (v > amax) amax = v;
    }
    scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int i = 0; i < n; ++i) codes[i] = orc_e4m3_encode(bf16_to_f32(x[i]) / scale);
    return scale;
}

/* One MLA KV row in the fp8 layout: latent codes (d_latent) | one fp32 scale per
 * 128 latent values | rope bf16 (d_rope), from bf16 latent and rope. */
void orc_quantize_mla_row(const uint16_t *latent, const uint16_t *rope, int d_latent, int d_rope, uint8_t *row)
{
    for (int b = 0; b < d_latent / 128; ++b) {
        float sc = quantize_block(latent + 128 * b, 128, row + 128 * b);
        memcpy(row + d_latent + 4 * b, &sc, 4);
    }
    memcpy(row + d_latent + 4 * (d_latent / 128), rope, 2 * (size_t)d_rope);
}

/* One fp8 MLA row back to bf16: code * scale rounded once to fp32 (the exact
 * product of two fp32 values fits a double), then to bf16. */
void orc_dequantize_mla_row(const uint8_t *row, int d_latent, int d_rope, uint16_t *out)
{
    for (int d = 0; d < d_latent; ++d) {
        float sc;
        memcpy(&sc, row + d_latent + 4 * (d / 128), 4);
        out[d] = orc_f32_to_bf16((float)(orc_e4m3_to_f64(row[d]) * (double)sc));
    }
    memcpy(out + d_latent, row + d_latent + 4 * (d_latent / 128), 2 * (size_t)d_rope);
}

/* One indexer key row: D codes and one fp32 scale. */
float orc_quantize_index_row(const uint16_t *k, int D, uint8_t *codes)
{
    return quantize_block(k, D, codes);
}

/* ------------------------------------------------------------------------ */
/* RAGGED extend: the top-k as positions in a request-contiguous KV buffer.  */
/* ------------------------------------------------------------------------ */

/* [DSA] RAGGED topk transform: the selected positions s of the row (the same
 * set and order as orc_topk_row), each shifted by the row's offset (the start
 * of its request in the flattened KV, cu_seqlens_k[b]); -1 stays -1. */
int orc_topk_ragged_row(const float *logits_row, int L, int topk, int32_t offset, int32_t *out_row)
{
    int32_t *ident = (int32_t *)malloc(sizeof(int32_t) * (size_t)(L > 0 ? L : 1));
    int n;
    for (int s = 0; s < L; ++s) ident[s] = s;
    n = orc_topk_row(logits_row, L, topk, ident, out_row);
    for (int i = 0; i < topk; ++i)
        if (out_row[i] != -1) out_row[i] += offset;
    free(ident);
    return n;
}

/* [DSA] page_table_1_flattened: the first kv_len[b] entries of each request's
 * page-table row, requests one after another (request b starts at
 * sum_{b' < b} kv_len[b']). Returns the total length. */
int64_t orc_flatten_page_table(int B, const int32_t *page_table_1, int64_t pt_ld, const int32_t *kv_len,
                               int32_t *out)
{
    int64_t n = 0;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < kv_len[b]; ++t) out[n++] = page_table_1[(int64_t)b * pt_ld + t];
    return n;
}

/* ------------------------------------------------------------------------ */
/* Chunk-local dense attention over the local virtual batches.              */
/* ------------------------------------------------------------------------ */

/*
 * [FA3-diff] FlashAttentionBackend with local attention: for virtual batch
 * b (from make_local_attention_virtual_batches) the queries
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 attend, causally with the queries
 * aligned to the end of the keys, to the first seqused_k[b] keys of the
 * chunk, key j stored in page block_table[b, j / ps] at offset j % ps; query
 * head h reads key/value head h / (Hq / Hkv).  Query i of n_q sees keys
 * j <= seqused_k[b] - n_q + i.  out = softmax(sm_scale q.k) v, lse = ln sum exp;
 * a query that sees no key gets out 0, lse -inf.  One query token, all heads;
 * q [Hq][D], caches [pages][ps][Hkv][D] (bf16 bits), out [Hq][D], lse [Hq].
 */
int orc_local_attention_row(int b, int i, int Hq, int Hkv, int D, int ps, int64_t num_pages,
                            const int32_t *block_table, int64_t bt_ld, const int32_t *cu_seqlens_q,
                            const int32_t *seqused_k, const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, double sm_scale, double *out, double *lse)
{
    int nq = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    int nk = seqused_k[b];
    int last = nk - nq + i; /* last key this query sees */
    int G = Hq / Hkv;
    double *s = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    for (int h = 0; h < Hq; ++h) {
        int hk = h / G;
        double m = -INFINITY, sum = 0.0;
        for (int d = 0; d < D; ++d) out[(int64_t)h * D + d] = 0.0;
        for (int j = 0; j <= last && j < nk; ++j) {
            int32_t page = block_table[(int64_t)b * bt_ld + j / ps];
            const uint16_t *kr;
            double dot = 0.0;
            if (page < 0 || page >= num_pages) { free(s); return ORC_EBOUNDS; }
            kr = k_cache + (((int64_t)page * ps + j % ps) * Hkv + hk) * D;
            for (int d = 0; d < D; ++d) dot += orc_bf16_to_f64(q[(int64_t)h * D + d]) * orc_bf16_to_f64(kr[d]);
            s[j] = sm_scale * dot;
            if (s[j] > m) m = s[j];
        }
        if (last < 0 || nk <= 0) { lse[h] = -INFINITY; continue; }
        for (int j = 0; j <= last && j < nk; ++j) sum += exp(s[j] - m);
        lse[h] = m + log(sum);
        for (int j = 0; j <= last && j < nk; ++j) {
            int32_t page = block_table[(int64_t)b * bt_ld + j / ps];
            const uint16_t *vr = v_cache + (((int64_t)page * ps + j % ps) * Hkv + hk) * D;
            double p = exp(s[j] - lse[h]);
            for (int d = 0; d < D; ++d) out[(int64_t)h * D + d] += p * orc_bf16_to_f64(vr[d]);
        }
    }
    free(s);
    return ORC_OK;
}
