// nsa_local_virtual_batches / nsa_effective_chunk_size: chunk-local attention
// as independent virtual requests, computed on the host like the page does.
//
// [FA3-diff] make_local_attention_virtual_batches and the effective chunk
// rule in FlashAttentionBackend.init_forward_metadata.  Each request's query
// rows occupy key positions [kv - q, kv); every attention chunk of the key
// axis that those positions touch becomes one virtual request holding the
// queries that fall in it and the keys of that chunk up to the request end.
#include <stdint.h>

#include "../../include/nsa.h"

namespace {

// Python semantics of // and % (the page relies on them for negative divisors).
inline int64_t pydiv(int64_t a, int64_t b)
{
    int64_t q = a / b, r = a % b;
    return (r != 0 && ((r < 0) != (b < 0))) ? q - 1 : q;
}
inline int64_t pymod(int64_t a, int64_t b) { return a - b * pydiv(a, b); }

}  // namespace

extern "C" int nsa_effective_chunk_size(int attn_chunk_size, int max_seq_len, int page_size)
{
    if (attn_chunk_size < 1 || page_size < 1 || max_seq_len < 0) return -1;
    int c = attn_chunk_size < max_seq_len ? attn_chunk_size : max_seq_len;
    c = (c / page_size) * page_size;
    return c < page_size ? page_size : c;
}

extern "C" nsa_status nsa_local_virtual_batches(
    int c, int ps, int B, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
    const int32_t *block_table, int64_t bt_ld, int64_t bt_cols, int max_vb, int *num_vb,
    int32_t *seqlens_q_local, int32_t *cu_seqlens_q_local, int32_t *seqlens_k_local,
    int32_t *k_seqstarts_absolute, int32_t *block_table_local)
{
    if (c < 1 || ps < 1 || c % ps != 0 || B < 0 || !num_vb) return NSA_ERR_INVALID_ARG;
    if (B > 0 && (!cu_seqlens_q || !seq_lens)) return NSA_ERR_INVALID_ARG;
    const bool fill = seqlens_q_local && cu_seqlens_q_local && seqlens_k_local &&
                      k_seqstarts_absolute && block_table_local;
    if (fill && (!block_table || bt_ld < bt_cols)) return NSA_ERR_INVALID_ARG;
    const int ppl = c / ps;
    int64_t vb = 0;
    if (fill) cu_seqlens_q_local[0] = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t q = (int64_t)cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        const int64_t kv = seq_lens[b];
        if (q < 1 || kv < q) return NSA_ERR_INVALID_ARG;
        int64_t q_first = c - pymod(kv - q, c);  // queries in the first (partial) chunk
        if (q_first > q) q_first = q;
        const int64_t last = c + pymod(kv, -(int64_t)c);  // keys in the final chunk
        const int64_t blocks = 1 + (-pydiv(q - q_first, -(int64_t)c));  // 1 + cdiv
        for (int64_t j = 0; j < blocks; ++j, ++vb) {
            if (!fill) continue;
            if (vb >= max_vb) return NSA_ERR_INVALID_ARG;
            int64_t sq = q_first;
            if (j > 0) {
                sq = (q - q_first) - (int64_t)c * (j - 1);
                if (sq > c) sq = c;
            }
            const int64_t start = kv - ((blocks - j - 1) * c + last);
            seqlens_q_local[vb] = (int32_t)sq;
            cu_seqlens_q_local[vb + 1] = cu_seqlens_q_local[vb] + (int32_t)sq;
            seqlens_k_local[vb] = (int32_t)(j == blocks - 1 ? last : c);
            k_seqstarts_absolute[vb] = (int32_t)start;
            const int64_t p0 = pydiv(start, ps);
            if (p0 < 0 || p0 + ppl > bt_cols) return NSA_ERR_INVALID_ARG;
            for (int i = 0; i < ppl; ++i)
                block_table_local[vb * ppl + i] = block_table[(int64_t)b * bt_ld + p0 + i];
        }
    }
    *num_vb = (int)vb;
    return NSA_OK;
}
