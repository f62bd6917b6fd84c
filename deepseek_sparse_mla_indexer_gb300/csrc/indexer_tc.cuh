// Tensor-core (tcgen05) indexer kernel entry, used by nsa_indexer_logits.
#pragma once
#include "nsa_internal.cuh"

namespace nsa {
// Launches the tensor-core indexer when the problem fits its shape; returns
// NSA_ERR_UNSUPPORTED (without launching) when it does not.
nsa_status indexer_tc_try_launch(nsa_dtype dtype, const void *q, const float *w, const void *k_cache,
                                 const float *k_scale, int64_t num_pages, int page_size, int Hi, int Di,
                                 const int32_t *rpt, int64_t rpt_ld, const int32_t *row_to_req,
                                 const int32_t *row_len, int R, int max_row_len, float *logits,
                                 int64_t logits_ld, uint32_t *score_hist, int32_t *status, cudaStream_t stream,
                                 int rows_per_group);
}  // namespace nsa
