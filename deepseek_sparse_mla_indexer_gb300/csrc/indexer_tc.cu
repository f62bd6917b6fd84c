// Tensor-core indexer (placeholder until the tcgen05 kernel lands).
#include "indexer_tc.cuh"

namespace nsa {
nsa_status indexer_tc_try_launch(nsa_dtype, const void *, const float *, const void *, const float *, int64_t,
                                 int, int, int, const int32_t *, int64_t, const int32_t *, const int32_t *, int,
                                 int, float *, int64_t, int32_t *, cudaStream_t)
{
    return NSA_ERR_UNSUPPORTED;
}
}  // namespace nsa
