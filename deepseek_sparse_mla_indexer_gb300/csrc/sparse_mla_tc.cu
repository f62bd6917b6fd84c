// Tensor-core sparse MLA (placeholder until the tcgen05 kernel lands).
#include "sparse_mla_tc.cuh"

namespace nsa {
size_t sparse_mla_tc_workspace_bytes(nsa_dtype, nsa_dtype, int, int, int, int, int) { return 0; }
nsa_status sparse_mla_tc_try_launch(nsa_dtype, nsa_dtype, const void *, int64_t, int64_t, const void *, int64_t,
                                    int64_t, const void *, int64_t, const int32_t *, int64_t, int, int, int, int,
                                    int, float, void *, float *, void *, int32_t *, cudaStream_t)
{
    return NSA_ERR_UNSUPPORTED;
}
}  // namespace nsa
