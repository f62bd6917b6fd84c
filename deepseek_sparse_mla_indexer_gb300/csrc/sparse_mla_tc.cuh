// Tensor-core (tcgen05) sparse-MLA kernel entry, used by nsa_sparse_mla.
#pragma once
#include "nsa_internal.cuh"

namespace nsa {
size_t sparse_mla_tc_workspace_bytes(nsa_dtype q_dtype, nsa_dtype kv_dtype, int R, int H, int d_latent,
                                     int d_rope, int topk);
// Split count and kernel launches of the tensor-core path; false when it does not apply.
bool sparse_mla_tc_plan(nsa_dtype q_dtype, nsa_dtype kv_dtype, int R, int H, int d_latent, int d_rope, int topk,
                        int *nsplit, int *launches);
// Launches the tensor-core kernel when the problem fits its shape; returns
// NSA_ERR_UNSUPPORTED (without launching) when it does not.
nsa_status sparse_mla_tc_try_launch(nsa_dtype q_dtype, nsa_dtype kv_dtype, const void *q_nope,
                                    int64_t nope_ld_r, int64_t nope_ld_h, const void *q_rope,
                                    int64_t rope_ld_r, int64_t rope_ld_h, const void *kv, int64_t num_slots,
                                    const int32_t *indices, int64_t indices_ld, int R, int H, int d_latent,
                                    int d_rope, int topk, float sm_scale, void *out, float *lse,
                                    void *workspace, int32_t *status, cudaStream_t stream);
}  // namespace nsa
