// nsa_sparse_mla: MLA attention over only the selected KV rows.
//
// [DSA] _forward_flashmla_sparse / _forward_flashmla_kv call contract and
// [NSA] "here, we use page size = 1": every index is a row of the flat KV
// view; keys and values share the latent (V = the first d_latent columns of
// the same row).  Per row r and head h:
//   s_j = sm_scale * q[r,h] . KV[idx_j]     lse = ln sum_j exp(s_j)
//   out = sum_j exp(s_j - lse) * KV[idx_j, 0:d_latent]
//
// This file holds the generic CUDA-core kernel (any dims, f32 / bf16 / e4m3
// rows) with a streaming (online) softmax.  The tensor-core kernel for the
// 576 / 512 shape is in sparse_mla_tc.cu and is chosen when it applies.
#include "nsa_internal.cuh"
#include "sparse_mla_tc.cuh"

namespace nsa {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;      // indices per tile (one per lane in the softmax warps)
constexpr int kMaxAcc = 32;    // accumulator entries per thread: heads_per_block * d_latent <= 8192

template <int QDT>
__device__ __forceinline__ float load_q(const void *p, int64_t i)
{
    if (QDT == NSA_DT_BF16) return bf16_bits_to_float(((const uint16_t *)p)[i]);
    return ((const float *)p)[i];
}

// Element d of KV row `slot` as float.
template <int KDT>
__device__ __forceinline__ float load_kv(const void *kv, int64_t slot, int d, int d_latent, int d_rope)
{
    const int dq = d_latent + d_rope;
    if (KDT == NSA_DT_F32) return ((const float *)kv)[slot * dq + d];
    if (KDT == NSA_DT_BF16) return bf16_bits_to_float(((const uint16_t *)kv)[slot * dq + d]);
    const int nb = d_latent / 128;
    const uint8_t *row = (const uint8_t *)kv + slot * (int64_t)(d_latent + 4 * nb + 2 * d_rope);
    if (d < d_latent) {
        const float sc = *(const float *)(row + d_latent + 4 * (d / 128));
        return e4m3_to_float(row[d]) * sc;
    }
    return bf16_bits_to_float(*(const uint16_t *)(row + d_latent + 4 * nb + 2 * (d - d_latent)));
}

template <int QDT, int KDT>
__global__ void __launch_bounds__(kThreads)
sparse_mla_simt_kernel(const void *q_nope, int64_t nope_ld_r, int64_t nope_ld_h, const void *q_rope,
                       int64_t rope_ld_r, int64_t rope_ld_h, const void *kv, int64_t num_slots,
                       const int32_t *indices, int64_t indices_ld, int H, int HG, int d_latent,
                       int d_rope, int topk, float sm_scale, void *out, float *lse, int32_t *status)
{
    extern __shared__ float smem[];
    const int r = blockIdx.x;
    const int h0 = blockIdx.y * HG;
    const int hg = min(HG, H - h0);
    const int dq = d_latent + d_rope, ld = dq + 1;
    float *qs = smem;                 // [HG][dq+1]
    float *kvs = qs + HG * ld;        // [kTile][dq+1]
    float *S = kvs + kTile * ld;      // [HG][kTile]
    float *alpha = S + HG * kTile;    // [HG]
    float *m_run = alpha + HG;        // [HG]
    float *l_run = m_run + HG;        // [HG]
    int *idx = (int *)(l_run + HG);   // [kTile]

    for (int i = threadIdx.x; i < hg * dq; i += kThreads) {
        const int h = i / dq, d = i % dq;
        qs[h * ld + d] = d < d_latent
                             ? load_q<QDT>(q_nope, r * nope_ld_r + (int64_t)(h0 + h) * nope_ld_h + d)
                             : load_q<QDT>(q_rope, r * rope_ld_r + (int64_t)(h0 + h) * rope_ld_h + d - d_latent);
    }
    for (int h = threadIdx.x; h < HG; h += kThreads) { m_run[h] = -INFINITY; l_run[h] = 0.f; }

    float acc[kMaxAcc];
    const int n_acc = (hg * d_latent + kThreads - 1) / kThreads;
#pragma unroll
    for (int i = 0; i < kMaxAcc; ++i) acc[i] = 0.f;

    const int32_t *irow = indices + (int64_t)r * indices_ld;
    for (int j0 = 0; j0 < topk; j0 += kTile) {
        __syncthreads();
        for (int j = threadIdx.x; j < kTile; j += kThreads) {
            int s = (j0 + j < topk) ? irow[j0 + j] : -1;
            if (s < -1 || s >= num_slots) {
                set_status(status, NSA_ERR_BOUNDS);
                s = -1;
            }
            idx[j] = s;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kTile * dq; i += kThreads) {
            const int j = i / dq, d = i % dq;
            const int s = idx[j];
            kvs[j * ld + d] = s >= 0 ? load_kv<KDT>(kv, s, d, d_latent, d_rope) : 0.f;
        }
        __syncthreads();
        for (int p = threadIdx.x; p < hg * kTile; p += kThreads) {
            const int h = p / kTile, j = p % kTile;
            float dot = 0.f;
            const float *a = qs + h * ld, *bb = kvs + j * ld;
            for (int d = 0; d < dq; ++d) dot = fmaf(a[d], bb[d], dot);
            S[h * kTile + j] = idx[j] >= 0 ? dot * sm_scale : -INFINITY;
        }
        __syncthreads();
        {
            const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
            for (int h = warp; h < hg; h += kThreads / 32) {
                const float s = S[h * kTile + lane];
                float mx = s;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_old = m_run[h];
                const float m_new = fmaxf(m_old, mx);
                float pj = 0.f, a = 1.f;
                if (m_new != -INFINITY) {
                    pj = s == -INFINITY ? 0.f : expf(s - m_new);
                    a = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
                }
                float sum = pj;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                S[h * kTile + lane] = pj;
                __syncwarp();
                if (lane == 0) {
                    alpha[h] = a;
                    m_run[h] = m_new;
                    l_run[h] = l_run[h] * a + sum;
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kMaxAcc; ++i) {
            if (i < n_acc) {
                const int e = threadIdx.x + i * kThreads;
                if (e < hg * d_latent) {
                    const int h = e / d_latent, d = e % d_latent;
                    float v = acc[i] * alpha[h];
                    const float *pr = S + h * kTile;
                    for (int j = 0; j < kTile; ++j) v = fmaf(pr[j], kvs[j * ld + d], v);
                    acc[i] = v;
                }
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kMaxAcc; ++i) {
        if (i < n_acc) {
            const int e = threadIdx.x + i * kThreads;
            if (e < hg * d_latent) {
                const int h = e / d_latent, d = e % d_latent;
                const float l = l_run[h];
                const float v = l > 0.f ? acc[i] / l : 0.f;
                const int64_t o = ((int64_t)r * H + h0 + h) * d_latent + d;
                if (QDT == NSA_DT_BF16)
                    ((__nv_bfloat16 *)out)[o] = __float2bfloat16_rn(v);
                else
                    ((float *)out)[o] = v;
            }
        }
    }
    for (int h = threadIdx.x; h < hg; h += kThreads) {
        const float l = l_run[h];
        lse[(int64_t)r * H + h0 + h] = l > 0.f ? m_run[h] + logf(l) : -INFINITY;
    }
}

template <int QDT, int KDT>
nsa_status launch_simt(const void *q_nope, int64_t nope_ld_r, int64_t nope_ld_h, const void *q_rope,
                       int64_t rope_ld_r, int64_t rope_ld_h, const void *kv, int64_t num_slots,
                       const int32_t *indices, int64_t indices_ld, int R, int H, int d_latent,
                       int d_rope, int topk, float sm_scale, void *out, float *lse, int32_t *status,
                       cudaStream_t stream)
{
    int HG = H < 16 ? H : 16;
    while (HG > 1 && HG * d_latent > kThreads * kMaxAcc) --HG;
    if (HG * d_latent > kThreads * kMaxAcc) return NSA_ERR_UNSUPPORTED;
    const int ld = d_latent + d_rope + 1;
    const size_t smem = sizeof(float) * ((size_t)(HG + kTile) * ld + HG * kTile + 3 * HG) + sizeof(int) * kTile;
    if (smem > 227 * 1024) return NSA_ERR_UNSUPPORTED;
    auto k = sparse_mla_simt_kernel<QDT, KDT>;
    NSA_CUDA_TRY(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    dim3 grid((unsigned)R, (unsigned)ceil_div(H, HG));
    k<<<grid, kThreads, smem, stream>>>(q_nope, nope_ld_r, nope_ld_h, q_rope, rope_ld_r, rope_ld_h, kv,
                                        num_slots, indices, indices_ld, H, HG, d_latent, d_rope, topk,
                                        sm_scale, out, lse, status);
    return launch_status();
}

}  // namespace
}  // namespace nsa

extern "C" size_t nsa_sparse_mla_workspace_bytes(nsa_dtype q_dtype, nsa_dtype kv_dtype, int R, int H,
                                                 int d_latent, int d_rope, int topk)
{
    return nsa::sparse_mla_tc_workspace_bytes(q_dtype, kv_dtype, R, H, d_latent, d_rope, topk);
}

extern "C" nsa_status nsa_sparse_mla_plan(nsa_dtype q_dtype, nsa_dtype kv_dtype, int R, int H, int d_latent,
                                          int d_rope, int topk, int *nsplit, int *launches)
{
    if (!nsplit || !launches) return NSA_ERR_INVALID_ARG;
    if (R < 0 || H < 1 || d_latent < 1 || d_rope < 0 || topk < 1) return NSA_ERR_INVALID_ARG;
    const bool combo_ok = (q_dtype == NSA_DT_F32 && kv_dtype == NSA_DT_F32) ||
                          (q_dtype == NSA_DT_BF16 && (kv_dtype == NSA_DT_BF16 || kv_dtype == NSA_DT_E4M3));
    if (!combo_ok || (kv_dtype == NSA_DT_E4M3 && d_latent % 128 != 0)) return NSA_ERR_UNSUPPORTED;
    *nsplit = 1;
    *launches = R == 0 ? 0 : 1;
    if (R > 0) nsa::sparse_mla_tc_plan(q_dtype, kv_dtype, R, H, d_latent, d_rope, topk, nsplit, launches);
    return NSA_OK;
}

extern "C" nsa_status nsa_sparse_mla(nsa_dtype q_dtype, nsa_dtype kv_dtype, const void *q_nope_dev,
                                     int64_t nope_ld_r, int64_t nope_ld_h, const void *q_rope_dev,
                                     int64_t rope_ld_r, int64_t rope_ld_h, const void *kv_dev,
                                     int64_t num_slots, const int32_t *indices_dev, int64_t indices_ld,
                                     int R, int H, int d_latent, int d_rope, int topk, float sm_scale,
                                     void *out_dev, float *lse_dev, void *workspace_dev,
                                     size_t workspace_bytes, int32_t *status_dev, nsa_stream_t stream)
{
    using namespace nsa;
    if (R < 0 || H < 1 || d_latent < 1 || d_rope < 0 || topk < 1 || num_slots < 0) return NSA_ERR_INVALID_ARG;
    if (indices_ld < topk) return NSA_ERR_INVALID_ARG;
    const bool combo_ok = (q_dtype == NSA_DT_F32 && kv_dtype == NSA_DT_F32) ||
                          (q_dtype == NSA_DT_BF16 && (kv_dtype == NSA_DT_BF16 || kv_dtype == NSA_DT_E4M3));
    if (!combo_ok) return NSA_ERR_UNSUPPORTED;
    if (kv_dtype == NSA_DT_E4M3 && d_latent % 128 != 0) return NSA_ERR_UNSUPPORTED;
    if (R == 0) return NSA_OK;
    if (!q_nope_dev || (d_rope > 0 && !q_rope_dev) || !kv_dev || !indices_dev || !out_dev || !lse_dev)
        return NSA_ERR_INVALID_ARG;
    if ((int64_t)R > 2147483647 || H > 65535) return NSA_ERR_UNSUPPORTED;
    const size_t need = sparse_mla_tc_workspace_bytes(q_dtype, kv_dtype, R, H, d_latent, d_rope, topk);
    if (need > 0 && (workspace_bytes < need || !workspace_dev || ((uintptr_t)workspace_dev & 15)))
        return NSA_ERR_INVALID_ARG;

    const cudaStream_t s = (cudaStream_t)stream;
    nsa_status st = sparse_mla_tc_try_launch(q_dtype, kv_dtype, q_nope_dev, nope_ld_r, nope_ld_h, q_rope_dev,
                                             rope_ld_r, rope_ld_h, kv_dev, num_slots, indices_dev,
                                             indices_ld, R, H, d_latent, d_rope, topk, sm_scale, out_dev,
                                             lse_dev, workspace_dev, status_dev, s);
    if (st != NSA_ERR_UNSUPPORTED) return st;
    if (q_dtype == NSA_DT_F32)
        return launch_simt<NSA_DT_F32, NSA_DT_F32>(q_nope_dev, nope_ld_r, nope_ld_h, q_rope_dev, rope_ld_r,
                                                    rope_ld_h, kv_dev, num_slots, indices_dev, indices_ld, R,
                                                    H, d_latent, d_rope, topk, sm_scale, out_dev, lse_dev,
                                                    status_dev, s);
    if (kv_dtype == NSA_DT_BF16)
        return launch_simt<NSA_DT_BF16, NSA_DT_BF16>(q_nope_dev, nope_ld_r, nope_ld_h, q_rope_dev, rope_ld_r,
                                                      rope_ld_h, kv_dev, num_slots, indices_dev, indices_ld,
                                                      R, H, d_latent, d_rope, topk, sm_scale, out_dev,
                                                      lse_dev, status_dev, s);
    return launch_simt<NSA_DT_BF16, NSA_DT_E4M3>(q_nope_dev, nope_ld_r, nope_ld_h, q_rope_dev, rope_ld_r,
                                                  rope_ld_h, kv_dev, num_slots, indices_dev, indices_ld, R,
                                                  H, d_latent, d_rope, topk, sm_scale, out_dev, lse_dev,
                                                  status_dev, s);
}
