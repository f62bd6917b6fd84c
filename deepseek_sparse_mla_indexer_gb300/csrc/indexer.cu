// nsa_indexer_logits: lightning-indexer scores over the paged key cache.
//   logits[r, s] = k_scale[slot] * sum_h w[r,h] * ReLU(q[r,h,:] . k[slot,:])
// The score the DeepSeek sparse-attention pages feed to top-k ([NSA]
// NSAIndexerMetadata: get_page_table_64 / get_seqlens_int32; [DSA] the paged
// MQA logits call).
//
// This file holds the generic CUDA-core kernel (any head count / dim, e4m3 or
// float32).  The tensor-core kernel for the 64 x 128 e4m3 shape lives in
// indexer_tc.cu and is chosen by nsa_indexer_logits when it applies.
#include "nsa_internal.cuh"
#include "indexer_tc.cuh"

namespace nsa {
namespace {

constexpr int kTok = 64;       // tokens per block
constexpr int kThreads = 256;  // 4 threads per token, heads split among them
constexpr int kMaxQ = 8192;    // Hi * Di limit

template <int DT>
__device__ __forceinline__ float load_idx(const void *p, int64_t i)
{
    if (DT == NSA_DT_E4M3) return e4m3_to_float(((const uint8_t *)p)[i]);
    return ((const float *)p)[i];
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
indexer_simt_kernel(const void *q, const float *w, const void *k_cache, const float *k_scale,
                    int64_t num_pages, int ps, int Hi, int Di, const int32_t *rpt, int64_t rpt_ld,
                    const int32_t *row_to_req, const int32_t *row_len, int max_row_len, float *logits,
                    int64_t logits_ld, uint32_t *score_hist, int32_t *status)
{
    extern __shared__ float smem[];
    const int r = blockIdx.y;
    int L = row_len[r];
    if (L > max_row_len) {  // caller's bound is wrong: score only what the buffers hold
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, NSA_ERR_BOUNDS);
        L = max_row_len;
    }
    const int s0 = blockIdx.x * kTok;
    if (s0 >= L) return;
    const int ldq = Di + 1;  // padded rows: heads read the same d without bank conflicts
    float *qs = smem;                  // [Hi][Di+1]
    float *ks = qs + Hi * ldq;         // [kTok][Di+1]
    float *ws = ks + kTok * ldq;       // [Hi]
    float *sc = ws + Hi;               // [kTok] scale, or NaN for a bad page
    const int b = row_to_req[r];

    for (int i = threadIdx.x; i < Hi * Di; i += kThreads)
        qs[(i / Di) * ldq + i % Di] = load_idx<DT>(q, (int64_t)r * Hi * Di + i);
    for (int i = threadIdx.x; i < Hi; i += kThreads) ws[i] = w[(int64_t)r * Hi + i];
    for (int t = threadIdx.x; t < kTok; t += kThreads) {
        const int s = s0 + t;
        float v = 0.f;
        if (s < L) {
            const int64_t page = rpt[(int64_t)b * rpt_ld + s / ps];
            if (page < 0 || page >= num_pages) {
                set_status(status, NSA_ERR_BOUNDS);
                v = __int_as_float(0x7fc00000);
            } else {
                v = k_scale[page * ps + s % ps];
            }
        }
        sc[t] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTok * Di; i += kThreads) {
        const int t = i / Di, d = i % Di, s = s0 + t;
        float v = 0.f;
        if (s < L && !isnan(sc[t])) {
            const int64_t page = rpt[(int64_t)b * rpt_ld + s / ps];
            v = load_idx<DT>(k_cache, (page * ps + s % ps) * Di + d);
        }
        ks[t * ldq + d] = v;
    }
    __syncthreads();

    const int t = threadIdx.x >> 2, part = threadIdx.x & 3;
    float acc = 0.f;
    const float *kr = ks + t * ldq;
    for (int h = part; h < Hi; h += 4) {
        const float *qr = qs + h * ldq;
        float dot = 0.f;
        for (int d = 0; d < Di; ++d) dot = fmaf(qr[d], kr[d], dot);
        acc = fmaf(ws[h], fmaxf(dot, 0.f), acc);
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    const int s = s0 + t;
    if (part == 0 && s < L) {
        const float scale = sc[t];
        const float v = isnan(scale) ? -INFINITY : acc * scale;
        logits[(int64_t)r * logits_ld + s] = v;
        if (score_hist) atomicAdd(&score_hist[(int64_t)r * kScoreBins + (order_key(v) >> kScoreDigitShift)], 1u);
    }
}

}  // namespace
}  // namespace nsa

extern "C" nsa_status nsa_indexer_logits(nsa_dtype dtype, const void *q_dev, const float *weights_dev,
                                         const void *k_cache_dev, const float *k_scale_dev,
                                         int64_t num_pages, int page_size, int Hi, int Di,
                                         const int32_t *real_page_table_dev, int64_t rpt_ld,
                                         const int32_t *row_to_req_dev, const int32_t *row_len_dev,
                                         int R, int rows_per_group, int max_row_len, float *logits_dev,
                                         int64_t logits_ld, uint32_t *score_hist_dev, int32_t *status_dev,
                                         nsa_stream_t stream)
{
    using namespace nsa;
    if (dtype != NSA_DT_E4M3 && dtype != NSA_DT_F32) return NSA_ERR_UNSUPPORTED;
    if (R < 0 || Hi < 1 || Di < 1 || page_size < 1 || num_pages < 0 || max_row_len < 0 || rows_per_group < 1)
        return NSA_ERR_INVALID_ARG;
    if (Hi * Di > kMaxQ || Di % 16 != 0) return NSA_ERR_UNSUPPORTED;
    if (logits_ld < max_row_len || rpt_ld < ceil_div(max_row_len, page_size)) return NSA_ERR_INVALID_ARG;
    if (R == 0 || max_row_len == 0) return NSA_OK;
    if (!q_dev || !weights_dev || !k_cache_dev || !k_scale_dev || !real_page_table_dev ||
        !row_to_req_dev || !row_len_dev || !logits_dev)
        return NSA_ERR_INVALID_ARG;
    if ((int64_t)R > 65535) return NSA_ERR_UNSUPPORTED;

    nsa_status st = indexer_tc_try_launch(dtype, q_dev, weights_dev, k_cache_dev, k_scale_dev,
                                          num_pages, page_size, Hi, Di, real_page_table_dev, rpt_ld,
                                          row_to_req_dev, row_len_dev, R, max_row_len, logits_dev,
                                          logits_ld, score_hist_dev, status_dev, (cudaStream_t)stream,
                                          rows_per_group);
    if (st != NSA_ERR_UNSUPPORTED) return st;

    const size_t smem = sizeof(float) * ((size_t)(Hi + kTok) * (Di + 1) + Hi + kTok);
    dim3 grid((unsigned)ceil_div(max_row_len, kTok), (unsigned)R);
    if (dtype == NSA_DT_E4M3) {
        auto k = indexer_simt_kernel<NSA_DT_E4M3>;
        NSA_CUDA_TRY(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        k<<<grid, kThreads, smem, (cudaStream_t)stream>>>(q_dev, weights_dev, k_cache_dev, k_scale_dev,
                                                          num_pages, page_size, Hi, Di, real_page_table_dev,
                                                          rpt_ld, row_to_req_dev, row_len_dev, max_row_len,
                                                          logits_dev, logits_ld, score_hist_dev, status_dev);
    } else {
        auto k = indexer_simt_kernel<NSA_DT_F32>;
        NSA_CUDA_TRY(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        k<<<grid, kThreads, smem, (cudaStream_t)stream>>>(q_dev, weights_dev, k_cache_dev, k_scale_dev,
                                                          num_pages, page_size, Hi, Di, real_page_table_dev,
                                                          rpt_ld, row_to_req_dev, row_len_dev, max_row_len,
                                                          logits_dev, logits_ld, score_hist_dev, status_dev);
    }
    return launch_status();
}
