// nsa_topk_transform: per-row top-k of the indexer scores, mapped to KV slots.
//
// [NSA] NSAIndexerMetadata.topk_transform (the fused variant that "returns a
// transformed page table directly"), [DSA] transform_index_page_table_* with
// page size 1 and _pad_topk_indices (-1 padding).
//
// One block per row.  Scores are mapped to order-preserving 32-bit keys
// (-0 folded onto +0, NaN below every number) and the exact k-th largest key
// T is found by a most-significant-digit radix select (4 passes of 8 bits,
// warp-aggregated shared-memory histograms).  A final ordered pass keeps
// every key > T and the first (k - #{key > T}) keys == T in position order,
// so ties go to the lower position and the output comes out sorted by
// position without a sort.  Rows up to kCacheCap scores are read from HBM
// once and kept in shared memory for the remaining passes.
#include "nsa_internal.cuh"

namespace nsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kCacheCap = 48 * 1024;  // scores cached in shared memory (192 KB)

__device__ __forceinline__ uint32_t order_key(float x)
{
    uint32_t u = __float_as_uint(x);
    if (x != x) return 0u;            // NaN ranks lowest
    if ((u << 1) == 0u) u = 0u;       // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block scan of one int per thread; returns the exclusive prefix and
// writes the block total to *total (all threads see it after the call).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_buf, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_buf[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = warp_buf[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_buf[lane] = w;
        if (lane == 31) *total = w;
    }
    __syncthreads();
    uint32_t excl = x - v + (warp > 0 ? warp_buf[warp - 1] : 0u);
    __syncthreads();
    return excl;
}

__global__ void __launch_bounds__(kThreads)
topk_transform_kernel(const float *logits, int64_t logits_ld, const int32_t *row_len,
                      const int32_t *row_to_req, const int32_t *pt, int64_t pt_ld, int topk,
                      int max_row_len, int cache_cap, int32_t *indices, int64_t indices_ld,
                      int32_t *status)
{
    extern __shared__ uint32_t cache[];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t warp_buf[32];
    __shared__ uint32_t chunk_total;
    __shared__ uint32_t sel_digit, sel_remaining;

    const int r = blockIdx.x;
    const int L = row_len[r];
    const int b = row_to_req[r];
    int32_t *out = indices + (int64_t)r * indices_ld;
    const int32_t *ptr = pt + (int64_t)b * pt_ld;
    const float *lg = logits + (int64_t)r * logits_ld;

    if (L < 0 || L > max_row_len) {
        if (threadIdx.x == 0) set_status(status, NSA_ERR_BOUNDS);
        for (int i = threadIdx.x; i < topk; i += kThreads) out[i] = -1;
        return;
    }
    if (L <= topk) {
        for (int i = threadIdx.x; i < topk; i += kThreads) out[i] = i < L ? ptr[i] : -1;
        return;
    }

    const bool cached = L <= cache_cap;
    if (cached) {
        for (int i = threadIdx.x; i < L; i += kThreads) cache[i] = order_key(lg[i]);
    }
    auto key_at = [&](int i) -> uint32_t { return cached ? cache[i] : order_key(lg[i]); };

    uint32_t prefix = 0u, mask = 0u, remaining = (uint32_t)topk;
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kThreads) hist[i] = 0u;
        __syncthreads();
        for (int base = 0; base < L; base += kThreads) {
            const int i = base + threadIdx.x;
            bool in = false;
            uint32_t digit = 0u;
            if (i < L) {
                const uint32_t k = key_at(i);
                in = (k & mask) == prefix;
                digit = (k >> shift) & 0xFFu;
            }
            // warp-aggregated histogram update: one atomic per distinct digit
            const uint32_t active = __ballot_sync(0xffffffffu, in);
            if (in) {
                const uint32_t peers = __match_any_sync(active, digit);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[digit], (uint32_t)__popc(peers));
            }
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l owns bins 255-8l .. 248-8l (largest digits first)
            const int top = 255 - 8 * lane;
            uint32_t c[8], s = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) { c[j] = hist[top - j]; s += c[j]; }
            uint32_t incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t excl = incl - s;
            if (excl < remaining && remaining <= incl) {
                uint32_t cum = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (cum + c[j] >= remaining) {
                        sel_digit = (uint32_t)(top - j);
                        sel_remaining = remaining - cum;
                        break;
                    }
                    cum += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= sel_digit << shift;
        mask |= 0xFFu << shift;
        remaining = sel_remaining;
        __syncthreads();
    }

    // Ordered selection: keys > T, then the first `remaining` keys == T.
    const uint32_t T = prefix, need_eq = remaining;
    uint32_t gt_run = 0u, eq_run = 0u;
    for (int base = 0; base < L; base += kThreads) {
        const int i = base + threadIdx.x;
        uint32_t k = 0u;
        bool gt = false, eq = false;
        if (i < L) {
            k = key_at(i);
            gt = k > T;
            eq = k == T;
        }
        const uint32_t packed = (gt ? 1u : 0u) | (eq ? (1u << 16) : 0u);
        const uint32_t excl = block_excl_scan(packed, warp_buf, &chunk_total);
        const uint32_t gt_before = gt_run + (excl & 0xFFFFu);
        const uint32_t eq_before = eq_run + (excl >> 16);
        if (gt || (eq && eq_before < need_eq)) {
            const uint32_t pos = gt_before + (eq_before < need_eq ? eq_before : need_eq);
            out[pos] = ptr[i];
        }
        const uint32_t tot = chunk_total;
        gt_run += tot & 0xFFFFu;
        eq_run += tot >> 16;
        __syncthreads();
    }
}

}  // namespace
}  // namespace nsa

extern "C" nsa_status nsa_topk_transform(const float *logits_dev, int64_t logits_ld,
                                         const int32_t *row_len_dev, const int32_t *row_to_req_dev,
                                         const int32_t *page_table_1_dev, int64_t pt_ld, int R,
                                         int topk, int max_row_len, int32_t *indices_dev,
                                         int64_t indices_ld, int32_t *status_dev, nsa_stream_t stream)
{
    using namespace nsa;
    if (R < 0 || topk < 1 || topk > 4096 || max_row_len < 0) return NSA_ERR_INVALID_ARG;
    if (indices_ld < topk || logits_ld < max_row_len || pt_ld < max_row_len) return NSA_ERR_INVALID_ARG;
    if (R == 0) return NSA_OK;
    if (!logits_dev || !row_len_dev || !row_to_req_dev || !page_table_1_dev || !indices_dev)
        return NSA_ERR_INVALID_ARG;
    int cap = max_row_len > topk ? (max_row_len < kCacheCap ? max_row_len : kCacheCap) : 0;
    const size_t smem = (size_t)cap * sizeof(uint32_t);
    NSA_CUDA_TRY(cudaFuncSetAttribute(topk_transform_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem));
    topk_transform_kernel<<<(unsigned)R, kThreads, smem, (cudaStream_t)stream>>>(
        logits_dev, logits_ld, row_len_dev, row_to_req_dev, page_table_1_dev, pt_ld, topk, max_row_len,
        cap, indices_dev, indices_ld, status_dev);
    return launch_status();
}
