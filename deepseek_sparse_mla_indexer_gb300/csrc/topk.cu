// nsa_topk_transform: per-row top-k of the indexer scores, mapped to KV slots.
//
// [NSA] NSAIndexerMetadata.topk_transform (the fused variant that emits KV
// slots of the page table instead of positions), [DSA]
// transform_index_page_table_* with page size 1 and _pad_topk_indices (-1
// padding).
//
// Rows up to kCacheCap scores: one block of 1024 threads per row, the scores
// read from HBM once and kept in shared memory; longer rows: a cluster of up
// to 8 blocks per row (below).  Scores become order-preserving 32-bit keys
// (-0 folded onto +0, NaN below every number).  The k-th largest key is
// located by a most-significant-digit radix select with 11/11/10-bit digits:
// each pass histograms the keys that still match the chosen prefix (eight
// replicated shared-memory histograms spread the atomic traffic of the few
// crowded bins), and a block scan over the bins, largest
// digit first, picks the digit holding the k-th key.  A pass stops the search
// early when the whole bin is selected.  A final ordered pass keeps every key
// above the threshold and the first (k - #above) keys equal to it, in
// position order, so ties go to the lower position and the output comes out
// sorted without a sort: each thread owns a run of consecutive positions and
// one block scan of its (#above, #equal) counts places them; the page-table
// gathers of all output slots then go out together.
#include <algorithm>

#include "nsa_internal.cuh"

namespace nsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kBins = 2048;
constexpr int kCopies = 8;             // replicated histograms (warp w adds into copy w % 8)
constexpr int kCacheCap = 40 * 1024;  // 160 KB of keys (+ 64 KB of histograms)
// Dynamic shared memory of topk_transform_kernel: the histograms, then `cap` cached keys.
constexpr size_t row_kernel_smem_bytes(int cap) { return (size_t)(kCopies * kBins + cap) * sizeof(uint32_t); }
static_assert(row_kernel_smem_bytes(kCacheCap) <= 232448, "shared memory per block");
constexpr int kItems = 4;             // consecutive elements per thread in the cluster's ordered pass

__device__ __forceinline__ uint32_t order_key(float x)
{
    uint32_t u = __float_as_uint(x);
    if (x != x) return 0u;       // NaN ranks lowest
    if ((u << 1) == 0u) u = 0u;  // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive block scan of one value per thread; *total receives the block sum.
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t *warp_buf, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_buf[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < (int)(blockDim.x >> 5) ? warp_buf[lane] : 0u;  // only the block's real warps
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_buf[lane] = w;
        if (lane == 31) *total = w;
    }
    __syncthreads();
    const uint32_t incl = x + (warp > 0 ? warp_buf[warp - 1] : 0u);
    __syncthreads();
    return incl;
}

// Keys of lg[s0 .. s0 + n) into cache[0 .. n): 16-byte loads, all in flight at once.
template <int NT, int MAXV>
__device__ __forceinline__ void fill_keys(const float *lg, int s0, int n, uint32_t *cache)
{
    const float *src = lg + s0;
    if ((((uintptr_t)src) & 15) == 0) {
        const int nv = n >> 2;
        for (int base = 0; base < nv; base += NT * MAXV) {
            float4 v[MAXV];
#pragma unroll
            for (int u = 0; u < MAXV; ++u) {
                const int j = base + u * NT + (int)threadIdx.x;
                if (j < nv) v[u] = __ldg(reinterpret_cast<const float4 *>(src) + j);
            }
#pragma unroll
            for (int u = 0; u < MAXV; ++u) {
                const int j = base + u * NT + (int)threadIdx.x;
                if (j < nv)
                    reinterpret_cast<uint4 *>(cache)[j] =
                        make_uint4(order_key(v[u].x), order_key(v[u].y), order_key(v[u].z), order_key(v[u].w));
            }
        }
        for (int i = (nv << 2) + (int)threadIdx.x; i < n; i += NT) cache[i] = order_key(src[i]);
    } else {
        for (int i = threadIdx.x; i < n; i += NT) cache[i] = order_key(src[i]);
    }
}

__global__ void __launch_bounds__(kThreads)
topk_transform_kernel(const float *logits, int64_t logits_ld, const int32_t *row_len,
                      const int32_t *row_to_req, const int32_t *pt, int64_t pt_ld, const int32_t *req_offset,
                      int topk, int max_row_len, int cache_cap, int32_t *indices, int64_t indices_ld,
                      int32_t *status)
{
    extern __shared__ uint32_t dyn[];
    uint32_t *hist = dyn;                     // [kCopies][kBins]; then the selected positions
    uint32_t *cache = dyn + kCopies * kBins;  // [cache_cap]
    __shared__ uint32_t warp_buf[32];
    __shared__ uint32_t total;
    __shared__ uint32_t sel_digit, sel_need, sel_exact;

    pdl_trigger();
    pdl_wait();  // the scores come from the indexer
    const int r = blockIdx.x;
    const int L = row_len[r];
    const int b = row_to_req[r];
    int32_t *out = indices + (int64_t)r * indices_ld;
    // paged: the KV slot page_table_1[b, s]; ragged: s + the request's offset
    const int32_t *ptr = pt ? pt + (int64_t)b * pt_ld : nullptr;
    const int32_t off = req_offset ? req_offset[b] : 0;
    auto slot_of = [&](int s) -> int32_t { return ptr ? ptr[s] : off + s; };
    const float *lg = logits + (int64_t)r * logits_ld;
    const int tid = threadIdx.x;

    if (L < 0 || L > max_row_len) {
        if (tid == 0) set_status(status, NSA_ERR_BOUNDS);
        for (int i = tid; i < topk; i += kThreads) out[i] = -1;
        return;
    }
    if (L <= topk) {
        for (int i = tid; i < topk; i += kThreads) out[i] = i < L ? slot_of(i) : -1;
        return;
    }

    const bool cached = L <= cache_cap;
    if (cached) fill_keys<kThreads, 8>(lg, 0, L, cache);
    auto key_at = [&](int i) -> uint32_t { return cached ? cache[i] : order_key(lg[i]); };

    // radix select: find the resolution shift S, value V and count `need`
    // such that keys with (key >> S) > V are all selected and `need` of the
    // keys with (key >> S) == V are selected (the lowest positions).
    uint32_t prefix = 0u, need = (uint32_t)topk;
    int S = 32;
    uint32_t *myhist = hist + (size_t)((tid >> 5) % kCopies) * kBins;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int width = pass < 2 ? 11 : 10;
        const int shift = S - width;
        const uint32_t dmask = (1u << width) - 1u;
        for (int i = tid; i < kCopies * kBins; i += kThreads) hist[i] = 0u;
        __syncthreads();
        auto count_key = [&](uint32_t k) {
            if (S == 32 || (k >> S) == prefix) atomicAdd(&myhist[(k >> shift) & dmask], 1u);
        };
        if (cached) {  // 16-byte reads of four consecutive keys
            for (int i4 = tid; i4 < (L >> 2); i4 += kThreads) {
                const uint4 k = reinterpret_cast<const uint4 *>(cache)[i4];
                count_key(k.x); count_key(k.y); count_key(k.z); count_key(k.w);
            }
            for (int i = (L & ~3) + tid; i < L; i += kThreads) count_key(cache[i]);
        } else {
            for (int i = tid; i < L; i += kThreads) count_key(key_at(i));
        }
        __syncthreads();
        // thread t owns digits (2047 - 2t) and (2046 - 2t): largest digits first
        const int d_hi = kBins - 1 - 2 * tid, d_lo = d_hi - 1;
        uint32_t c_hi = 0u, c_lo = 0u;
        if (d_hi <= (int)dmask) {
#pragma unroll
            for (int c = 0; c < kCopies; ++c) c_hi += hist[c * kBins + d_hi];
        }
        if (d_lo >= 0 && d_lo <= (int)dmask) {
#pragma unroll
            for (int c = 0; c < kCopies; ++c) c_lo += hist[c * kBins + d_lo];
        }
        const uint32_t incl = block_incl_scan(c_hi + c_lo, warp_buf, &total);
        const uint32_t excl = incl - c_hi - c_lo;
        if (excl < need && need <= incl) {
            if (excl + c_hi >= need) {
                sel_digit = (uint32_t)d_hi;
                sel_need = need - excl;
                sel_exact = (c_hi == need - excl);
            } else {
                sel_digit = (uint32_t)d_lo;
                sel_need = need - excl - c_hi;
                sel_exact = (c_lo == need - excl - c_hi);
            }
        }
        __syncthreads();
        prefix = (S == 32 ? 0u : (prefix << width)) | sel_digit;
        need = sel_need;
        S = shift;
        const bool exact = sel_exact != 0u;
        __syncthreads();
        if (exact) break;
    }

    // ordered selection: thread t owns the C consecutive positions from t*C (C = 4 x an
    // odd number: 16-byte reads, and the threads of a warp hit different bank groups);
    // one block scan of (#above, #equal) places every selected position in order
    const int C = 4 * (((L + 4 * kThreads - 1) / (4 * kThreads)) | 1);
    const int p0 = min(L, tid * C), p1 = min(L, p0 + C);
    uint32_t *sel = hist;  // output slot -> position (the histograms are dead)
    auto place = [&](uint32_t n_gt, uint32_t n_eq, uint32_t &gt_before, uint32_t &eq_before) {
        if (L < 65536) {  // both counts fit 16 bits
            const uint32_t packed = n_gt | (n_eq << 16);
            const uint32_t ex = block_incl_scan(packed, warp_buf, &total) - packed;
            gt_before = ex & 0xFFFFu;
            eq_before = ex >> 16;
        } else {
            gt_before = block_incl_scan(n_gt, warp_buf, &total) - n_gt;
            eq_before = block_incl_scan(n_eq, warp_buf, &total) - n_eq;
        }
    };
    auto record = [&](bool above, int pos, uint32_t &gt_before, uint32_t &eq_before) {
        if (above) {
            sel[gt_before + (eq_before < need ? eq_before : need)] = (uint32_t)pos;
            ++gt_before;
        } else {
            if (eq_before < need) sel[gt_before + eq_before] = (uint32_t)pos;
            ++eq_before;
        }
    };
    if (cached && C <= 64) {
        // one read of the run: its classes kept as two 64-bit masks (above, equal)
        uint64_t mgt = 0ull, meq = 0ull;
        for (int i = p0; i < p1; i += 4) {
            uint32_t k[4];
            if (i + 4 <= p1) {
                const uint4 v = *reinterpret_cast<const uint4 *>(cache + i);
                k[0] = v.x; k[1] = v.y; k[2] = v.z; k[3] = v.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) k[j] = i + j < p1 ? cache[i + j] : 0u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (i + j >= p1) continue;
                const uint32_t v = k[j] >> S;
                const uint64_t bit = 1ull << (i + j - p0);
                if (v > prefix) mgt |= bit;
                else if (v == prefix) meq |= bit;
            }
        }
        uint32_t gt_before, eq_before;
        place((uint32_t)__popcll(mgt), (uint32_t)__popcll(meq), gt_before, eq_before);
        for (uint64_t m = mgt | meq; m; m &= m - 1) {
            const int bit = __ffsll((long long)m) - 1;
            record(((mgt >> bit) & 1ull) != 0ull, p0 + bit, gt_before, eq_before);
        }
    } else {
        auto cls_of = [&](int i) -> uint32_t {
            const uint32_t v = key_at(i) >> S;
            return v > prefix ? 2u : (v == prefix ? 1u : 0u);
        };
        uint32_t n_gt = 0u, n_eq = 0u;
        for (int i = p0; i < p1; ++i) {
            const uint32_t c = cls_of(i);
            n_gt += c == 2u;
            n_eq += c == 1u;
        }
        uint32_t gt_before, eq_before;
        place(n_gt, n_eq, gt_before, eq_before);
        for (int i = p0; i < p1; ++i) {
            const uint32_t c = cls_of(i);
            if (c != 0u) record(c == 2u, i, gt_before, eq_before);
        }
    }
    __syncthreads();
    for (int j = tid; j < topk; j += kThreads) out[j] = slot_of((int)sel[j]);
}


// ---------------------------------------------------------------- cluster variant
// Long rows: a thread-block cluster of C CTAs per row, each owning a slice of
// the row.  Histograms and selection counts are combined through distributed
// shared memory between hardware cluster barriers (no spin-waits); every CTA
// reaches the same decisions from the same merged data, so control flow stays
// uniform across the cluster.
constexpr int kCThreads = 512;
constexpr int kCCopies = 4;
constexpr int kCMaxCluster = 8;
constexpr int kCSliceCap = 16 * 1024;  // keys of one slice cached in shared memory

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 32-bit load from the same shared-memory variable of CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t ld_cluster(const uint32_t *local, uint32_t rank)
{
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), ra, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
    return v;
}

// 16-byte load from CTA `rank` of the cluster (address 16-byte aligned).
__device__ __forceinline__ uint4 ld_cluster4(const uint32_t *local, uint32_t rank)
{
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), ra;
    uint4 v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(ra)
                 : "memory");
    return v;
}

__global__ void __launch_bounds__(kCThreads)
topk_cluster_kernel(const float *logits, int64_t logits_ld, const int32_t *row_len, const int32_t *row_to_req,
                    const int32_t *pt, int64_t pt_ld, const int32_t *req_offset, int topk, int max_row_len,
                    int32_t *indices, int64_t indices_ld, int32_t *status)
{
    extern __shared__ uint32_t cache[];           // [kCSliceCap] keys of this slice
    __shared__ uint32_t hist[kCCopies * kBins];  // replicated local histogram
    __shared__ __align__(16) uint32_t merged[kBins];  // this CTA's combined copy (read by the peers)
    __shared__ uint32_t warp_buf[32];
    __shared__ uint32_t total;
    __shared__ uint32_t sel_digit, sel_need, sel_exact;
    __shared__ uint32_t counts[2];               // (#above, #equal) in this slice

    pdl_trigger();
    pdl_wait();  // the scores come from the indexer
    const uint32_t rank = cluster_rank();
    uint32_t csize;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
    const int r = blockIdx.x / (int)csize;
    const int tid = threadIdx.x;
    int L = row_len[r];
    const int b = row_to_req[r];
    int32_t *out = indices + (int64_t)r * indices_ld;
    // paged: the KV slot page_table_1[b, s]; ragged: s + the request's offset
    const int32_t *ptr = pt ? pt + (int64_t)b * pt_ld : nullptr;
    const int32_t off = req_offset ? req_offset[b] : 0;
    auto slot_of = [&](int s) -> int32_t { return ptr ? ptr[s] : off + s; };
    const float *lg = logits + (int64_t)r * logits_ld;

    if (L < 0 || L > max_row_len) {  // same decision in every CTA of the cluster
        if (rank == 0) {
            if (tid == 0) set_status(status, NSA_ERR_BOUNDS);
            for (int i = tid; i < topk; i += kCThreads) out[i] = -1;
        }
        return;
    }
    if (L <= topk) {
        if (rank == 0)
            for (int i = tid; i < topk; i += kCThreads) out[i] = i < L ? slot_of(i) : -1;
        return;
    }

    // this CTA's slice of the row (a multiple of 4 positions)
    const int seg = ((L + (int)csize - 1) / (int)csize + 3) & ~3;
    const int s0 = min(L, (int)rank * seg), s1 = min(L, s0 + seg);
    const int n = s1 - s0;
    const bool cached = n <= kCSliceCap;
    if (cached) fill_keys<kCThreads, 8>(lg, s0, n, cache);
    auto key_at = [&](int i) -> uint32_t { return cached ? cache[i] : order_key(lg[s0 + i]); };

    uint32_t prefix = 0u, need = (uint32_t)topk;
    int S = 32;
    uint32_t *myhist = hist + (size_t)((tid >> 5) % kCCopies) * kBins;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int width = pass < 2 ? 11 : 10;
        const int shift = S - width;
        const uint32_t dmask = (1u << width) - 1u;
        for (int i = tid; i < kCCopies * kBins; i += kCThreads) hist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < n; i += kCThreads) {
            const uint32_t k = key_at(i);
            if (S == 32 || (k >> S) == prefix) atomicAdd(&myhist[(k >> shift) & dmask], 1u);
        }
        __syncthreads();
        for (int d = tid; d < kBins; d += kCThreads) {
            uint32_t v = 0u;
#pragma unroll
            for (int c = 0; c < kCCopies; ++c) v += hist[c * kBins + d];
            merged[d] = v;
        }
        if (tid == 0) {  // a decision every CTA agrees on even if no bin were chosen
            sel_digit = 0u;
            sel_need = need;
            sel_exact = 1u;
        }
        cluster_sync();  // every slice histogram is complete
        // thread t owns digits 2047-4t .. 2044-4t (largest first); sum them over the cluster
        const int dlo = kBins - 4 - 4 * tid;  // digits dlo .. dlo+3, one 16-byte vector
        uint4 acc = make_uint4(0u, 0u, 0u, 0u);
        if (dlo <= (int)dmask) {
            for (uint32_t q = 0; q < csize; ++q) {
                const uint4 v = ld_cluster4(&merged[dlo], q);
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
        }
        const uint32_t c4[4] = {acc.w, acc.z, acc.y, acc.x};  // digit dlo+3 first
        const uint32_t sum = acc.x + acc.y + acc.z + acc.w;
        const uint32_t incl = block_incl_scan(sum, warp_buf, &total);
        uint32_t excl = incl - sum;
        if (excl < need && need <= incl) {
            uint32_t cum = excl;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (cum + c4[j] >= need) {
                    sel_digit = (uint32_t)(kBins - 1 - 4 * tid - j);
                    sel_need = need - cum;
                    sel_exact = (c4[j] == need - cum);
                    break;
                }
                cum += c4[j];
            }
        }
        cluster_sync();  // peers are done reading `merged`; sel_* written
        prefix = (S == 32 ? 0u : (prefix << width)) | sel_digit;
        need = sel_need;
        S = shift;
        const bool exact = sel_exact != 0u;
        __syncthreads();
        if (exact) break;
    }

    // counts of this slice, then the offsets of the lower-ranked slices
    uint32_t n_gt = 0u, n_eq = 0u;
    for (int i = tid; i < n; i += kCThreads) {
        const uint32_t v = key_at(i) >> S;
        n_gt += v > prefix;
        n_eq += v == prefix;
    }
    block_incl_scan(n_gt, warp_buf, &total);
    if (tid == 0) counts[0] = total;
    block_incl_scan(n_eq, warp_buf, &total);
    if (tid == 0) counts[1] = total;
    cluster_sync();
    uint32_t gt_run = 0u, eq_run = 0u;
    for (uint32_t q = 0; q < rank; ++q) {
        gt_run += ld_cluster(&counts[0], q);
        eq_run += ld_cluster(&counts[1], q);
    }

    for (int base = 0; base < n; base += kCThreads * kItems) {
        const int i0 = base + tid * kItems;
        uint32_t cls[kItems];
        uint32_t a_gt = 0u, a_eq = 0u;
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            cls[j] = 0u;
            if (i0 + j < n) {
                const uint32_t v = key_at(i0 + j) >> S;
                cls[j] = v > prefix ? 2u : (v == prefix ? 1u : 0u);
            }
            a_gt += cls[j] == 2u;
            a_eq += cls[j] == 1u;
        }
        const uint32_t packed = a_gt | (a_eq << 16);
        const uint32_t incl = block_incl_scan(packed, warp_buf, &total);
        uint32_t gt_before = gt_run + ((incl - packed) & 0xFFFFu);
        uint32_t eq_before = eq_run + ((incl - packed) >> 16);
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            if (cls[j] == 2u) {
                out[gt_before + (eq_before < need ? eq_before : need)] = slot_of(s0 + i0 + j);
                ++gt_before;
            } else if (cls[j] == 1u) {
                if (eq_before < need) out[gt_before + eq_before] = slot_of(s0 + i0 + j);
                ++eq_before;
            }
        }
        gt_run += total & 0xFFFFu;
        eq_run += total >> 16;
    }
    cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

}  // namespace
}  // namespace nsa

namespace nsa {
namespace {

nsa_status topk_launch(const float *logits_dev, int64_t logits_ld, const int32_t *row_len_dev,
                       const int32_t *row_to_req_dev, const int32_t *page_table_1_dev, int64_t pt_ld,
                       const int32_t *req_offset_dev, int R, int topk, int max_row_len, int32_t *indices_dev,
                       int64_t indices_ld, int32_t *status_dev, nsa_stream_t stream)
{
    using namespace nsa;
    if (R < 0 || topk < 1 || topk > 4096 || max_row_len < 0) return NSA_ERR_INVALID_ARG;
    if (indices_ld < topk || logits_ld < max_row_len || (page_table_1_dev && pt_ld < max_row_len))
        return NSA_ERR_INVALID_ARG;
    if (R == 0) return NSA_OK;
    if (!logits_dev || !row_len_dev || !row_to_req_dev || !indices_dev || (!page_table_1_dev && !req_offset_dev))
        return NSA_ERR_INVALID_ARG;
    // rows beyond the single-block key cache: one cluster of up to 8 CTAs per row
    const int csize = max_row_len > kCacheCap ? (int)std::min<int64_t>(kCMaxCluster, ceil_div(max_row_len, kCSliceCap)) : 1;
    if (csize > 1 && (int64_t)R * csize <= 2147483647LL) {
        NSA_CUDA_TRY(cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)(kCSliceCap * sizeof(uint32_t))));
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(R * csize));
        cfg.blockDim = dim3(kCThreads);
        cfg.dynamicSmemBytes = kCSliceCap * sizeof(uint32_t);
        cfg.stream = (cudaStream_t)stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)csize;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1] = pdl_attribute();
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        NSA_CUDA_TRY(cudaLaunchKernelEx(&cfg, topk_cluster_kernel, logits_dev, logits_ld, row_len_dev,
                                        row_to_req_dev, page_table_1_dev, pt_ld, req_offset_dev, topk, max_row_len,
                                        indices_dev, indices_ld, status_dev));
        return NSA_OK;
    }
    const int cap = max_row_len > topk ? (max_row_len < kCacheCap ? max_row_len : kCacheCap) : 0;
    const size_t smem = row_kernel_smem_bytes(cap);
    NSA_CUDA_TRY(cudaFuncSetAttribute(topk_transform_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)R);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    NSA_CUDA_TRY(cudaLaunchKernelEx(&cfg, topk_transform_kernel, logits_dev, logits_ld, row_len_dev, row_to_req_dev,
                                    page_table_1_dev, pt_ld, req_offset_dev, topk, max_row_len, cap, indices_dev,
                                    indices_ld, status_dev));
    return NSA_OK;
}

}  // namespace
}  // namespace nsa

extern "C" nsa_status nsa_topk_transform(const float *logits_dev, int64_t logits_ld,
                                         const int32_t *row_len_dev, const int32_t *row_to_req_dev,
                                         const int32_t *page_table_1_dev, int64_t pt_ld, int R,
                                         int topk, int max_row_len, int32_t *indices_dev,
                                         int64_t indices_ld, int32_t *status_dev, nsa_stream_t stream)
{
    if (!page_table_1_dev && R > 0) return NSA_ERR_INVALID_ARG;
    return nsa::topk_launch(logits_dev, logits_ld, row_len_dev, row_to_req_dev, page_table_1_dev, pt_ld, nullptr, R,
                            topk, max_row_len, indices_dev, indices_ld, status_dev, stream);
}

extern "C" nsa_status nsa_topk_transform_ragged(const float *logits_dev, int64_t logits_ld,
                                                const int32_t *row_len_dev, const int32_t *row_to_req_dev,
                                                const int32_t *req_offset_dev, int R, int topk, int max_row_len,
                                                int32_t *indices_dev, int64_t indices_ld, int32_t *status_dev,
                                                nsa_stream_t stream)
{
    if (!req_offset_dev && R > 0) return NSA_ERR_INVALID_ARG;
    return nsa::topk_launch(logits_dev, logits_ld, row_len_dev, row_to_req_dev, nullptr, 0, req_offset_dev, R, topk,
                            max_row_len, indices_dev, indices_ld, status_dev, stream);
}
