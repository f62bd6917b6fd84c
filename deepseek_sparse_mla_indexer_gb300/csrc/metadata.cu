// nsa_metadata: the per-step metadata of the sparse-attention backend in one
// launch.  Block 0 builds every length / offset array (they are O(B + R)
// and need block-wide prefix sums) and records the pool rows it read
// (req_rows); the other blocks copy the page table rows out of req_to_token
// and derive the page-granular table on the fly, or, when no page_table_1 is
// asked for, read only each page's first slot to derive its page id.
//
// Follows [DSA] DeepseekSparseAttnBackend.init_forward_metadata (decode,
// target-verify and extend branches), _cal_indexer_k_start_end and
// compute_cu_seqlens; [NSA-diff] the target-verify branch.
#include "nsa_internal.cuh"

namespace nsa {
namespace {

constexpr int kRowThreads = 1024;

struct MetaParams {
    int mode, B, R, W, n_draft, topk, ps;
    const int32_t *seq_lens, *extend_lens, *r2t, *rpi;
    int64_t r2t_ld, pool_rows;
    nsa_metadata_out out;
    int32_t *status;
};

// out[0] = 0, out[i + 1] = f(0) + ... + f(i) for i < n, with the whole block;
// the same values also go to `copy` (shared memory) when it is given.
template <class F>
__device__ void block_cumsum_pad(int n, F f, int32_t *out, int32_t *copy = nullptr)
{
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    if (threadIdx.x == 0) {
        carry = 0;
        out[0] = 0;
        if (copy) copy[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < n; base += blockDim.x) {
        int i = base + threadIdx.x;
        int x = i < n ? f(i) : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_tot[lane] = w;
        }
        __syncthreads();
        int incl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x;
        if (i < n) {
            out[i + 1] = incl;
            if (copy) copy[i + 1] = incl;
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = incl;
        __syncthreads();
    }
}

constexpr int kSmemB = 2048;  // requests staged in shared memory by the fast path

// Per-request lengths staged once in shared memory; every per-row value is
// computed from there, so the block never reads back what it wrote to global.
__device__ void build_rows_smem(const MetaParams &p)
{
    __shared__ int32_t s_seq[kSmemB], s_ext[kSmemB], s_cuq[kSmemB + 1], s_cuk[kSmemB + 1];
    const nsa_metadata_out &o = p.out;
    const int draft = p.mode == NSA_MODE_TARGET_VERIFY ? p.n_draft : 0;
    const bool extend = p.mode == NSA_MODE_EXTEND;
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
        const int c = p.seq_lens[b] + draft;
        s_seq[b] = c;
        if (extend) s_ext[b] = p.extend_lens[b];
        if (c < 0 || c > p.W) set_status(p.status, NSA_ERR_BOUNDS);
        o.cache_seqlens[b] = c;
    }
    __syncthreads();
    block_cumsum_pad(p.B, [&](int b) { return s_seq[b]; }, o.cu_seqlens_k, s_cuk);
    if (extend) {
        block_cumsum_pad(p.B, [&](int b) { return s_ext[b]; }, o.cu_seqlens_q, s_cuq);
    } else {
        const int n = p.mode == NSA_MODE_DECODE ? p.B : p.R;
        for (int i = threadIdx.x; i <= n; i += blockDim.x) o.cu_seqlens_q[i] = i;
    }
    __syncthreads();
    // (request, position in the request, rows of the request) of row r
    auto row_info = [&](int r, int &b, int &q, int &i) {
        if (p.mode == NSA_MODE_DECODE) {
            b = r; q = 1; i = 0;
        } else if (p.mode == NSA_MODE_TARGET_VERIFY) {
            b = r / p.n_draft; q = p.n_draft; i = r - b * p.n_draft;
        } else {
            int lo = 0, hi = p.B - 1;  // largest b with cu_seqlens_q[b] <= r
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_cuq[mid] <= r) lo = mid; else hi = mid - 1;
            }
            b = lo; q = s_ext[b]; i = r - s_cuq[b];
        }
    };
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
        int b, q, i;
        row_info(r, b, q, i);
        if (i >= q) set_status(p.status, NSA_ERR_BOUNDS);  // R exceeds sum(extend_lens)
        const int L = s_seq[b] - q + 1 + i;  // arange(kv - q + 1, kv + 1)[i]
        o.seqlens_expanded[r] = L;
        o.nsa_cache_seqlens[r] = L < p.topk ? L : p.topk;
        o.row_to_req[r] = b;
        if (extend && o.indexer_ks) {
            const int ks = s_cuk[b];
            o.indexer_ks[r] = ks;
            o.indexer_ke[r] = ks + L;
        }
    }
    block_cumsum_pad(p.R, [&](int r) {
        int b, q, i;
        row_info(r, b, q, i);
        const int L = s_seq[b] - q + 1 + i;
        return L < p.topk ? L : p.topk;
    }, o.nsa_cu_seqlens_k);
    for (int i = threadIdx.x; i <= p.R; i += blockDim.x) o.nsa_cu_seqlens_q[i] = i;
}

__device__ void build_rows(const MetaParams &p)
{
    const nsa_metadata_out &o = p.out;
    const int draft = p.mode == NSA_MODE_TARGET_VERIFY ? p.n_draft : 0;

    // cache_seqlens and cu_seqlens_k
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
        int c = p.seq_lens[b] + draft;
        if (c < 0 || c > p.W) set_status(p.status, NSA_ERR_BOUNDS);
        o.cache_seqlens[b] = c;
    }
    block_cumsum_pad(p.B, [&](int b) { return p.seq_lens[b] + draft; }, o.cu_seqlens_k);

    // cu_seqlens_q
    if (p.mode == NSA_MODE_EXTEND) {
        block_cumsum_pad(p.B, [&](int b) { return p.extend_lens[b]; }, o.cu_seqlens_q);
    } else {
        const int n = p.mode == NSA_MODE_DECODE ? p.B : p.R;
        for (int i = threadIdx.x; i <= n; i += blockDim.x) o.cu_seqlens_q[i] = i;
    }
    __syncthreads();

    // per-row arrays
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
        int b, q, i;
        if (p.mode == NSA_MODE_DECODE) {
            b = r; q = 1; i = 0;
        } else if (p.mode == NSA_MODE_TARGET_VERIFY) {
            b = r / p.n_draft; q = p.n_draft; i = r - b * p.n_draft;
        } else {
            int lo = 0, hi = p.B - 1;  // largest b with cu_seqlens_q[b] <= r
            while (lo < hi) {
                int mid = (lo + hi + 1) >> 1;
                if (o.cu_seqlens_q[mid] <= r) lo = mid; else hi = mid - 1;
            }
            b = lo; q = p.extend_lens[b]; i = r - o.cu_seqlens_q[b];
            if (i >= q) set_status(p.status, NSA_ERR_BOUNDS);  // R exceeds sum(extend_lens)
        }
        const int L = p.seq_lens[b] + draft - q + 1 + i;  // arange(kv - q + 1, kv + 1)[i]
        o.seqlens_expanded[r] = L;
        o.nsa_cache_seqlens[r] = L < p.topk ? L : p.topk;
        o.row_to_req[r] = b;
        if (p.mode == NSA_MODE_EXTEND && o.indexer_ks) {
            const int ks = o.cu_seqlens_k[b];
            o.indexer_ks[r] = ks;
            o.indexer_ke[r] = ks + L;
        }
    }
    __syncthreads();
    block_cumsum_pad(p.R, [&](int r) { return o.nsa_cache_seqlens[r]; }, o.nsa_cu_seqlens_k);
    for (int i = threadIdx.x; i <= p.R; i += blockDim.x) o.nsa_cu_seqlens_q[i] = i;
}

constexpr int kSeg = 4096;  // page-table entries per copy segment (one 16-byte load per thread)

// page_table_1[b, 0:W] = req_to_token[rpi[b], 0:W], and every page start also
// lands in real_page_table.  Segments of kSeg entries are spread over the copy
// blocks; 16-byte vector accesses when both rows are 16-byte aligned.
__device__ void copy_tables(const MetaParams &p, int first_seg, int seg_stride)
{
    const nsa_metadata_out &o = p.out;
    if (!o.page_table_1) {
        // no copied table: only the page ids, one thread per page of each request
        const int npg = (int)ceil_div(p.W, p.ps);
        const int64_t total_pg = (int64_t)p.B * npg;
        for (int64_t g = (int64_t)first_seg * blockDim.x + threadIdx.x; g < total_pg;
             g += (int64_t)seg_stride * blockDim.x) {
            const int b = (int)(g / npg), q = (int)(g - (int64_t)b * npg);
            const int32_t row = p.rpi[b];
            if (row < 0 || row >= p.pool_rows) {
                if (q == 0) set_status(p.status, NSA_ERR_BOUNDS);
                continue;
            }
            o.real_page_table[(int64_t)b * o.real_page_table_ld + q] =
                floor_div(p.r2t[(int64_t)row * p.r2t_ld + (int64_t)q * p.ps], p.ps);
        }
        return;
    }
    const int segs_per_row = (int)ceil_div(p.W, kSeg);
    const int64_t total = (int64_t)p.B * segs_per_row;
    for (int64_t g = first_seg; g < total; g += seg_stride) {
        const int b = (int)(g / segs_per_row);
        const int t0 = (int)(g - (int64_t)b * segs_per_row) * kSeg;
        const int t1 = min(p.W, t0 + kSeg);
        const int32_t row = p.rpi[b];
        if (row < 0 || row >= p.pool_rows) {
            if (threadIdx.x == 0 && t0 == 0) set_status(p.status, NSA_ERR_BOUNDS);
            continue;
        }
        const int32_t *src = p.r2t + (int64_t)row * p.r2t_ld;
        int32_t *dst = o.page_table_1 + (int64_t)b * o.page_table_1_ld;
        int32_t *real = o.real_page_table + (int64_t)b * o.real_page_table_ld;
        const bool vec = (((uintptr_t)src | (uintptr_t)dst) & 15) == 0;
        if (vec) {
            // 4 independent 16-byte loads in flight per thread
            constexpr int kU = 4;
            for (int tb = t0 + 4 * (int)threadIdx.x; tb < t1; tb += 4 * kU * blockDim.x) {
                int4 v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int t = tb + u * 4 * blockDim.x;
                    if (t + 4 <= t1) v[u] = *reinterpret_cast<const int4 *>(src + t);
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int t = tb + u * 4 * blockDim.x;
                    if (t + 4 <= t1) {
                        *reinterpret_cast<int4 *>(dst + t) = v[u];
                        const int32_t e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                        const int first = (p.ps - t % p.ps) % p.ps;  // offset of the first page start in t..t+3
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (j >= first && (j - first) % p.ps == 0) real[(t + j) / p.ps] = floor_div(e[j], p.ps);
                    } else {
                        for (int j = t; j < t1; ++j) {
                            const int32_t x = src[j];
                            dst[j] = x;
                            if (j % p.ps == 0) real[j / p.ps] = floor_div(x, p.ps);
                        }
                    }
                }
            }
        } else {
            for (int t = t0 + (int)threadIdx.x; t < t1; t += blockDim.x) {
                const int32_t v = src[t];
                dst[t] = v;
                if (t % p.ps == 0) real[t / p.ps] = floor_div(v, p.ps);
            }
        }
    }
}

// Two 1024-thread blocks per SM (at most 32 registers a thread): the copy blocks of
// a 32-request decode step then start in one wave instead of two.
__global__ void __launch_bounds__(kRowThreads, 2) metadata_kernel(MetaParams p)
{
    pdl_trigger();
    pdl_wait();  // the previous step's kernels may still read these tables
    if (blockIdx.x == 0) {
        if (p.B <= kSmemB) build_rows_smem(p);
        else build_rows(p);
        if (p.out.req_rows)
            for (int b = threadIdx.x; b < p.B; b += blockDim.x) p.out.req_rows[b] = p.rpi[b];
    } else {
        copy_tables(p, (int)blockIdx.x - 1, (int)gridDim.x - 1);
    }
}

}  // namespace
}  // namespace nsa

extern "C" nsa_status nsa_metadata(nsa_mode mode, int B, int R, int W, int n_draft, int topk,
                                   int page_size, const int32_t *seq_lens_dev,
                                   const int32_t *extend_lens_dev, const int32_t *req_to_token_dev,
                                   int64_t req_to_token_ld, int64_t pool_rows,
                                   const int32_t *req_pool_indices_dev, const nsa_metadata_out *out,
                                   int32_t *status_dev, nsa_stream_t stream)
{
    using namespace nsa;
    if (!out || B < 0 || R < 0 || W < 0 || topk < 1 || page_size < 1) return NSA_ERR_INVALID_ARG;
    if (mode != NSA_MODE_DECODE && mode != NSA_MODE_EXTEND && mode != NSA_MODE_TARGET_VERIFY)
        return NSA_ERR_INVALID_ARG;
    if (mode == NSA_MODE_DECODE && R != B) return NSA_ERR_INVALID_ARG;
    if (mode == NSA_MODE_TARGET_VERIFY && (n_draft < 1 || (int64_t)R != (int64_t)B * n_draft))
        return NSA_ERR_INVALID_ARG;
    if (mode == NSA_MODE_EXTEND && B > 0 && !extend_lens_dev) return NSA_ERR_INVALID_ARG;
    if (mode == NSA_MODE_EXTEND && B == 0 && R != 0) return NSA_ERR_INVALID_ARG;
    if (B > 0 && (!seq_lens_dev || !req_to_token_dev || !req_pool_indices_dev)) return NSA_ERR_INVALID_ARG;
    if (B > 0 && (req_to_token_ld < W || pool_rows < 1)) return NSA_ERR_INVALID_ARG;
    // arrays of length >= 1 must exist; per-request / per-row arrays only when non-empty
    if (!out->cu_seqlens_k || !out->cu_seqlens_q || !out->nsa_cu_seqlens_k || !out->nsa_cu_seqlens_q)
        return NSA_ERR_INVALID_ARG;
    if (B > 0 && !out->cache_seqlens) return NSA_ERR_INVALID_ARG;
    if (R > 0 && (!out->seqlens_expanded || !out->nsa_cache_seqlens || !out->row_to_req))
        return NSA_ERR_INVALID_ARG;
    if (B > 0 && W > 0 && !out->real_page_table) return NSA_ERR_INVALID_ARG;
    if ((out->page_table_1 && out->page_table_1_ld < W) || out->real_page_table_ld < ceil_div(W, page_size))
        return NSA_ERR_INVALID_ARG;
    if ((out->indexer_ks == nullptr) != (out->indexer_ke == nullptr)) return NSA_ERR_INVALID_ARG;

    MetaParams p;
    p.mode = mode; p.B = B; p.R = R; p.W = W; p.n_draft = n_draft; p.topk = topk; p.ps = page_size;
    p.seq_lens = seq_lens_dev; p.extend_lens = extend_lens_dev; p.r2t = req_to_token_dev;
    p.rpi = req_pool_indices_dev; p.r2t_ld = req_to_token_ld; p.pool_rows = pool_rows;
    p.out = *out; p.status = status_dev;

    const int sms = current_sm_count();
    if (sms <= 0) return NSA_ERR_CUDA;
    // copy blocks: one per 4096-entry segment of page_table_1, or without it one
    // thread per page id
    const int64_t segs = out->page_table_1 ? (int64_t)B * ceil_div(W, kSeg)
                                           : ceil_div((int64_t)B * ceil_div(W, page_size), kRowThreads);
    int64_t copy_blocks = segs;
    if (copy_blocks > (int64_t)sms * 4) copy_blocks = (int64_t)sms * 4;
    if (copy_blocks < 1) copy_blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(1 + copy_blocks));
    cfg.blockDim = dim3(kRowThreads);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    NSA_CUDA_TRY(cudaLaunchKernelEx(&cfg, metadata_kernel, p));
    return NSA_OK;
}

namespace nsa {
namespace {

// out[kv_start[b] + t] = page_table_1[b, t] for t < kv_len[b]: 4096-entry segments
// of each request spread over the blocks.
__global__ void __launch_bounds__(256)
flatten_page_table_kernel(int B, const int32_t *pt, int64_t pt_ld, const int32_t *kv_len, const int32_t *kv_start,
                          int32_t *out, int64_t out_len, int segs_per_row, int32_t *status)
{
    const int64_t total = (int64_t)B * segs_per_row;
    for (int64_t g = blockIdx.x; g < total; g += gridDim.x) {
        const int b = (int)(g / segs_per_row);
        const int t0 = (int)(g - (int64_t)b * segs_per_row) * kSeg;
        const int L = kv_len[b];
        const int64_t start = kv_start[b];
        if (L < 0 || L > pt_ld || start < 0 || start + L > out_len) {
            if (threadIdx.x == 0 && t0 == 0) set_status(status, NSA_ERR_BOUNDS);
            continue;
        }
        const int t1 = min(L, t0 + kSeg);
        for (int t = t0 + (int)threadIdx.x; t < t1; t += blockDim.x) out[start + t] = pt[(int64_t)b * pt_ld + t];
    }
}

}  // namespace
}  // namespace nsa

extern "C" nsa_status nsa_flatten_page_table(int B, const int32_t *page_table_1_dev, int64_t pt_ld,
                                             const int32_t *kv_len_dev, const int32_t *kv_start_dev,
                                             int32_t *out_dev, int64_t out_len, int32_t *status_dev,
                                             nsa_stream_t stream)
{
    using namespace nsa;
    if (B < 0 || pt_ld < 0 || out_len < 0) return NSA_ERR_INVALID_ARG;
    if (B == 0 || pt_ld == 0) return NSA_OK;
    if (!page_table_1_dev || !kv_len_dev || !kv_start_dev || (!out_dev && out_len > 0)) return NSA_ERR_INVALID_ARG;
    const int segs = (int)ceil_div(pt_ld, kSeg);
    const int sms = current_sm_count();
    if (sms <= 0) return NSA_ERR_CUDA;
    int64_t blocks = (int64_t)B * segs;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    flatten_page_table_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
        B, page_table_1_dev, pt_ld, kv_len_dev, kv_start_dev, out_dev, out_len, segs, status_dev);
    return launch_status();
}
