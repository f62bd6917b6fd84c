// Chunk-local dense attention over the local virtual batches.
//
// [FA3-diff] FlashAttentionBackend, local attention: after
// make_local_attention_virtual_batches, virtual batch b holds the queries
// cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and the first seqused_k[b] keys of one
// attention chunk, reached through its local block table.  The queries sit at
// the end of the keys and attend causally: query i of n_q sees keys
// j <= seqused_k[b] - n_q + i.  Query head h reads key/value head h / G,
// G = Hq / Hkv.  out = softmax(sm_scale q.k) v; lse = ln sum_j exp(sm_scale q.k_j).
//
// Design.  One query token and one key/value head per CTA, its G query heads
// as the 16 rows (zero-padded) of warp-level bf16 tensor-core MMAs
// (mma.sync m16n8k16, fp32 accumulate):
//   S  = Q K^T  per 16-key tile: 2 n-tiles x D/16 k-steps, K rows as the B operand
//   O += P V    per 16-key tile: D/8 n-tiles, P (bf16) taken straight from S's
//               accumulator layout, V read transposed by ldmatrix.trans.
// Each warp runs its own pipeline of 16-key tiles: its lanes copy the tile's
// K and V rows (D*2 bytes each, found through the block table) into padded
// shared-memory rows with 16-byte asynchronous copies, kLaStages tiles ahead
// of the one it computes (one commit group per tile).  Warps take the tiles round robin and keep their own online-softmax
// state (running max per head, refreshed lazily: only when a tile's max passes
// it by more than 2^8); at the end the warps' states are merged in shared
// memory and the CTAs of a cluster -- which split one query's keys -- merge
// theirs through distributed shared memory.  With one query per chunk (decode)
// every K / V row is read from HBM once; the kernel is bound by HBM.
#include "nsa_internal.cuh"
#include "sm100.cuh"

namespace nsa {
namespace {

using namespace sm100;

constexpr int kLaWarps = 4;       // warps per CTA
constexpr int kLaThreads = 32 * kLaWarps;
constexpr int kLaStages = 3;      // tiles in flight per warp
constexpr int kLaTile = 16;       // keys per tile
constexpr int kLaMaxSplit = 8;    // CTAs of a cluster splitting one query's keys
constexpr int kLaRows = 16;       // MMA rows: query heads, zero-padded
constexpr int kLaSplitTarget = 4;   // CTAs per SM the key split aims for

template <int D>
struct LaCfg {
    static constexpr int kRowBytes = D * 2;
    // 16 bytes of padding per row: eight consecutive rows start in eight
    // different 16-byte bank groups, so every ldmatrix phase is conflict free.
    static constexpr int kPitch = kRowBytes + 16;
    static constexpr int kStageBytes = 2 * kLaTile * kPitch;  // 16 K rows, then 16 V rows
    static constexpr int kPipeBytes = kLaWarps * kLaStages * kStageBytes;
    // merge area, aliasing the pipelines once they are drained: per warp and
    // for the CTA, O[16][D] (unnormalised), m[16] (log2 units), l[16]
    static constexpr int kStateFloats = kLaRows * D + 2 * kLaRows;
    static constexpr int kMergeBytes = (kLaWarps + 1) * kStateFloats * 4;
    static constexpr int kDataBytes = kPipeBytes > kMergeBytes ? kPipeBytes : kMergeBytes;
    static constexpr int kSmemBytes = kDataBytes;
};
static_assert(LaCfg<128>::kPitch % 128 == 16 && LaCfg<64>::kPitch % 128 == 16, "conflict-free row pitch");
static_assert(2 * (LaCfg<128>::kSmemBytes + 1024) <= 232448, "two CTAs per SM");

struct LaParams {
    const uint16_t *q;             // [total_q][q_ld] bf16: head h at h*D
    int64_t q_ld;
    const uint16_t *k_cache, *v_cache;  // [num_pages][ps][Hkv][D] bf16
    int64_t num_pages;
    int ps, Hq, Hkv, G;
    const int32_t *block_table;
    int64_t bt_ld;
    const int32_t *cu_seqlens_q, *seqused_k;
    int nvb, nsplit, total_q;
    float scale_log2;
    uint16_t *out;                 // [total_q][Hq][D] bf16
    float *lse;                    // [total_q][Hq]
    int32_t *status;
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&d)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&d)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// The virtual batch holding query token t: the largest b < nvb with
// cu[b] <= t, found by the whole CTA -- each round every thread tests one of
// up to kLaThreads evenly spaced candidates, so decode batches (nvb <= 128)
// take a single round of loads.
__device__ __forceinline__ int block_batch_of(const int32_t *cu, int nvb, int t)
{
    int lo = 0, n = nvb;  // the answer lies in [lo, lo + n); cu[lo] <= t
    while (n > kLaThreads) {
        const int stride = (n + kLaThreads - 1) / kLaThreads;
        const int i = (int)threadIdx.x * stride;
        const int c = __syncthreads_count(i < n && cu[lo + i] <= t);
        lo += (c - 1) * stride;
        n = min(stride, n - (c - 1) * stride);
    }
    const int c = __syncthreads_count((int)threadIdx.x < n && cu[lo + threadIdx.x] <= t);
    return lo + max(c, 1) - 1;
}

template <int D>
__global__ void __launch_bounds__(kLaThreads, 2) local_attention_kernel(LaParams p)
{
    using C = LaCfg<D>;
    constexpr int kNt = D / 8;    // O n-tiles
    constexpr int kKs = D / 16;   // S k-steps
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float cl_m[kLaMaxSplit][kLaRows], cl_l[kLaMaxSplit][kLaRows];
    __shared__ float wts[kLaMaxSplit][kLaRows];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;  // MMA fragment row group and column pair
    const int rank = (int)cluster_ctarank();
    // CTA order: split fastest (the cluster), then query token, then key/value
    // head (measured a little faster than keeping a token's heads together)
    const int pair = (int)(blockIdx.x / (unsigned)p.nsplit);
    const int hk = pair / p.total_q, t = pair - hk * p.total_q;
    const int b = block_batch_of(p.cu_seqlens_q, p.nvb, t);
    const int q0 = p.cu_seqlens_q[b], q1 = p.cu_seqlens_q[b + 1];
    int nk = p.seqused_k[b];
    // A batch whose key count its block-table row cannot hold, or whose query rows do
    // not contain t, is reported and treated as having no keys: every table read below
    // then stays inside the row.
    if (nk < 0 || (int64_t)nk > p.bt_ld * p.ps || t < q0 || t >= q1) {
        if (threadIdx.x == 0) set_status(p.status, NSA_ERR_BOUNDS);
        nk = 0;
    }
    const int nq = q1 - q0;
    const int visible = max(0, min(nk, nk - nq + (t - q0) + 1));  // keys 0 .. visible-1

    // this CTA's tiles of the query's keys, then this warp's (round robin)
    const int T = (visible + kLaTile - 1) / kLaTile;
    const int per = (T + p.nsplit - 1) / p.nsplit;
    const int tile0 = min(T, rank * per), tile1 = min(T, tile0 + per);
    const int kend = min(visible, tile1 * kLaTile);
    const int n_mine = tile1 - tile0 > warp ? (tile1 - tile0 - warp + kLaWarps - 1) / kLaWarps : 0;

    uint8_t *stages = smem + warp * kLaStages * C::kStageBytes;

    const int32_t *bt = p.block_table + (int64_t)b * p.bt_ld;
    const int64_t row_stride = (int64_t)p.Hkv * D;
    // A tile's copy: the 16 K rows then the 16 V rows of its keys, 16 bytes a
    // lane per instruction (kCpr lanes a row, kRpi rows an instruction).  Lane
    // l < 16 looks up the page of the tile's key l; the others get it by shuffle.
    constexpr int kCpr = C::kRowBytes / 16, kRpi = 32 / kCpr;
    auto issue = [&](int n) {
        const int s = n % kLaStages;
        const int key = min(tile0 * kLaTile + (warp + n * kLaWarps) * kLaTile + (lane & 15), kend - 1);
        int32_t page = bt[key / p.ps];
        if (page < 0 || page >= p.num_pages) {
            set_status(p.status, NSA_ERR_BOUNDS);
            page = 0;  // read a real row; the status reports the result invalid
        }
        const int64_t rowoff = ((int64_t)page * p.ps + key % p.ps) * row_stride + (int64_t)hk * D;
        uint8_t *dst = stages + s * C::kStageBytes + (lane % kCpr) * 16;
#pragma unroll
        for (int j = 0; j < kLaTile / kRpi; ++j) {
            const int r = j * kRpi + lane / kCpr;  // key of the tile
            const int64_t off = __shfl_sync(0xffffffffu, rowoff, r) + (lane % kCpr) * 8;
            cp_async16(dst + r * C::kPitch, p.k_cache + off);
            cp_async16(dst + (kLaTile + r) * C::kPitch, p.v_cache + off);
        }
    };

    float o[kNt][4];
#pragma unroll
    for (int u = 0; u < kNt; ++u) o[u][0] = o[u][1] = o[u][2] = o[u][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

    // one commit group per tile slot, empty ones included, so that before tile n
    // is read exactly kLaStages - 1 newer groups may still be in flight
    int issued = 0;
    for (; issued < kLaStages; ++issued) {
        if (issued < n_mine) issue(issued);
        cp_async_commit();
    }

    // Q as the MMA A operand: rows g and g+8 are heads hk*G+g and hk*G+g+8
    // (zero beyond G); a k-step covers 16 dims.
    uint32_t qa[kKs][4];
    {
        const uint16_t *q0 = p.q + (int64_t)t * p.q_ld + (int64_t)hk * p.G * D;
        const bool lo_ok = g < p.G, hi_ok = g + 8 < p.G;
#pragma unroll
        for (int k = 0; k < kKs; ++k) {
            const int d0 = 16 * k + 2 * tq;
            qa[k][0] = lo_ok ? *reinterpret_cast<const uint32_t *>(q0 + (int64_t)g * D + d0) : 0u;
            qa[k][1] = hi_ok ? *reinterpret_cast<const uint32_t *>(q0 + (int64_t)(g + 8) * D + d0) : 0u;
            qa[k][2] = lo_ok ? *reinterpret_cast<const uint32_t *>(q0 + (int64_t)g * D + d0 + 8) : 0u;
            qa[k][3] = hi_ok ? *reinterpret_cast<const uint32_t *>(q0 + (int64_t)(g + 8) * D + d0 + 8) : 0u;
        }
    }

    // ldmatrix lane addresses within a stage: matrix lane>>3, row lane&7
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t kaddr0 = smem_u32(stages) + (8 * (mi >> 1) + rr) * C::kPitch + (mi & 1) * 16;
    const uint32_t vaddr0 = smem_u32(stages) + (kLaTile + 8 * (mi & 1) + rr) * C::kPitch + (mi >> 1) * 16;

    for (int done = 0; done < n_mine; ++done) {
        const int s = done % kLaStages;
        cp_async_wait_group<kLaStages - 1>();
        __syncwarp();  // every lane's part of the tile has landed
        const uint32_t st_off = s * C::kStageBytes;
        // S = Q K^T over the tile's 16 keys (two n-tiles of 8)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int k = 0; k < kKs; ++k) {
            uint32_t kb[4];
            ldmatrix_x4(kaddr0 + st_off + k * 32, kb);
            mma_bf16_16816(sc[0], qa[k], kb[0], kb[1]);
            mma_bf16_16816(sc[1], qa[k], kb[2], kb[3]);
        }
        // online softmax in log2 units; keys at or past kend are masked
        const int key0 = tile0 * kLaTile + (warp + done * kLaWarps) * kLaTile;
        float mt_lo = -INFINITY, mt_hi = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + 8 * nt + 2 * tq + (e & 1);
                const float v = key < kend ? sc[nt][e] * p.scale_log2 : -INFINITY;
                sc[nt][e] = v;
                if (e < 2) mt_lo = fmaxf(mt_lo, v); else mt_hi = fmaxf(mt_hi, v);
            }
        mt_lo = fmaxf(mt_lo, __shfl_xor_sync(0xffffffffu, mt_lo, 1));
        mt_lo = fmaxf(mt_lo, __shfl_xor_sync(0xffffffffu, mt_lo, 2));
        mt_hi = fmaxf(mt_hi, __shfl_xor_sync(0xffffffffu, mt_hi, 1));
        mt_hi = fmaxf(mt_hi, __shfl_xor_sync(0xffffffffu, mt_hi, 2));
        if (mt_lo > m_lo + 8.f) {
            const float f = exp2f(m_lo - mt_lo);
            m_lo = mt_lo;
            l_lo *= f;
#pragma unroll
            for (int u = 0; u < kNt; ++u) { o[u][0] *= f; o[u][1] *= f; }
        }
        if (mt_hi > m_hi + 8.f) {
            const float f = exp2f(m_hi - mt_hi);
            m_hi = mt_hi;
            l_hi *= f;
#pragma unroll
            for (int u = 0; u < kNt; ++u) { o[u][2] *= f; o[u][3] *= f; }
        }
        uint32_t pa[4];
        {
            float pr[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                pr[nt][0] = exp2f(sc[nt][0] - m_lo);
                pr[nt][1] = exp2f(sc[nt][1] - m_lo);
                pr[nt][2] = exp2f(sc[nt][2] - m_hi);
                pr[nt][3] = exp2f(sc[nt][3] - m_hi);
                l_lo += pr[nt][0] + pr[nt][1];
                l_hi += pr[nt][2] + pr[nt][3];
            }
            pa[0] = pack_bf16(pr[0][0], pr[0][1]);
            pa[1] = pack_bf16(pr[0][2], pr[0][3]);
            pa[2] = pack_bf16(pr[1][0], pr[1][1]);
            pa[3] = pack_bf16(pr[1][2], pr[1][3]);
        }
        // O += P V: V^T fragments by transposing ldmatrix, two n-tiles per load
#pragma unroll
        for (int u = 0; u < kNt; u += 2) {
            uint32_t vb[4];
            ldmatrix_x4_trans(vaddr0 + st_off + u * 16, vb);
            mma_bf16_16816(o[u], pa, vb[0], vb[1]);
            mma_bf16_16816(o[u + 1], pa, vb[2], vb[3]);
        }
        __syncwarp();  // the stage is read out before it is refilled
        if (issued < n_mine) issue(issued);
        cp_async_commit();
        ++issued;
    }
    cp_async_wait_all();
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);

    // ---- merge: warps -> CTA (shared memory), CTAs of the cluster -> output
    __syncthreads();  // every warp's pipeline is drained; the merge area aliases it
    float *ms = reinterpret_cast<float *>(smem);
    {
        float *st = ms + warp * C::kStateFloats;
#pragma unroll
        for (int u = 0; u < kNt; ++u) {
            *reinterpret_cast<float2 *>(st + g * D + 8 * u + 2 * tq) = make_float2(o[u][0], o[u][1]);
            *reinterpret_cast<float2 *>(st + (g + 8) * D + 8 * u + 2 * tq) = make_float2(o[u][2], o[u][3]);
        }
        if (tq == 0) {
            st[kLaRows * D + g] = m_lo;
            st[kLaRows * D + g + 8] = m_hi;
            st[kLaRows * D + kLaRows + g] = l_lo;
            st[kLaRows * D + kLaRows + g + 8] = l_hi;
        }
    }
    __syncthreads();
    float *cta = ms + kLaWarps * C::kStateFloats;  // this CTA's merged state
    for (int x = threadIdx.x; x < p.G * D; x += kLaThreads) {
        const int r = x / D, d = x - r * D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kLaWarps; ++w) mx = fmaxf(mx, ms[w * C::kStateFloats + kLaRows * D + r]);
        float lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kLaWarps; ++w) {
            const float mw = ms[w * C::kStateFloats + kLaRows * D + r];
            const float a = mw == -INFINITY ? 0.f : exp2f(mw - mx);
            lsum += a * ms[w * C::kStateFloats + kLaRows * D + kLaRows + r];
            acc += a * ms[w * C::kStateFloats + r * D + d];
        }
        cta[r * D + d] = acc;
        if (d == 0) {
            cta[kLaRows * D + r] = mx;
            cta[kLaRows * D + kLaRows + r] = lsum;
        }
    }
    cluster_sync_all();  // every CTA of the cluster has its merged state
    const int ns = p.nsplit;
    if ((int)threadIdx.x < ns * p.G) {
        const int q = threadIdx.x / p.G, r = threadIdx.x - q * p.G;
        cl_m[q][r] = dsmem_ld_f32(cta + kLaRows * D + r, (uint32_t)q);
        cl_l[q][r] = dsmem_ld_f32(cta + kLaRows * D + kLaRows + r, (uint32_t)q);
    }
    __syncthreads();
    if ((int)threadIdx.x < p.G) {
        const int r = threadIdx.x;
        float mx = -INFINITY;
        for (int q = 0; q < ns; ++q) mx = fmaxf(mx, cl_m[q][r]);
        float lsum = 0.f;
        for (int q = 0; q < ns; ++q) {
            const float a = cl_m[q][r] == -INFINITY ? 0.f : exp2f(cl_m[q][r] - mx);
            wts[q][r] = a;
            lsum += a * cl_l[q][r];
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        for (int q = 0; q < ns; ++q) wts[q][r] *= inv;
        if (rank == 0)
            p.lse[(int64_t)t * p.Hq + hk * p.G + r] =
                lsum > 0.f ? (mx + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    {
        const int per_rank = p.G * D / ns;
        for (int x = rank * per_rank + (int)threadIdx.x; x < (rank + 1) * per_rank; x += kLaThreads) {
            const int r = x / D, d = x - r * D;
            float acc = 0.f;
            for (int q = 0; q < ns; ++q) acc += wts[q][r] * dsmem_ld_f32(cta + r * D + d, (uint32_t)q);
            const __nv_bfloat16 ob = __float2bfloat16_rn(acc);
            p.out[((int64_t)t * p.Hq + hk * p.G + r) * D + d] = *reinterpret_cast<const uint16_t *>(&ob);
        }
    }
    cluster_sync_all();  // peers' shared memory stays alive until every read is done
}

template <int D>
bool cluster_fits(int ns)
{
    constexpr int kMaxDev = 64;
    static int cache[kMaxDev][kLaMaxSplit + 1];  // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return ns == 1;
    int &c = cache[dev][ns];
    if (c == 0) {
        const void *kern = (const void *)local_attention_kernel<D>;
        int n = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ns, 1, 1);
        cfg.blockDim = dim3(kLaThreads);
        cfg.dynamicSmemBytes = LaCfg<D>::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)ns;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             LaCfg<D>::kSmemBytes) == cudaSuccess &&
                        cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1;
        if (!ok) (void)cudaGetLastError();  // a failed query is not the caller's error
        c = ok ? 1 : 2;
    }
    return c == 1;
}

int device_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || n <= 0)
        return 148;
    return n;
}

template <int D>
nsa_status launch(LaParams p, int total_q, cudaStream_t stream)
{
    // Split each query's keys over a cluster of up to 8 CTAs when the grid of
    // (query, key/value head) pairs alone would not give every SM several CTAs.
    const int64_t pairs = (int64_t)total_q * p.Hkv;
    const int64_t want = (int64_t)kLaSplitTarget * device_sms();
    int ns = 1;
    while (ns < kLaMaxSplit && pairs * ns < want) ns *= 2;
    while (ns > 1 && !cluster_fits<D>(ns)) ns /= 2;
    if (pairs * ns > 0x7fffffffLL) return NSA_ERR_UNSUPPORTED;
    p.nsplit = ns;
    NSA_CUDA_TRY(cudaFuncSetAttribute(local_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      LaCfg<D>::kSmemBytes));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(pairs * ns), 1, 1);
    cfg.blockDim = dim3(kLaThreads);
    cfg.dynamicSmemBytes = LaCfg<D>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ns;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    NSA_CUDA_TRY(cudaLaunchKernelEx(&cfg, local_attention_kernel<D>, p));
    return NSA_OK;
}

}  // namespace
}  // namespace nsa

extern "C" nsa_status nsa_local_attention(const void *q_dev, int64_t q_ld, const void *k_cache_dev,
                                          const void *v_cache_dev, int64_t num_pages, int page_size,
                                          const int32_t *block_table_dev, int64_t bt_ld,
                                          const int32_t *cu_seqlens_q_dev, const int32_t *seqused_k_dev, int nvb,
                                          int total_q, int Hq, int Hkv, int D, float sm_scale, void *out_dev,
                                          float *lse_dev, int32_t *status_dev, nsa_stream_t stream)
{
    using namespace nsa;
    if (nvb < 0 || total_q < 0 || Hq < 1 || Hkv < 1 || page_size < 1 || num_pages < 0 || bt_ld < 0)
        return NSA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !(sm_scale > 0.f) || !(sm_scale < INFINITY)) return NSA_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (G > kLaRows || (D != 64 && D != 128)) return NSA_ERR_UNSUPPORTED;
    if (q_ld < (int64_t)Hq * D || q_ld % 2 != 0) return NSA_ERR_INVALID_ARG;
    if (total_q == 0) return NSA_OK;
    if (nvb == 0 || num_pages < 1 || !q_dev || !k_cache_dev || !v_cache_dev || !block_table_dev ||
        !cu_seqlens_q_dev || !seqused_k_dev || !out_dev || !lse_dev)
        return NSA_ERR_INVALID_ARG;
    // rows move in aligned 16-byte pieces; Q is read as bf16 pairs
    if (((uintptr_t)k_cache_dev | (uintptr_t)v_cache_dev) % 16 != 0 || (uintptr_t)q_dev % 4 != 0 ||
        (uintptr_t)lse_dev % 4 != 0 || (uintptr_t)out_dev % 2 != 0)
        return NSA_ERR_INVALID_ARG;
    LaParams p;
    p.q = (const uint16_t *)q_dev;
    p.q_ld = q_ld;
    p.k_cache = (const uint16_t *)k_cache_dev;
    p.v_cache = (const uint16_t *)v_cache_dev;
    p.num_pages = num_pages;
    p.ps = page_size;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = G;
    p.block_table = block_table_dev;
    p.bt_ld = bt_ld;
    p.cu_seqlens_q = cu_seqlens_q_dev;
    p.seqused_k = seqused_k_dev;
    p.nvb = nvb;
    p.nsplit = 1;
    p.total_q = total_q;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.out = (uint16_t *)out_dev;
    p.lse = lse_dev;
    p.status = status_dev;
    const cudaStream_t s = (cudaStream_t)stream;
    return D == 64 ? launch<64>(p, total_q, s) : launch<128>(p, total_q, s);
}
