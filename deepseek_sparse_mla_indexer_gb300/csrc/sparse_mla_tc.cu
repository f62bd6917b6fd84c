// Tensor-core sparse MLA for d_qk = 576 (512 latent + 64 rope), d_v = 512,
// bf16 query, bf16 or fp8 (e4m3 + per-128 fp32 scale + bf16 rope) KV rows.
//
// [DSA] _forward_flashmla_sparse / _forward_flashmla_kv call contract: for
// each query row r and head h, attention over the KV rows listed in
// indices[r, :] (slots of the flat KV view, -1 = none); keys and values share
// the latent (V = first 512 columns of the same row).
//
// One CTA = one query row x 64 heads x one split of the top-k list.  Per tile
// of 128 selected KV rows:
//   1. the loader threads (warps 0, 2..11) copy the 128 rows into shared
//      memory with 16-byte cp.async (fp8 rows: loaded into registers,
//      dequantised to bf16 and stored), laid out as 9 column blocks of 64 bf16,
//      128-byte swizzled, K-major; the five block pairs of a tile are all in
//      flight at once (one commit group each) and each is released to the MMA
//      warp as it lands; the next tile's rows are prefetched into L2;
//   2. warp 1 issues S^T[128 tok, 64 heads] = KV_tile . Q^T on tcgen05 (TMEM);
//   3. warps 4..11 (two groups of 4 warps, 32 heads each; one thread per
//      token) run the online softmax over the token axis: a lazily refreshed
//      running max per head (refreshed only when a score exceeds it by 2^8; the
//      TMEM accumulators are rescaled then), and P^T written as bf16 into the
//      rope block (free once S^T is done) in the MN-major layout;
//   4. warp 1 issues O^T[512 d, 64 heads] += V^T . P^T, reading the latent
//      tile a second time as an MN-major operand (4 blocks of 128 d rows,
//      256 TMEM columns), and the head sums l = ones . P^T.
// At the end the softmax warps normalise O^T by the head sums, stage it in the
// dead KV tile and write it out with 16-byte stores: the bf16 output (one
// split) or fp32 partials plus their log-sum-exp (several splits).  Up to 8
// splits of a (row, head group) form a thread-block cluster; after a cluster
// barrier each CTA merges one slice of the latent dimension from all partials
// (its own from shared memory, the others from L2).  More splits are merged by
// sparse_mla_combine_kernel.  Both merges sum the splits in a fixed order.
#include <cstddef>

#include "sparse_mla_tc.cuh"
#include "sm100.cuh"

namespace nsa {
namespace {

using namespace sm100;

constexpr int kTok = 128;
constexpr int kHc = 64;
constexpr int kDl = 512;
constexpr int kDr = 64;
constexpr int kBlocks = 9;
constexpr uint32_t kQBlk = kHc * 128;
constexpr uint32_t kKvBlk = kTok * 128;
constexpr uint32_t kQBytes = kBlocks * kQBlk;
constexpr uint32_t kKvBytes = kBlocks * kKvBlk;
constexpr int kThreads = 384;
constexpr int kWorkers = 352;         // warps 0, 2..11 load; warps 4..11 also run the softmax
constexpr int kHg = 32;               // heads per softmax group (warps 4..7: heads 0..31, 8..11: 32..63)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColL = 256;   // ones . P^T: every lane holds the running head sums
constexpr uint32_t kColS = 320;   // S^T accumulator
constexpr float kRescale = 8.0f;      // log2 units
constexpr long long kWaitBudget = 2000000000LL;
constexpr int kBf16RowBytes = (kDl + kDr) * 2;        // 1152
constexpr int kFp8RowBytes = kDl + 4 * (kDl / 128) + 2 * kDr;  // 656
constexpr int kMaxClusterSplit = 8;   // portable cluster size
constexpr int kPartRow = kDl + 4;     // floats per split partial row: raw O (512) | lse, l, 0, 0
constexpr int kMergeItems = (kHc * (kDl / 8) + kThreads - 1) / kThreads;  // 16-byte outputs per thread at 2 splits
static_assert(kHc * (kDl / 4 / 2) <= kMergeItems * kThreads, "a merge slice (2 or more splits) fits one pass");
static_assert(kHc * kDl * 4 <= 8 * (int)kKvBlk, "the fp32 partial fits in the latent part of the KV tile");

struct MlaParams {
    const uint8_t *kv;
    const uint16_t *q_nope;
    const uint16_t *q_rope;
    int64_t nope_ld_r, nope_ld_h, rope_ld_r, rope_ld_h;
    const int32_t *indices;
    int64_t indices_ld;
    int R, H, topk, nsplit, tiles_per_split;
    int64_t num_slots;
    float scale_log2;
    __nv_bfloat16 *out;
    float *lse;
    float *o_part;      // [nsplit][R][H][kPartRow]
    int cluster_merge;  // splits merged inside the cluster (cluster y = nsplit, rank = split)
    int32_t *status;
};

struct __align__(16) MlaShared {
    alignas(16) float m_run[kHc];  // running max per head, log2 units (read as float4)
    alignas(16) float alpha[kHc];
    alignas(16) float red[4][kHc];
    alignas(16) float l_head[kHc];    // final head sums of this split
    alignas(16) float lse_head[kHc];  // natural-log LSE of this split per head
    alignas(16) float wts[kMaxClusterSplit][kHc];  // merge weights exp(lse_q - lse) / l_q
    alignas(16) int idx[kTok];
    const uint8_t *rowbase[kTok];  // KV row of each token of the tile (slot 0 for masked ones)
    uint64_t kvb_full[5];          // block pair m of the tile landed (m = 4: rope block)
    uint64_t o_done[5];            // O^T block m of the tile done (m = 4: every MMA of the tile)
    uint64_t q_full, s_full, p_full, done;
    uint32_t tmem_base;
    volatile int abort;
};
static_assert(offsetof(MlaShared, m_run) % 16 == 0, "m_run is read with 16-byte loads");
static_assert(offsetof(MlaShared, kvb_full) % 8 == 0, "mbarriers need 8-byte alignment");
static_assert(1024 + kQBytes + kKvBytes + 1024 + sizeof(MlaShared) <= 232448, "shared memory per CTA");

__device__ __forceinline__ void fail(MlaShared *sm, int32_t *status)
{
    sm->abort = 1;
    set_status(status, NSA_ERR_TIMEOUT);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Eight e4m3 codes (a 64-bit word) times `sc` -> four packed bf16 pairs.
__device__ __forceinline__ void dequant8(uint2 w, float sc, uint32_t *dst4)
{
    const uint32_t words[2] = {w.x, w.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)((words[i] >> (16 * j)) & 0xFFFFu);
            const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
            dst4[2 * i + j] = pack_bf16x2(f.x * sc, f.y * sc);
        }
    }
}

// Float offset of 16-byte chunk c (d = 4c .. 4c+3) of head h in the staged
// accumulator: O^T block m = d / 128 sits in the two latent blocks that block m's
// MMAs read (dead once they complete), heads x 128 d within it.
__device__ __forceinline__ int stage_off(int h, int c) { return (c >> 5) * (kHc * 128) + h * 128 + ((c & 31) << 2); }

// Worker-group barrier (warps 0, 2..11).
__device__ __forceinline__ void worker_sync() { bar_sync(2, kWorkers); }

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_tc_kernel(MlaParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *q_s = base;
    uint8_t *kv_s = base + kQBytes;
    uint8_t *p_s = kv_s + 8 * kKvBlk;  // P^T reuses the rope block
    uint8_t *ones_s = kv_s + kKvBytes;  // 1 KB of bf16 1.0: an all-ones MN-major operand atom
    MlaShared *sm = (MlaShared *)(ones_s + 1024);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hg = blockIdx.x, sp = blockIdx.y, r = blockIdx.z;
    pdl_trigger();
    const int ntiles_all = (p.topk + kTok - 1) / kTok;
    const int t0 = sp * p.tiles_per_split;
    const int nt = max(0, min(t0 + p.tiles_per_split, ntiles_all) - t0);
    const int64_t row_bytes = FP8 ? kFp8RowBytes : kBf16RowBytes;

    if (threadIdx.x == 0) {
        mbar_init(&sm->q_full, kWorkers);
        for (int m = 0; m < 5; ++m) {
            mbar_init(&sm->kvb_full[m], kWorkers);
            mbar_init(&sm->o_done[m], 1);
        }
        mbar_init(&sm->s_full, 1);
        mbar_init(&sm->p_full, 256);
        mbar_init(&sm->done, 1);
        sm->abort = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < 64) reinterpret_cast<uint4 *>(ones_s)[threadIdx.x] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(&sm->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;

    if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        pdl_wait();  // every thread passes the wait before this grid writes global memory
        if (lane == 0) {
            const uint32_t idesc_s = instr_desc(1, 1, 0, 0, kTok, kHc);  // bf16, K-major A and B
            const uint32_t idesc_o = instr_desc(1, 1, 1, 1, 128, kHc);   // bf16, MN-major A and B
            const uint32_t q_addr = smem_u32(q_s), kv_addr = smem_u32(kv_s), p_addr = smem_u32(p_s);
            const uint64_t ones_d = smem_desc(smem_u32(ones_s), 0, 0, kSwizzle128B);
            bool ok = mbar_wait(&sm->q_full, 0, kWaitBudget);
            if (!ok) fail(sm, p.status);
            for (int i = 0; i < nt && ok && !sm->abort; ++i) {
                // S^T = KV (128 x 576) . Q^T (576 x 64), block pair by block pair as they land
#pragma unroll 1
                for (int m = 0; m < 5 && ok; ++m) {
                    if (!mbar_wait(&sm->kvb_full[m], i & 1, kWaitBudget)) { fail(sm, p.status); ok = false; break; }
                    tc_fence_after();
                    const int c0 = m < 4 ? 2 * m : 8, nc = m < 4 ? 2 : 1;
                    for (int c = c0; c < c0 + nc; ++c) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint64_t ad = smem_desc(kv_addr + c * kKvBlk + ks * 32, 16, 1024, kSwizzle128B);
                            const uint64_t bd = smem_desc(q_addr + c * kQBlk + ks * 32, 16, 1024, kSwizzle128B);
                            mma_f16(tmem + kColS, ad, bd, idesc_s, (c | ks) != 0);
                        }
                    }
                }
                if (!ok) break;
                mma_commit(&sm->s_full);
                if (!mbar_wait(&sm->p_full, i & 1, kWaitBudget)) { fail(sm, p.status); break; }
                tc_fence_after();
                // O^T[d, h] += sum_t V[t, d] P[t, h]: A = V^T (MN-major), B = P^T (MN-major);
                // each finished block pair goes back to the loaders at once
#pragma unroll 1
                for (int m = 0; m < 4; ++m) {
#pragma unroll
                    for (int k = 0; k < kTok / 16; ++k) {
                        const uint64_t ad =
                            smem_desc(kv_addr + 2 * m * kKvBlk + k * 2048, kKvBlk, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(p_addr + k * 2048, kKvBlk, 1024, kSwizzle128B);
                        mma_f16(tmem + m * kHc, ad, bd, idesc_o, (i > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(&sm->o_done[m]);
                }
                // head sums l[h] = sum_t P[t, h] in every lane: A = all-ones (one atom, zero strides)
#pragma unroll
                for (int k = 0; k < kTok / 16; ++k) {
                    const uint64_t bd = smem_desc(p_addr + k * 2048, kKvBlk, 1024, kSwizzle128B);
                    mma_f16(tmem + kColL, ones_d, bd, idesc_o, (i > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&sm->o_done[4]);
            }
            mma_commit(&sm->done);
            mbar_wait(&sm->done, 0, kWaitBudget);
        }
    } else {
        // ---------------------------------------------------------------- workers
        // Warps 0, 2, 3 and the softmax warps 4..11 all load the KV tiles; warps
        // 4..11 also run the softmax and the epilogue, in two groups of four
        // warps that own 32 heads each.
        const int lid = (warp == 0 ? 0 : warp - 1) * 32 + lane;  // 0 .. 351
        const bool softmax_warp = warp >= 4;
        // Q of this head group: 64 heads x (64 latent + 8 rope) 16-byte chunks; its
        // commit group is the oldest, so it completes under the first tile's loads
        for (int q = lid; q < kHc * 72; q += kWorkers) {
            const int h = q / 72, c = q - h * 72;
            uint8_t *dst = q_s + (c >> 3) * kQBlk + sw128_offset(h, c & 7);
            const int hh = hg * kHc + h;
            if (hh < p.H) {
                const uint16_t *src = c < 64 ? p.q_nope + r * p.nope_ld_r + hh * p.nope_ld_h + c * 8
                                             : p.q_rope + r * p.rope_ld_r + hh * p.rope_ld_h + (c - 64) * 8;
                cp_async16(dst, src);
            } else {
                *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);  // padded head
            }
        }
        cp_async_commit();
        pdl_wait();  // the indices come from the top-k kernel (q and the KV cache do not)
        auto release_q = [&]() {
            fence_proxy_async_smem();
            mbar_arrive(&sm->q_full);
        };
        if (nt == 0) {
            cp_async_wait_all();
            release_q();
        }

        const int32_t *irow = p.indices + (int64_t)r * p.indices_ld;
        // the index of token j of a tile is read one tile ahead by worker j
        auto fetch_idx = [&](int tile) -> int {
            const int pos = tile * kTok + lid;
            return (lid < kTok && tile < t0 + nt && pos < p.topk) ? __ldg(irow + pos) : -1;
        };
        // Block pair m of the tile (latent blocks 2m, 2m+1 for m < 4; the rope block for m = 4) by cp.async
        auto issue_pair = [&](int m) {
            if (m == 4) {
                for (int q = lid; q < kTok * 8; q += kWorkers) {
                    const int row = q >> 3, c = q & 7;
                    cp_async16(kv_s + 8 * kKvBlk + sw128_offset(row, c),
                               sm->rowbase[row] + (FP8 ? kDl + 16 : 2 * kDl) + c * 16);
                }
            } else {
                for (int q = lid; q < kTok * 16; q += kWorkers) {
                    const int row = q >> 4, c = 16 * m + (q & 15);
                    cp_async16(kv_s + (c >> 3) * kKvBlk + sw128_offset(row, c & 7), sm->rowbase[row] + c * 16);
                }
            }
        };
        auto release_pair = [&](int m) {
            fence_proxy_async_smem();
            mbar_arrive(&sm->kvb_full[m]);
        };
        // fp8 rows: each worker dequantises up to kF8Items groups of 16 e4m3 codes per latent block pair
        constexpr int kF8Items = (kTok * 8 + kWorkers - 1) / kWorkers;
        // softmax state: group g (warps 4+4g .. 7+4g) owns heads hb .. hb+31
        const int grp = softmax_warp ? (warp - 4) >> 2 : 0;
        const int hb = grp * kHg;
        const int gbar = grp == 0 ? 1 : 3;                 // named barrier of the group
        const float4 *m_run4 = reinterpret_cast<const float4 *>(sm->m_run + hb);
        const int quad = warp & 3;
        const int t = quad * 32 + lane;  // token row of S^T; d row of each O^T block
        const int et = (threadIdx.x - 128) & 127;           // thread index inside the group
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        if (softmax_warp) {
            if (et < kHg) sm->m_run[hb + et] = -INFINITY;
            bar_sync(gbar, 128);
        }
        int done_tiles = 0;
        int cur = fetch_idx(t0);
        for (int i = 0; i < nt; ++i) {
            // block pair 0 (and the token table) is free once the previous tile's O^T block 0 is done
            if (i > 0 && !mbar_wait(&sm->o_done[0], (i - 1) & 1, kWaitBudget)) fail(sm, p.status);
            if (bar_red_or(2, kWorkers, sm->abort != 0)) break;  // uniform over the workers
            if (lid < kTok) {
                int v = cur;
                if (v < -1 || v >= p.num_slots) {
                    set_status(p.status, NSA_ERR_BOUNDS);
                    v = -1;
                }
                sm->idx[lid] = v;
                sm->rowbase[lid] = p.kv + (int64_t)(v < 0 ? 0 : v) * row_bytes;  // masked rows read slot 0
            }
            const int nxt = fetch_idx(t0 + i + 1);
            worker_sync();
            if (!FP8) {
                // two block pairs in flight per thread: pair m is issued, then pair m-1 (tile 0:
                // first the Q rows) is awaited and released to the MMA warp
#pragma unroll 1
                for (int m = 0; m < 5; ++m) {
                    if (m > 0 && i > 0 && !mbar_wait(&sm->o_done[m], (i - 1) & 1, kWaitBudget)) fail(sm, p.status);
                    issue_pair(m);
                    cp_async_commit();
                    if (m == 0 && i == 0) {
                        cp_async_wait_group<1>();
                        release_q();
                    } else if (m > 0) {
                        cp_async_wait_group<1>();
                        release_pair(m - 1);
                    }
                }
                if (nxt >= 0 && nxt < p.num_slots) prefetch_l2_bulk(p.kv + (int64_t)nxt * row_bytes, (uint32_t)row_bytes);
                cp_async_wait_group<0>();
                release_pair(4);
            } else {
                // latent codes (16 a load) and the four block scales of each row (one 16-byte
                // load) of the whole tile go into registers first; the rope rows (bf16) go by
                // cp.async. Item q: row q / 8, codes 16k .. 16k+15 (k = q % 8) of a block pair,
                // which expand to the pair's chunks 2k, 2k+1; threads k >= 4 store the odd chunk
                // first, so that eight neighbouring threads store to eight distinct bank groups.
                uint4 w[4][kF8Items];
                float4 sc4[kF8Items];
#pragma unroll
                for (int u = 0; u < kF8Items; ++u) {
                    const int q = lid + u * kWorkers;
                    sc4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int m = 0; m < 4; ++m) w[m][u] = make_uint4(0u, 0u, 0u, 0u);
                    if (q < kTok * 8) {
                        const uint8_t *rowp = sm->rowbase[q >> 3];
                        sc4[u] = __ldg(reinterpret_cast<const float4 *>(rowp + kDl));
#pragma unroll
                        for (int m = 0; m < 4; ++m)
                            w[m][u] = __ldg(reinterpret_cast<const uint4 *>(rowp + 128 * m + 16 * (q & 7)));
                    }
                }
                if (nxt >= 0 && nxt < p.num_slots) prefetch_l2_bulk(p.kv + (int64_t)nxt * row_bytes, (uint32_t)row_bytes);
                if (i == 0) {
                    cp_async_wait_group<0>();  // the Q rows (the only group in flight)
                    release_q();
                }
                // latent pairs first, each as soon as the previous tile's O^T block that reads
                // its buffer is done; the rope rows last (their block holds P^T until every O^T
                // block of the previous tile is done)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    if (m > 0 && i > 0 && !mbar_wait(&sm->o_done[m], (i - 1) & 1, kWaitBudget)) fail(sm, p.status);
#pragma unroll
                    for (int u = 0; u < kF8Items; ++u) {
                        const int q = lid + u * kWorkers;
                        if (q < kTok * 8) {
                            const int row = q >> 3, k = q & 7;
                            const float sc = m == 0 ? sc4[u].x : m == 1 ? sc4[u].y : m == 2 ? sc4[u].z : sc4[u].w;
                            uint32_t lo[4], hi[4];
                            dequant8(make_uint2(w[m][u].x, w[m][u].y), sc, lo);
                            dequant8(make_uint2(w[m][u].z, w[m][u].w), sc, hi);
                            uint8_t *blk = kv_s + (2 * m + (k >> 2)) * kKvBlk;
                            const int c0 = (2 * k) & 7;  // the pair's chunk 2k inside its block
                            const uint4 v0 = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                            const uint4 v1 = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                            if (k < 4) {
                                *reinterpret_cast<uint4 *>(blk + sw128_offset(row, c0)) = v0;
                                *reinterpret_cast<uint4 *>(blk + sw128_offset(row, c0 + 1)) = v1;
                            } else {
                                *reinterpret_cast<uint4 *>(blk + sw128_offset(row, c0 + 1)) = v1;
                                *reinterpret_cast<uint4 *>(blk + sw128_offset(row, c0)) = v0;
                            }
                        }
                    }
                    release_pair(m);
                }
                if (i > 0 && !mbar_wait(&sm->o_done[4], (i - 1) & 1, kWaitBudget)) fail(sm, p.status);
                issue_pair(4);
                cp_async_commit();
                cp_async_wait_group<0>();
                release_pair(4);
            }
            cur = nxt;
            if (softmax_warp) {
                const bool ok = mbar_wait(&sm->kvb_full[0], i & 1, kWaitBudget) && mbar_wait(&sm->s_full, i & 1, kWaitBudget);
                if (!ok) fail(sm, p.status);
                if (bar_red_or(gbar, 128, !ok || sm->abort)) continue;  // the worker-wide check ends the loop
                tc_fence_after();
                uint32_t sa[32];
                tmem_ld32(lane_base + kColS + hb, sa);
                tmem_ld_wait();
                const bool valid = sm->idx[t] >= 0;
                float s[kHg];
                bool exceed = false;
#pragma unroll
                for (int c = 0; c < kHg / 4; ++c) {
                    const float4 mr = m_run4[c];
                    const float mv[4] = {mr.x, mr.y, mr.z, mr.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int h = 4 * c + j;
                        s[h] = valid ? __uint_as_float(sa[h]) * p.scale_log2 : -INFINITY;
                        exceed |= s[h] > mv[j] + kRescale;
                    }
                }
                if (bar_red_or(gbar, 128, exceed)) {
                    // refresh the running max of the group's heads from this tile's column maxima
#pragma unroll
                    for (int h = 0; h < kHg; ++h) {
                        float v = s[h];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                        if (lane == 0) sm->red[quad][hb + h] = v;
                    }
                    bar_sync(gbar, 128);
                    if (et < kHg) {
                        const int h = hb + et;
                        const float cm = fmaxf(fmaxf(sm->red[0][h], sm->red[1][h]), fmaxf(sm->red[2][h], sm->red[3][h]));
                        const float mo = sm->m_run[h];
                        const float mn = fmaxf(mo, cm);
                        sm->alpha[h] = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
                        sm->m_run[h] = mn;
                    }
                    bar_sync(gbar, 128);  // alpha[] and m_run[] complete; red[] free for the next refresh
                    if (i > 0) {
                        // the previous tile's O^T and head sums must be complete before they are rescaled
                        if (!mbar_wait(&sm->o_done[4], (i - 1) & 1, kWaitBudget)) fail(sm, p.status);
                        tc_fence_after();
#pragma unroll 1
                        for (int m = 0; m < 5; ++m) {  // 4 O^T blocks + the head-sum block, this group's columns
                            uint32_t v[32];
                            const uint32_t a = lane_base + m * kHc + hb;
                            tmem_ld32(a, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                v[j] = __float_as_uint(__uint_as_float(v[j]) * sm->alpha[hb + j]);
                            tmem_st32(a, v);
                        }
                        tmem_st_wait();
                    }
                }
                // probabilities relative to the running max, written into P^T row t (bf16)
#pragma unroll
                for (int c = 0; c < kHg / 8; ++c) {  // heads hb+8c .. hb+8c+7 -> one 16-byte chunk of row t
                    const float4 ma = m_run4[2 * c], mb = m_run4[2 * c + 1];
                    const float mv[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
                    uint32_t pk[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int h = 8 * c + 2 * j;
                        const float p0 = s[h] == -INFINITY ? 0.f : exp2f(s[h] - mv[2 * j]);
                        const float p1 = s[h + 1] == -INFINITY ? 0.f : exp2f(s[h + 1] - mv[2 * j + 1]);
                        pk[j] = pack_bf16x2(p0, p1);
                    }
                    *reinterpret_cast<uint4 *>(p_s + sw128_offset(t, hb / 8 + c)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&sm->p_full);
                done_tiles = i + 1;
            }
        }
        if (softmax_warp) {
            // ------------------------------------------------------------ epilogue
            // each O^T block is staged raw (fp32) in the two latent blocks its MMAs read, as
            // soon as they complete; the head sums arrive last and scale the copy-out or merge
            const int hv = min(kHc, p.H - hg * kHc);  // real heads of this CTA
            const int nh = max(0, min(kHg, hv - hb));  // real heads of this group
            const int64_t row0 = (int64_t)r * p.H + hg * kHc + hb;
            const uint32_t last = (uint32_t)(done_tiles - 1) & 1u;
            bool have_o = done_tiles > 0 && !sm->abort;
            float *stage_f = reinterpret_cast<float *>(kv_s);
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
                if (have_o && !mbar_wait(&sm->o_done[m], last, kWaitBudget)) {
                    fail(sm, p.status);
                    have_o = false;
                }
                tc_fence_after();
                uint32_t v[32];
                if (have_o) {
                    tmem_ld32(lane_base + m * kHc + hb, v);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0u;
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) stage_f[m * (kHc * 128) + (hb + j) * 128 + t] = __uint_as_float(v[j]);
            }
            if (have_o && !mbar_wait(&sm->o_done[4], last, kWaitBudget)) {
                fail(sm, p.status);
                have_o = false;
            }
            tc_fence_after();
            uint32_t la[32];  // head sums of the group's heads (identical in every lane)
            if (have_o) {
                tmem_ld32(lane_base + kColL + hb, la);
                tmem_ld_wait();
            }
            if (et < kHg) {
                float l = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j == et) l = have_o ? __uint_as_float(la[j]) : 0.f;
                const float lse = l > 0.f ? (sm->m_run[hb + et] + log2f(l)) * 0.69314718055994531f : -INFINITY;
                sm->l_head[hb + et] = l;
                sm->lse_head[hb + et] = lse;
                if (hb + et < hv) {
                    if (p.nsplit == 1)
                        p.lse[row0 + et] = lse;
                    else
                        *reinterpret_cast<float4 *>(p.o_part + ((int64_t)sp * p.R * p.H + row0 + et) * kPartRow + kDl) =
                            make_float4(lse, l, 0.f, 0.f);
                }
            }
            bar_sync(gbar, 128);  // the group's staged rows and head sums are complete
            if (p.nsplit == 1) {
                // the group's heads are contiguous in global memory: normalised 8-byte chunks out
                uint2 *dst = reinterpret_cast<uint2 *>(p.out + row0 * kDl);
                for (int k = et; k < nh * (kDl / 4); k += 128) {
                    const int h = hb + k / (kDl / 4);
                    const float l = sm->l_head[h];
                    const float il = l > 0.f ? 1.f / l : 0.f;
                    const float4 v = *reinterpret_cast<const float4 *>(stage_f + stage_off(h, k & (kDl / 4 - 1)));
                    dst[k] = make_uint2(pack_bf16x2(v.x * il, v.y * il), pack_bf16x2(v.z * il, v.w * il));
                }
            } else {
                // raw partial rows out; in a cluster merge only the slices the other splits merge
                const int ns = p.nsplit;
                const int s0 = p.cluster_merge ? sp * (kDl / 4) / ns : 0;
                const int s1 = p.cluster_merge ? (sp + 1) * (kDl / 4) / ns : 0;
                float *dst = p.o_part + ((int64_t)sp * p.R * p.H + row0) * kPartRow;
                for (int k = et; k < nh * (kDl / 4); k += 128) {
                    const int hl = k / (kDl / 4), c = k & (kDl / 4 - 1);
                    if (c < s0 || c >= s1)
                        *reinterpret_cast<float4 *>(dst + hl * kPartRow + 4 * c) =
                            *reinterpret_cast<const float4 *>(stage_f + stage_off(hb + hl, c));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }

    if (p.cluster_merge) {
        // ---------------------------------------------------------------- split merge
        // out = sum_q exp(lse_q - lse) O_q / l_q, lse = ln sum_q exp(lse_q), with O_q the raw
        // accumulator and l_q the head sums of split q.  The splits of this (row, head group)
        // are the CTAs of the cluster (rank = split); each merges one slice of the latent
        // dimension: its own accumulator from shared memory, the other splits' partial rows
        // from L2 (all loads of one split in flight at once), summed in split order.
        cluster_sync_all();  // every split's partial rows are in global memory
        const int ns = p.nsplit;
        const int hv = min(kHc, p.H - hg * kHc);
        const int64_t hrow0 = (int64_t)r * p.H + hg * kHc;
        const float *stage_f = reinterpret_cast<const float *>(kv_s);
        // this CTA's slice of the latent dimension, in 16-byte chunks, for every real head
        // (at most 64 heads x 64 chunks: one pass of kMergeItems per thread)
        const int c0 = sp * (kDl / 4) / ns, c1 = (sp + 1) * (kDl / 4) / ns, nc = c1 - c0;
        const int items = hv * nc;
        const int kcount = min(kMergeItems, (items - (int)threadIdx.x + kThreads - 1) / kThreads);
        int hh[kMergeItems], cc[kMergeItems];
#pragma unroll
        for (int k = 0; k < kMergeItems; ++k) {
            const int e = min(k * kThreads + (int)threadIdx.x, items - 1);  // clamped: a valid address
            hh[k] = e / nc;
            cc[k] = c0 + e - hh[k] * nc;
        }
        // the first other split's partial rows are in flight while the weights are formed
        const int q0 = sp == 0 ? 1 : 0;
        float4 v0[kMergeItems];
        {
            const float *rowq = p.o_part + ((int64_t)q0 * p.R * p.H + hrow0) * kPartRow;
#pragma unroll
            for (int k = 0; k < kMergeItems; ++k)
                if (k < kcount) v0[k] = __ldcg(reinterpret_cast<const float4 *>(rowq + hh[k] * kPartRow + 4 * cc[k]));
        }
        if (threadIdx.x < kHc) {
            const int h = threadIdx.x;
            float ls[kMaxClusterSplit], l[kMaxClusterSplit];
#pragma unroll
            for (int q = 0; q < kMaxClusterSplit; ++q) {
                ls[q] = -INFINITY;
                l[q] = 0.f;
                if (q < ns && h < hv) {
                    if (q == sp) {
                        ls[q] = sm->lse_head[h];
                        l[q] = sm->l_head[h];
                    } else {
                        const float2 hd = __ldcg(reinterpret_cast<const float2 *>(
                            p.o_part + ((int64_t)q * p.R * p.H + hrow0 + h) * kPartRow + kDl));
                        ls[q] = hd.x;
                        l[q] = hd.y;
                    }
                }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int q = 0; q < kMaxClusterSplit; ++q) mx = fmaxf(mx, ls[q]);
            float wsum = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxClusterSplit; ++q)
                if (mx != -INFINITY && ls[q] != -INFINITY) wsum += __expf(ls[q] - mx);
#pragma unroll
            for (int q = 0; q < kMaxClusterSplit; ++q)
                sm->wts[q][h] = (wsum > 0.f && ls[q] != -INFINITY && l[q] > 0.f) ? __expf(ls[q] - mx) / (wsum * l[q]) : 0.f;
            if (sp == 0 && h < hv) p.lse[hrow0 + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
        }
        __syncthreads();
        // split q0 (its rows already here) opens the sums, the others follow in index order
        float4 acc[kMergeItems];
#pragma unroll
        for (int k = 0; k < kMergeItems; ++k) {
            const float w = k < kcount ? sm->wts[q0][hh[k]] : 0.f;
            acc[k] = make_float4(w * v0[k].x, w * v0[k].y, w * v0[k].z, w * v0[k].w);
        }
#pragma unroll 1
        for (int q = 0; q < ns; ++q) {
            if (q == q0) continue;
            float4 v[kMergeItems];
            if (q == sp) {
#pragma unroll
                for (int k = 0; k < kMergeItems; ++k) v[k] = *reinterpret_cast<const float4 *>(stage_f + stage_off(hh[k], cc[k]));
            } else {
                const float *rowq = p.o_part + ((int64_t)q * p.R * p.H + hrow0) * kPartRow;
#pragma unroll
                for (int k = 0; k < kMergeItems; ++k)
                    if (k < kcount) v[k] = __ldcg(reinterpret_cast<const float4 *>(rowq + hh[k] * kPartRow + 4 * cc[k]));
            }
#pragma unroll
            for (int k = 0; k < kMergeItems; ++k) {
                if (k < kcount) {
                    const float w = sm->wts[q][hh[k]];
                    acc[k].x += w * v[k].x; acc[k].y += w * v[k].y;
                    acc[k].z += w * v[k].z; acc[k].w += w * v[k].w;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kMergeItems; ++k)
            if (k < kcount)
                *reinterpret_cast<uint2 *>(p.out + (hrow0 + hh[k]) * kDl + 4 * cc[k]) =
                    make_uint2(pack_bf16x2(acc[k].x, acc[k].y), pack_bf16x2(acc[k].z, acc[k].w));
    }
}

// Several splits without a cluster: out[r, h, :] = sum_s exp(lse_s - lse) O_s / l_s,
// lse = ln sum_s exp(lse_s) (partial rows: raw O | lse, l).  Every split's header and
// 16-byte slice are loaded at once (all in flight), then weighed against the largest
// lse and summed in split order.
constexpr int kMaxSplit = 16;

__global__ void __launch_bounds__(128)
sparse_mla_combine_kernel(const float *o_part, int nsplit, int64_t rows, __nv_bfloat16 *out, float *lse)
{
    const int64_t row = blockIdx.x;
    const int d = threadIdx.x * 4;
    float ls[kMaxSplit], l[kMaxSplit];
    float4 v[kMaxSplit];
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s) {
        ls[s] = -INFINITY;
        l[s] = 0.f;
        v[s] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s < nsplit) {
            const float *pr = o_part + (s * rows + row) * kPartRow;
            const float2 hd = *reinterpret_cast<const float2 *>(pr + kDl);
            ls[s] = hd.x;
            l[s] = hd.y;
            v[s] = *reinterpret_cast<const float4 *>(pr + d);
        }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s)
        if (l[s] > 0.f) mx = fmaxf(mx, ls[s]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s) {
        if (!(l[s] > 0.f) || ls[s] == -INFINITY) continue;
        const float e = __expf(ls[s] - mx), w = e / l[s];
        acc = make_float4(acc.x + w * v[s].x, acc.y + w * v[s].y, acc.z + w * v[s].z, acc.w + w * v[s].w);
        wsum += e;
    }
    const float iw = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * iw, acc.y * iw), hi = __floats2bfloat162_rn(acc.z * iw, acc.w * iw);
    *reinterpret_cast<__nv_bfloat162 *>(out + row * kDl + d) = lo;
    *reinterpret_cast<__nv_bfloat162 *>(out + row * kDl + d + 2) = hi;
    if (threadIdx.x == 0) lse[row] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

// Splits of the top-k list per (row, head group), one CTA per SM: minimise
// waves x (tiles per split + per-CTA overhead), the overhead (Q load, TMEM
// set-up, epilogue, partial write) counted as about one and a half tiles.
void choose_split(int R, int H, int topk, int &nsplit, int &tiles_per_split)
{
    const int tiles = (topk + kTok - 1) / kTok;
    const int64_t base = (int64_t)R * ((H + kHc - 1) / kHc);
    const int sms = current_sm_count() > 0 ? current_sm_count() : 1;
    int best_ns = 1;
    double best_cost = -1.0;
    for (int ns = 1; ns <= kMaxSplit && ns <= tiles; ++ns) {
        const int tps = (tiles + ns - 1) / ns;
        if ((tiles + tps - 1) / tps != ns) continue;
        const int64_t units = base * ns;
        const double cost = (double)((units + sms - 1) / sms) * (tps + (ns > 1 ? 1.5 : 1.0));
        if (best_cost < 0.0 || cost < best_cost - 1e-9) {
            best_cost = cost;
            best_ns = ns;
        }
    }
    nsplit = best_ns;
    tiles_per_split = (tiles + best_ns - 1) / best_ns;
}

bool tc_applicable(nsa_dtype q_dtype, nsa_dtype kv_dtype, int H, int d_latent, int d_rope)
{
    return q_dtype == NSA_DT_BF16 && (kv_dtype == NSA_DT_BF16 || kv_dtype == NSA_DT_E4M3) && d_latent == kDl &&
           d_rope == kDr && (H % kHc == 0 || H < kHc) && H % 16 == 0;
}

size_t tc_smem_bytes() { return 1024 + kQBytes + kKvBytes + 1024 + sizeof(MlaShared); }

// Whether the `ns` splits of a (row, head group) can run as one thread-block
// cluster of this kernel on the current device (queried once per device,
// split count and KV type).
bool cluster_merge_ok(int ns, bool fp8)
{
    if (ns < 2 || ns > kMaxClusterSplit) return false;
    constexpr int kMaxDev = 64;
    static int cache[kMaxDev][kMaxClusterSplit + 1][2];  // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
    int &c = cache[dev][ns][fp8 ? 1 : 0];
    if (c == 0) {
        const void *kern = fp8 ? (const void *)sparse_mla_tc_kernel<true> : (const void *)sparse_mla_tc_kernel<false>;
        int n = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, (unsigned)ns, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = tc_smem_bytes();
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = (unsigned)ns;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes()) ==
                            cudaSuccess &&
                        cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1;
        if (!ok) (void)cudaGetLastError();  // a failed query is not the caller's error
        c = ok ? 1 : 2;
    }
    return c == 1;
}

}  // namespace

bool sparse_mla_tc_plan(nsa_dtype q_dtype, nsa_dtype kv_dtype, int R, int H, int d_latent, int d_rope, int topk,
                        int *nsplit, int *launches)
{
    if (!tc_applicable(q_dtype, kv_dtype, H, d_latent, d_rope) || R <= 0 || R > 65535 || topk <= 0) return false;
    int ns, tps;
    choose_split(R, H, topk, ns, tps);
    *nsplit = ns;
    *launches = (ns > 1 && !cluster_merge_ok(ns, kv_dtype == NSA_DT_E4M3)) ? 2 : 1;
    return true;
}

size_t sparse_mla_tc_workspace_bytes(nsa_dtype q_dtype, nsa_dtype kv_dtype, int R, int H, int d_latent, int d_rope,
                                     int topk)
{
    if (!tc_applicable(q_dtype, kv_dtype, H, d_latent, d_rope) || R <= 0 || topk <= 0) return 0;
    int ns, tps;
    choose_split(R, H, topk, ns, tps);
    if (ns <= 1) return 0;
    return (size_t)ns * R * H * kPartRow * sizeof(float);
}

nsa_status sparse_mla_tc_try_launch(nsa_dtype q_dtype, nsa_dtype kv_dtype, const void *q_nope, int64_t nope_ld_r,
                                    int64_t nope_ld_h, const void *q_rope, int64_t rope_ld_r, int64_t rope_ld_h,
                                    const void *kv, int64_t num_slots, const int32_t *indices, int64_t indices_ld,
                                    int R, int H, int d_latent, int d_rope, int topk, float sm_scale, void *out,
                                    float *lse, void *workspace, int32_t *status, cudaStream_t stream)
{
    if (!tc_applicable(q_dtype, kv_dtype, H, d_latent, d_rope)) return NSA_ERR_UNSUPPORTED;
    if (num_slots < 1 || num_slots > 2147483647LL) return NSA_ERR_UNSUPPORTED;
    if (((uintptr_t)q_nope & 15) || ((uintptr_t)q_rope & 15) || ((uintptr_t)kv & 15)) return NSA_ERR_UNSUPPORTED;
    if (nope_ld_h % 8 || nope_ld_r % 8 || rope_ld_h % 8 || rope_ld_r % 8) return NSA_ERR_UNSUPPORTED;
    if (R > 65535) return NSA_ERR_UNSUPPORTED;

    MlaParams p;
    p.kv = (const uint8_t *)kv;
    p.q_nope = (const uint16_t *)q_nope;
    p.q_rope = (const uint16_t *)q_rope;
    p.nope_ld_r = nope_ld_r; p.nope_ld_h = nope_ld_h; p.rope_ld_r = rope_ld_r; p.rope_ld_h = rope_ld_h;
    p.indices = indices; p.indices_ld = indices_ld; p.R = R; p.H = H; p.topk = topk; p.num_slots = num_slots;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    choose_split(R, H, topk, p.nsplit, p.tiles_per_split);
    p.out = (__nv_bfloat16 *)out; p.lse = lse; p.status = status;
    p.o_part = nullptr;
    const bool fp8 = kv_dtype == NSA_DT_E4M3;
    p.cluster_merge = cluster_merge_ok(p.nsplit, fp8) ? 1 : 0;
    if (p.nsplit > 1) {
        if (!workspace) return NSA_ERR_INVALID_ARG;
        p.o_part = (float *)workspace;
    }
    const size_t smem = tc_smem_bytes();
    auto kern = fp8 ? sparse_mla_tc_kernel<true> : sparse_mla_tc_kernel<false>;
    NSA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((H + kHc - 1) / kHc), (unsigned)p.nsplit, (unsigned)R);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = p.cluster_merge ? (unsigned)p.nsplit : 1u;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    NSA_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, p));
    if (p.nsplit > 1 && !p.cluster_merge) {
        const int64_t rows = (int64_t)R * H;
        sparse_mla_combine_kernel<<<(unsigned)rows, 128, 0, stream>>>(p.o_part, p.nsplit, rows,
                                                                     (__nv_bfloat16 *)out, lse);
        NSA_CUDA_TRY(cudaGetLastError());
    }
    return NSA_OK;
}

}  // namespace nsa
