// Tensor-core lightning indexer for e4m3 q / K with 64 heads x 128 dims.
//
//   logits[r, s] = k_scale[slot] * sum_h w[r,h] * ReLU(q[r,h,:] . k[slot,:])
//
// The score of the DeepSeek sparse-attention pages ([NSA] NSAIndexerMetadata,
// [DSA] the paged MQA logits call) computed as a dense fp8 contraction:
// for a tile of 128 consecutive positions of one request (two 64-token halves,
// each a contiguous run of one KV page) and the c <= 4 query rows of that
// request handled by the CTA,
//
//   D[128 tokens, 64*c] = K_tile[128, 128] (e4m3) x Q[64*c, 128]^T (e4m3)
//
// accumulates in TMEM (fp32) via tcgen05.mma kind::f8f6f4.  The epilogue
// (one thread per token) applies ReLU, the per-head weights, the head sum and
// the key's scale (bulk-copied into shared memory with the tile), and stores
// one fp32 logit per (row, token).  Given a digit-count buffer, it also counts
// each logit's leading 11-bit key digit (the top-k's first radix digit) per row
// in shared memory and adds the counts to the row's global histogram, so that
// the top-k can start from the threshold digit without reading the scores to
// count them.
//
// Grid: one CTA per SM, persistent, with a deep TMA ring: the tiles of all row groups,
// flattened in (group, subgroup, tile) order, are cut into equal shares, one
// per CTA (each CTA finds its start with one block-wide pass over the row
// lengths), so no SM idles while another works through a long row.
// Roles (320 threads): warp 0 issues TMA loads of K pages and q rows into
// 128B-swizzled shared memory; warp 1 owns TMEM and issues the MMAs; warps
// 2..9 are the epilogue in two sets of four (warp w reads TMEM lanes
// 32*(w%4) .. +31), set k reducing the tiles accumulated in TMEM buffer k.
// Stages are tracked with mbarriers; every wait is bounded and reports
// NSA_ERR_TIMEOUT instead of hanging.
#include <algorithm>
#include <cstddef>

#include "indexer_tc.cuh"
#include "sm100.cuh"
#include "tma_host.h"

namespace nsa {
namespace {

using namespace sm100;

constexpr int kTileTok = 128;
constexpr int kHalf = 64;
constexpr int kDi = 128;
constexpr int kHi = 64;
constexpr int kMaxStages = 12;      // TMA ring depth: as many 16 KB stages as fit one CTA per SM
constexpr int kThreadsTc = 320;     // TMA warp, MMA warp, two sets of four epilogue warps
constexpr int kEpi = kThreadsTc - 64;  // epilogue threads (both sets)
constexpr int kMaxG = 4;
constexpr int kPieceTiles = 16;  // tiles whose page ids the producer warp fetches at once (one half-tile per lane)
static_assert(kPieceTiles * 2 == 32, "the producer warp owns one half-tile per lane");
constexpr uint32_t kTileBytes = kTileTok * kDi;    // 16 KB of e4m3
constexpr uint32_t kHalfBytes = kHalf * kDi;       // 8 KB
constexpr uint32_t kQRowBytes = kHi * kDi;         // 8 KB per query row
constexpr long long kWaitBudget = 2000000000LL;    // ~1 s at 2 GHz
// Digit counts per row in shared memory: two 16-bit counters per word, flushed to
// the global histogram at the end of each segment and at least every kHistFlushTiles
// tiles (each adds at most 128 to a counter, so none passes 65535).
constexpr int kHistWords = kScoreBins / 2;
constexpr int kHistFlushTiles = 256;
static_assert(kHistFlushTiles * kTileTok < 65536, "16-bit digit counters");

struct TcParams {
    const float *w;
    const float *k_scale;
    const int32_t *rpt;
    int64_t rpt_ld;
    const int32_t *row_to_req;
    const int32_t *row_len;
    int R, G, max_row_len, ps;
    int64_t num_pages;
    float *logits;
    int64_t logits_ld;
    uint32_t *hist;       // optional [R][kScoreBins] counts of the logits' leading digits
    int32_t *status;
    uint32_t acc_stride;  // TMEM columns per accumulator buffer
    uint32_t tmem_cols;
    int stages;           // TMA ring depth (<= kMaxStages)
};

struct Bars {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t done;
    uint32_t tmem_base;
    volatile int abort;
    int g0, uo0;                       // first row group of this CTA's share, units into it
    long long u_begin, u_end;          // this CTA's share of the flattened tiles
    long long red[kThreadsTc / 32];
    alignas(16) float w[kMaxG * kHi];  // read as float4
    alignas(16) float scale[kMaxStages][kTileTok];  // key scales of each stage's tile (bulk-copied with it)
    int half_ok[kMaxStages][2];                     // the stage's 64-token halves hold real keys
};
static_assert(offsetof(Bars, scale) % 16 == 0, "bulk-copy destinations are 16-byte aligned");
static_assert(offsetof(Bars, w) % 16 == 0, "the weights are read as float4");

// Paired fp32 arithmetic: two lanes of a 64-bit register, each rounded as fmaf rounds.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float f32x2_sum(uint64_t v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}
static_assert(offsetof(Bars, full) % 8 == 0 && offsetof(Bars, u_begin) % 8 == 0, "mbarriers / 64-bit fields");

// Sub-group n of the CTA's row group: the n-th maximal run of rows sharing a request.
struct SubGroup {
    int r0, c, b, lmax;
};

__device__ __forceinline__ int clamp_len(const TcParams &p, int r)
{
    int L = p.row_len[r];
    return L < 0 ? 0 : (L > p.max_row_len ? p.max_row_len : L);
}

__device__ __forceinline__ bool next_subgroup(const TcParams &p, int g_end, int &r, SubGroup &sg)
{
    if (r >= g_end) return false;
    sg.r0 = r;
    sg.b = p.row_to_req[r];
    sg.lmax = 0;
    int c = 0;
    while (r < g_end && p.row_to_req[r] == sg.b) {
        int L = clamp_len(p, r);
        sg.lmax = L > sg.lmax ? L : sg.lmax;
        ++c;
        ++r;
    }
    sg.c = c;
    return true;
}

__device__ __forceinline__ void fail(Bars *bars, int32_t *status)
{
    bars->abort = 1;
    set_status(status, NSA_ERR_TIMEOUT);
}

// Units of work of row group g: the tiles of each of its subgroups.
__device__ __forceinline__ int group_units(const TcParams &p, int g)
{
    int r = g * p.G, units = 0;
    const int g_end = min(r + p.G, p.R);
    SubGroup sg;
    while (next_subgroup(p, g_end, r, sg)) units += (int)ceil_div(sg.lmax, kTileTok);
    return units;
}

// Walks the CTA's share of the work: calls seg(sg, tb, te) for each run of tiles
// [tb, te) of one subgroup, in (row group, subgroup, tile) order, until seg returns
// false.  check_abort: stop between row groups once the CTA has aborted (roles whose
// threads must agree on every segment pass false and decide inside seg, together).
template <class F>
__device__ __forceinline__ void for_each_segment(const TcParams &p, const Bars *bars, F seg, bool check_abort = true)
{
    int g = bars->g0, uo = bars->uo0;
    long long left = bars->u_end - bars->u_begin;
    const int ngroups = (int)ceil_div(p.R, p.G);
    while (left > 0 && g < ngroups && !(check_abort && bars->abort)) {
        int r = g * p.G;
        const int g_end = min(r + p.G, p.R);
        SubGroup sg;
        while (left > 0 && next_subgroup(p, g_end, r, sg)) {
            const int nt = (int)ceil_div(sg.lmax, kTileTok);
            if (uo >= nt) {
                uo -= nt;
                continue;
            }
            const int tb = uo;
            const int te = (int)min((long long)nt, (long long)tb + left);
            uo = 0;
            left -= te - tb;
            if (!seg(sg, tb, te)) return;
        }
        ++g;
    }
}

__global__ void __launch_bounds__(kThreadsTc, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap, TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *a_ring = smem;                              // stages x 16 KB
    uint8_t *q_smem = a_ring + p.stages * kTileBytes;    // G x 8 KB
    Bars *bars = (Bars *)(q_smem + p.G * kQRowBytes);
    uint32_t *hist_smem = (uint32_t *)(bars + 1);  // [G][kHistWords] when p.hist is set

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    if (threadIdx.x == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&qmap);
    }
    pdl_wait();  // row lengths and page tables come from the metadata kernel

    // ------------------------------------------------------------------ work split
    // The tiles of all row groups, flattened in (group, subgroup, tile) order, are cut
    // into gridDim.x equal shares: every CTA gets the same load and none is empty
    // while another holds a long row.
    const int ngroups = (int)ceil_div(p.R, p.G);
    {
        long long mine = 0;
        const int first_units = threadIdx.x < ngroups ? group_units(p, threadIdx.x) : 0;  // reused by the scan
        mine = first_units;
        for (int g = threadIdx.x + kThreadsTc; g < ngroups; g += kThreadsTc) mine += group_units(p, g);
        for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
        if (lane == 0) bars->red[warp] = mine;
        if (threadIdx.x == 0) {
            bars->g0 = ngroups;
            bars->uo0 = 0;
        }
        __syncthreads();
        long long total = 0;
        for (int w = 0; w < kThreadsTc / 32; ++w) total += bars->red[w];
        const long long u_begin = total * blockIdx.x / gridDim.x;
        const long long u_end = total * (blockIdx.x + 1) / gridDim.x;
        if (threadIdx.x == 0) {
            bars->u_begin = u_begin;
            bars->u_end = u_end;
        }
        // the group holding unit u_begin: a block scan over the groups, chunk by chunk
        long long carry = 0;
        for (int base = 0; base < ngroups && u_end > u_begin; base += kThreadsTc) {
            const int g = base + threadIdx.x;
            const long long u = g < ngroups ? (base == 0 ? first_units : group_units(p, g)) : 0;
            long long incl = u;
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            __syncthreads();  // red[] free
            if (lane == 31) bars->red[warp] = incl;
            __syncthreads();
            long long before = carry;
            for (int w = 0; w < warp; ++w) before += bars->red[w];
            long long chunk = 0;
            for (int w = 0; w < kThreadsTc / 32; ++w) chunk += bars->red[w];
            const long long excl = before + incl - u;
            if (g < ngroups && u > 0 && excl <= u_begin && u_begin < excl + u) {
                bars->g0 = g;
                bars->uo0 = (int)(u_begin - excl);
            }
            carry += chunk;
            if (carry > u_begin) break;  // uniform: every thread holds the same carry
        }
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&bars->full[i], 1);
            mbar_init(&bars->empty[i], 1 + 128);  // the MMA and every epilogue thread release a stage
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->acc_full[i], 1);
            mbar_init(&bars->acc_empty[i], 128);
        }
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        mbar_init(&bars->done, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        // The whole warp walks the tiles; lane l owns half-tile l of each piece of
        // up to kPieceTiles tiles, so its page ids arrive in one round trip.
        uint32_t it = 0, qi = 0;
        uint32_t issued_mask = 0, last_parity = 0;
        for_each_segment(p, bars, [&](const SubGroup &sg, int tb, int te) -> bool {
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait(&bars->q_empty, (qi & 1) ^ 1, kWaitBudget);
                if (ok) {
                    mbar_arrive_expect_tx(&bars->q_full, sg.c * kQRowBytes);
                    for (int i = 0; i < sg.c; ++i)
                        tma_load_2d(q_smem + i * kQRowBytes, &qmap, 0, (sg.r0 + i) * kHi, &bars->q_full);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) { if (lane == 0) fail(bars, p.status); return false; }
            ++qi;
            for (int pb = tb; pb < te; pb += kPieceTiles) {
                const int pe = min(te, pb + kPieceTiles);
                int my_row = -1;  // first KV slot of my half-tile, -1 if none
                {
                    const int s = (pb + (lane >> 1)) * kTileTok + (lane & 1) * kHalf;
                    if (pb + (lane >> 1) < pe && s < sg.lmax) {
                        const int64_t page = p.rpt[(int64_t)sg.b * p.rpt_ld + s / p.ps];
                        if (page >= 0 && page < p.num_pages)
                            my_row = (int)(page * p.ps + s % p.ps);
                        else
                            set_status(p.status, NSA_ERR_BOUNDS);  // its keys score -inf
                    }
                }
                for (int t = pb; t < pe; ++t, ++it) {
                    const int st = it % p.stages;
                    const uint32_t ph = (it / p.stages) & 1;
                    const int row0 = __shfl_sync(0xffffffffu, my_row, 2 * (t - pb));
                    const int row1 = __shfl_sync(0xffffffffu, my_row, 2 * (t - pb) + 1);
                    if (lane == 0) {
                        ok = mbar_wait(&bars->empty[st], ph ^ 1, kWaitBudget);
                        if (ok) {
                            // each real half: 8 KB of keys and their 64 scales (256 B)
                            constexpr uint32_t kScaleBytes = kHalf * sizeof(float);
                            bars->half_ok[st][0] = row0 >= 0;
                            bars->half_ok[st][1] = row1 >= 0;
                            const uint32_t bytes = (row0 >= 0 ? kHalfBytes + kScaleBytes : 0u) +
                                                   (row1 >= 0 ? kHalfBytes + kScaleBytes : 0u);
                            mbar_arrive_expect_tx(&bars->full[st], bytes);
                            if (row0 >= 0) {
                                tma_load_2d(a_ring + st * kTileBytes, &kmap, 0, row0, &bars->full[st]);
                                bulk_load(&bars->scale[st][0], p.k_scale + row0, kScaleBytes, &bars->full[st]);
                            }
                            if (row1 >= 0) {
                                tma_load_2d(a_ring + st * kTileBytes + kHalfBytes, &kmap, 0, row1, &bars->full[st]);
                                bulk_load(&bars->scale[st][kHalf], p.k_scale + row1, kScaleBytes, &bars->full[st]);
                            }
                            issued_mask |= 1u << st;
                            last_parity = (last_parity & ~(1u << st)) | (ph << st);
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, ok, 0)) { if (lane == 0) fail(bars, p.status); return false; }
                }
            }
            return true;
        });
        // drain: never leave with copies in flight
        if (lane == 0)
            for (int st = 0; st < p.stages; ++st)
                if (issued_mask & (1u << st)) mbar_wait(&bars->full[st], (last_parity >> st) & 1, kWaitBudget);
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t it = 0, ai = 0, qi = 0;
            for_each_segment(p, bars, [&](const SubGroup &sg, int tb, int te) -> bool {
                const uint32_t N = kHi * sg.c;
                const uint32_t idesc = instr_desc(0, 0, 0, 0, kTileTok, N);
                if (!mbar_wait(&bars->q_full, qi & 1, kWaitBudget)) { fail(bars, p.status); return false; }
                ++qi;
                for (int t = tb; t < te; ++t, ++it, ++ai) {
                    const int st = it % p.stages;
                    const uint32_t ph = (it / p.stages) & 1;
                    const int ab = ai & 1;
                    const uint32_t aph = (ai >> 1) & 1;
                    if (!mbar_wait(&bars->full[st], ph, kWaitBudget)) { fail(bars, p.status); return false; }
                    if (!mbar_wait(&bars->acc_empty[ab], aph ^ 1, kWaitBudget)) { fail(bars, p.status); return false; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(a_ring + st * kTileBytes);
                    const uint32_t b_addr = smem_u32(q_smem);
                    const uint32_t d = tmem + ab * p.acc_stride;
#pragma unroll
                    for (int k = 0; k < kDi / 32; ++k) {
                        const uint64_t ad = smem_desc(a_addr + k * 32, 16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(b_addr + k * 32, 16, 1024, kSwizzle128B);
                        mma_f8(d, ad, bd, idesc, k > 0 ? 1u : 0u);
                    }
                    mma_commit(&bars->empty[st]);
                    mma_commit(&bars->acc_full[ab]);
                }
                mma_commit(&bars->q_empty);
                return true;
            });
            // all MMAs retired before TMEM is released
            mma_commit(&bars->done);
            mbar_wait(&bars->done, 0, kWaitBudget);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        // Two sets of four warps (one per TMEM lane quadrant each): set k takes the tiles
        // whose accumulator is buffer k, so consecutive tiles are reduced concurrently.
        const int et = threadIdx.x - 64;          // 0 .. kEpi-1
        const int set = et >> 7;                  // 0: warps 2..5, 1: warps 6..9
        const int quad = warp & 3;                // TMEM lane quadrant of this warp
        const int tok = quad * 32 + lane;         // token within the tile
        uint32_t *hs = p.hist ? hist_smem : nullptr;
        if (hs)
            for (int j = et; j < p.G * kHistWords; j += kEpi) hs[j] = 0u;
        // the per-CTA digit counts of a segment's rows go to the global histogram
        auto flush_hist = [&](const SubGroup &sg) {
            asm volatile("bar.sync 1, %0;" ::"n"(kEpi) : "memory");  // every epilogue thread's counts are in
            for (int j = et; j < sg.c * kHistWords; j += kEpi) {
                const uint32_t v = hs[j];
                if (v == 0u) continue;
                hs[j] = 0u;
                uint32_t *g = p.hist + (int64_t)(sg.r0 + j / kHistWords) * kScoreBins + 2 * (j % kHistWords);
                if (v & 0xFFFFu) atomicAdd(g, v & 0xFFFFu);
                if (v >> 16) atomicAdd(g + 1, v >> 16);
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kEpi) : "memory");  // cleared before anyone counts again
        };
        // Both sets take every decision that guards a barrier together: after a failed wait a
        // set skips its work but keeps every barrier of the segment, and the segment's end
        // tells both sets whether to go on.
        uint32_t ai = 0, it = 0;
        for_each_segment(p, bars, [&](const SubGroup &sg, int tb, int te) -> bool {
            if (bar_red_or(1, kEpi, bars->abort != 0)) return false;  // the weights' buffer is free
            for (int i = et; i < sg.c * kHi; i += kEpi) bars->w[i] = p.w[(int64_t)sg.r0 * kHi + i];
            asm volatile("bar.sync 1, %0;" ::"n"(kEpi) : "memory");
            int Lrow[kMaxG];
#pragma unroll
            for (int i = 0; i < kMaxG; ++i) Lrow[i] = i < sg.c ? clamp_len(p, sg.r0 + i) : 0;
            int since_flush = 0;
            bool bad = false;
            for (int t = tb; t < te; ++t, ++ai, ++it) {
                const int ab = ai & 1;
                if (ab == set && !bad) {
                    const uint32_t aph = (ai >> 1) & 1;
                    const int s = t * kTileTok + tok;
                    // my token's key scale arrived with the tile; then the stage is released
                    const int st = it % p.stages;
                    if (!mbar_wait(&bars->full[st], (it / p.stages) & 1, kWaitBudget)) {
                        fail(bars, p.status);
                        bad = true;
                    }
                    const float scale = bars->scale[st][tok];
                    const bool valid_page = bars->half_ok[st][tok >> 6] != 0;
                    mbar_arrive(&bars->empty[st]);
                    if (!bad && !mbar_wait(&bars->acc_full[ab], aph, kWaitBudget)) {
                        fail(bars, p.status);
                        bad = true;
                    }
                    if (!bad) {  // after a failed wait the set only keeps the barriers
                        tc_fence_after();
                        const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16) + ab * p.acc_stride;
                        for (int i = 0; i < sg.c; ++i) {
                            uint32_t v0[32], v1[32];
                            tmem_ld32(tbase + i * kHi, v0);
                            tmem_ld32(tbase + i * kHi + 32, v1);
                            tmem_ld_wait();
                            const float4 *w4 = reinterpret_cast<const float4 *>(bars->w + i * kHi);
                            // four independent partial sums over the 64 heads (heads h = 0, 1, 2, 3 mod 4;
                            // short dependency chains), as two paired accumulators
                            uint64_t a01 = 0ull, a23 = 0ull;
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 w = w4[q];
                                const float r0 = fmaxf(__uint_as_float(v0[4 * q]), 0.f);
                                const float r1 = fmaxf(__uint_as_float(v0[4 * q + 1]), 0.f);
                                const float r2 = fmaxf(__uint_as_float(v0[4 * q + 2]), 0.f);
                                const float r3 = fmaxf(__uint_as_float(v0[4 * q + 3]), 0.f);
                                a01 = f32x2_fma(f32x2_pack(w.x, w.y), f32x2_pack(r0, r1), a01);
                                a23 = f32x2_fma(f32x2_pack(w.z, w.w), f32x2_pack(r2, r3), a23);
                            }
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 w = w4[8 + q];
                                const float r0 = fmaxf(__uint_as_float(v1[4 * q]), 0.f);
                                const float r1 = fmaxf(__uint_as_float(v1[4 * q + 1]), 0.f);
                                const float r2 = fmaxf(__uint_as_float(v1[4 * q + 2]), 0.f);
                                const float r3 = fmaxf(__uint_as_float(v1[4 * q + 3]), 0.f);
                                a01 = f32x2_fma(f32x2_pack(w.x, w.y), f32x2_pack(r0, r1), a01);
                                a23 = f32x2_fma(f32x2_pack(w.z, w.w), f32x2_pack(r2, r3), a23);
                            }
                            const float acc = f32x2_sum(a01) + f32x2_sum(a23);
                            const bool in = s < Lrow[i];
                            const float logit = valid_page ? acc * scale : -INFINITY;
                            if (in) p.logits[(int64_t)(sg.r0 + i) * p.logits_ld + s] = logit;
                            if (hs && in) {
                                const uint32_t d = order_key(logit) >> kScoreDigitShift;
                                atomicAdd(&hs[i * kHistWords + (d >> 1)], 1u << ((d & 1u) * 16));
                            }
                        }
                        tc_fence_before();
                        mbar_arrive(&bars->acc_empty[ab]);
                    }
                }
                if (hs && ++since_flush == kHistFlushTiles) {  // both sets count every tile: uniform
                    flush_hist(sg);
                    since_flush = 0;
                }
            }
            if (hs && since_flush > 0) flush_hist(sg);
            return !bar_red_or(1, kEpi, bad);
        }, false);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

}  // namespace

nsa_status indexer_tc_try_launch(nsa_dtype dtype, const void *q, const float *w, const void *k_cache,
                                 const float *k_scale, int64_t num_pages, int page_size, int Hi, int Di,
                                 const int32_t *rpt, int64_t rpt_ld, const int32_t *row_to_req,
                                 const int32_t *row_len, int R, int max_row_len, float *logits,
                                 int64_t logits_ld, uint32_t *score_hist, int32_t *status, cudaStream_t stream,
                                 int rows_per_group)
{
    if (dtype != NSA_DT_E4M3 || Hi != kHi || Di != kDi || page_size % kHalf != 0) return NSA_ERR_UNSUPPORTED;
    if (((uintptr_t)q & 15) || ((uintptr_t)k_cache & 15) || ((uintptr_t)k_scale & 15)) return NSA_ERR_UNSUPPORTED;
    if (num_pages * page_size > 2147483647LL || (int64_t)R * kHi > 2147483647LL) return NSA_ERR_UNSUPPORTED;
    const int G = rows_per_group < 1 ? 1 : (rows_per_group > kMaxG ? kMaxG : rows_per_group);

    CUtensorMap kmap, qmap;
    if (!make_tma_2d(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, k_cache, kDi, (uint64_t)num_pages * page_size, kDi,
                     kDi, kHalf, CU_TENSOR_MAP_SWIZZLE_128B))
        return NSA_ERR_CUDA;
    if (!make_tma_2d(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, kDi, (uint64_t)R * kHi, kDi, kDi, kHi,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return NSA_ERR_CUDA;

    TcParams p;
    p.w = w; p.k_scale = k_scale; p.rpt = rpt; p.rpt_ld = rpt_ld; p.row_to_req = row_to_req; p.row_len = row_len;
    p.R = R; p.G = G; p.max_row_len = max_row_len; p.ps = page_size; p.num_pages = num_pages;
    p.logits = logits; p.logits_ld = logits_ld; p.hist = score_hist; p.status = status;
    p.acc_stride = (uint32_t)(kHi * G);
    uint32_t cols = 32;
    while (cols < 2 * p.acc_stride) cols <<= 1;
    p.tmem_cols = cols;

    // one CTA per SM; the ring takes what the q rows and barriers leave of 227 KB
    const size_t fixed = 1024 + (size_t)G * kQRowBytes + sizeof(Bars) +
                         (score_hist ? (size_t)G * kHistWords * sizeof(uint32_t) : 0);
    p.stages = (int)std::min<size_t>(kMaxStages, (232448 - fixed) / kTileBytes);
    const size_t smem = fixed + (size_t)p.stages * kTileBytes;
    auto kern = indexer_tc_kernel;
    NSA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    // a persistent grid of one CTA per SM shares the flattened tiles evenly
    const int64_t units_max = ceil_div(R, G) * ceil_div(max_row_len, kTileTok);
    int dev = 0, sms = 0;
    NSA_CUDA_TRY(cudaGetDevice(&dev));
    NSA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>(units_max, (int64_t)sms));
    dim3 grid((unsigned)ctas);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreadsTc);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    NSA_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, kmap, qmap, p));
    return NSA_OK;
}

}  // namespace nsa
