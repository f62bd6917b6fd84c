// nsa_topk_transform: per-row top-k of the indexer scores, mapped to KV slots.
//
// [NSA] NSAIndexerMetadata.topk_transform (the fused variant that emits KV
// slots of the page table instead of positions), [DSA]
// transform_index_page_table_* with page size 1 and _pad_topk_indices (-1
// padding); the long-row multi-CTA plan and the indexer-to-top-k fusion follow
// [DSA]'s top-k v2 plan and its fused top-k switch.
//
// Scores become order-preserving 32-bit keys (-0 folded onto +0, NaN below
// every number).  The selection is a most-significant-digit radix select whose
// first 11-bit digit comes from a per-row histogram of the keys' leading bits,
// counted either by the indexer as it writes the scores (fused) or by
// topk_hist_kernel below, over all SMs.
//
// topk_row_kernel (rows up to 16 K positions: 512 threads at 40 registers, up to
// three CTAs per SM where the cached rows allow; up to 40 K positions when the rows
// fit one wave of CTAs: 1024 threads): one CTA per row.  The row's
// keys are read once into shared memory; each thread classifies its run of
// consecutive positions against d1 (from the histogram when it describes the
// scores, else from one shared-memory histogram pass), the positions in the
// threshold bin are compacted in order and resolved on their remaining 21 bits,
// and one scan of the selected counts places every position in order.
//
// topk_chunk_kernel (longer rows): one CTA per 4096-position chunk of a row.  Each CTA picks
// the threshold digit d1 from the row's histogram, reads its chunk once and
// writes, in position order, every position whose digit is above d1 (selected,
// with its KV slot) or equal to it (a candidate, with its key) to a per-chunk
// list, with its counts.  topk_assemble_kernel, launched behind it with one CTA
// per row, checks the counts against the histogram, resolves the remaining 21
// key bits on the candidates alone, and writes the ordered output: one scan over
// the concatenated lists gives every selected position its slot.  Ties go to the
// lower position.  A histogram that does not describe the scores (the counts
// disagree) makes that CTA select the row from the scores directly, so the
// result never depends on the histogram's contents.
#include <algorithm>

#include "nsa_internal.cuh"

namespace nsa {
namespace {

constexpr int kThreads = 512;
constexpr int kChunk = 4096;                       // positions per chunk CTA
constexpr int kHalfChunk = kChunk / 2;             // thread t reads 4t..4t+3 of each half
static_assert(kHalfChunk == 4 * kThreads, "two float4 per thread cover a chunk");
constexpr int kBins = kScoreBins;                  // 11-bit digits
constexpr int kBinsPerThread = kBins / kThreads;   // 4, largest digit first
constexpr int kCandCap = 6144;                     // candidates of the threshold bin held in shared memory
constexpr int kMaxChunks = kThreads;               // rows up to 2 M positions
constexpr int kRowCap = 16384;                     // rows the 512-thread one-CTA kernel caches whole
constexpr int kLongRowCap = 40960;                 // rows the 1024-thread one-CTA kernel caches whole
constexpr int kRowCand = 4096;                     // its threshold-bin capacity
constexpr int kRun = (4096 + kCandCap + kThreads - 1) / kThreads;  // list entries a thread of the assembling CTA holds
constexpr uint32_t kFlag = 0x80000000u;            // list entry: candidate (digit == d1); candidate: selected
constexpr uint32_t kNoDigit = 0xFFFFFFFFu;

// Token slots of request b: its row of the paged table (nullptr when the table's row
// map names no row of it: that request's positions then map to -1, with
// NSA_ERR_BOUNDS), or, ragged, positions offset by the request's first key.
struct SlotMap {
    const int32_t *row;
    int32_t off;
    bool ok;
    __device__ __forceinline__ int32_t operator()(int s) const { return row ? row[s] : (ok ? off + s : -1); }
};

// Dynamic shared memory of topk_assemble_kernel.
struct ChunkSmem {
    uint32_t hist[kBins];
    uint32_t cand_key[kCandCap];
    uint32_t cand_pos[kCandCap];
    uint32_t chunk_off[kMaxChunks + 1];
};

struct TopkArgs {
    const float *logits;
    int64_t logits_ld;
    const int32_t *row_len;
    const int32_t *row_to_req;
    const int32_t *pt;           // paged: page_table_1 (or req_to_token with pt_rows)
    int64_t pt_ld;
    const int32_t *pt_rows;      // optional: row of pt holding request b's slots (else row b)
    int64_t pt_rows_limit;       // rows of pt (pt_rows[b] is checked against it)
    const int32_t *req_offset;   // ragged: per-request offset
    int topk, max_row_len, nch_max;
    int32_t *indices;
    int64_t indices_ld;
    uint32_t *hist;              // [R][kBins] digit counts (cleared after use)
    uint32_t *counts;            // [R][nch_max] (#above | #candidates << 16) per chunk
    uint2 *lists;                // [R][nch_max * kChunk] (position | kFlag on candidates, slot or key)
    int32_t *status;
};

__device__ __forceinline__ SlotMap slot_map(const TopkArgs &a, int b)
{
    SlotMap m{nullptr, a.req_offset ? a.req_offset[b] : 0, true};
    if (a.pt) {
        const int64_t row = a.pt_rows ? (int64_t)a.pt_rows[b] : (int64_t)b;
        m.ok = !a.pt_rows || (row >= 0 && row < a.pt_rows_limit);
        if (m.ok) m.row = a.pt + row * a.pt_ld;
        else if (threadIdx.x == 0) set_status(a.status, NSA_ERR_BOUNDS);
    }
    return m;
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

// The digit of a radix pass that holds the need-th largest key.  Thread t of the NT
// holds the counts c[j] of digits kBins-1-(kBins/NT)t-j (largest first).  On return pick[0] = the
// digit, pick[1] = how many of its keys are still needed, pick[2] = its count
// (kNoDigit if the counts hold fewer than `need` keys); *total = all counts.
template <int NT>
__device__ __forceinline__ void pick_digit(const uint32_t (&c)[kBins / NT], uint32_t need, uint32_t *warp_buf,
                                           uint32_t *total, uint32_t *pick)
{
    constexpr int BPT = kBins / NT;
    uint32_t sum = 0u;
#pragma unroll
    for (int j = 0; j < BPT; ++j) sum += c[j];
    if (threadIdx.x == 0) pick[2] = kNoDigit;  // ordered before every write below by the scan's barriers
    const uint32_t incl = block_incl_scan(sum, warp_buf, total);
    uint32_t cum = incl - sum;
    if (cum < need && need <= incl) {
#pragma unroll
        for (int j = 0; j < BPT; ++j) {
            if (cum + c[j] >= need) {
                pick[0] = (uint32_t)(kBins - 1 - BPT * (int)threadIdx.x - j);
                pick[1] = need - cum;
                pick[2] = c[j];
                break;
            }
            cum += c[j];
        }
    }
    __syncthreads();
}

// The counts of a kBins-bin shared-memory histogram this thread owns, largest digit first.
template <int NT>
__device__ __forceinline__ void own_bins(const uint32_t *h, uint32_t (&c)[kBins / NT], uint32_t dmask)
{
#pragma unroll
    for (int j = 0; j < kBins / NT; ++j) {
        const int d = kBins - 1 - (kBins / NT) * (int)threadIdx.x - j;
        c[j] = d <= (int)dmask ? h[d] : 0u;
    }
}

// The whole block resolves the low 21 key bits on nc candidates whose leading
// digit is d1, `need` of which are to be selected (two radix passes, 11 + 10
// bits, over a kBins shared-memory histogram), then marks the selected ones:
// key above the threshold, or equal to it and among the first `need` such in
// candidate (position) order.  key_of(j) reads candidate j's key, mark(j) flags it.
template <int NT, class KeyOf, class Mark>
__device__ __forceinline__ void resolve_candidates(KeyOf key_of, Mark mark, int nc, uint32_t d1, uint32_t need1,
                                                   uint32_t *h, uint32_t *warp_buf, uint32_t *total, uint32_t *pick)
{
    const int tid = threadIdx.x;
    uint32_t prefix = d1, need = need1;
    int S = kScoreDigitShift;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const int width = pass == 0 ? 11 : 10;
        const int shift = S - width;
        const uint32_t dmask = (1u << width) - 1u;
        __syncthreads();  // the candidates are written; earlier readers of h are done
        for (int i = tid; i < kBins; i += NT) h[i] = 0u;
        __syncthreads();
        for (int j = tid; j < nc; j += NT) {
            const uint32_t k = key_of(j);
            if ((k >> S) == prefix) atomicAdd(&h[(k >> shift) & dmask], 1u);
        }
        __syncthreads();
        uint32_t c[kBins / NT];
        own_bins<NT>(h, c, dmask);
        pick_digit<NT>(c, need, warp_buf, total, pick);
        prefix = (prefix << width) | pick[0];
        need = pick[1];
        S = shift;
        if (pick[2] == need) break;  // the whole bin is selected
    }
    const int per = (nc + NT - 1) / NT;
    const int j0 = min(nc, tid * per), j1 = min(nc, j0 + per);
    uint32_t ties = 0u;
    for (int j = j0; j < j1; ++j) ties += (key_of(j) >> S) == prefix;
    uint32_t tie_before = block_incl_scan(ties, warp_buf, total) - ties;
    for (int j = j0; j < j1; ++j) {
        const uint32_t kv = key_of(j) >> S;
        bool s = kv > prefix;
        if (kv == prefix) s = tie_before++ < need;
        if (s) mark(j);
    }
    __syncthreads();
}

// ---------------------------------------------------------------- histogram pass
// Counts of the leading digits of every row longer than topk, one CTA per chunk:
// a shared-memory histogram of the chunk, its occupied bins added to the row's.
__global__ void __launch_bounds__(kThreads)
topk_hist_kernel(const float *logits, int64_t logits_ld, const int32_t *row_len, int topk, int max_row_len,
                 uint32_t *hist)
{
    __shared__ uint32_t h[kBins];
    pdl_trigger();
    pdl_wait();  // the scores come from the indexer
    const int r = blockIdx.x;
    const int L = row_len[r];
    if (L <= topk || L > max_row_len) return;
    const int s0 = blockIdx.y * kChunk;
    if (s0 >= L) return;
    const int n = min(kChunk, L - s0);
    for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = 0u;
    __syncthreads();
    const float *lg = logits + (int64_t)r * logits_ld + s0;
    for (int i = threadIdx.x; i < n; i += kThreads) atomicAdd(&h[order_key(lg[i]) >> kScoreDigitShift], 1u);
    __syncthreads();
    uint32_t *hrow = hist + (int64_t)r * kBins;
    for (int i = threadIdx.x; i < kBins; i += kThreads)
        if (h[i]) atomicAdd(&hrow[i], h[i]);
}

// ---------------------------------------------------------------- whole-row selection
// One CTA selects row r from its scores alone (up to three radix passes over
// global memory, then one ordered pass).  Used when the histogram does not
// describe the scores or the threshold bin holds more than kCandCap keys.
template <int NT>
__device__ void select_row_directly(const float *lg, int L, int topk, int32_t *out, uint32_t *h,
                                    uint32_t *warp_buf, uint32_t *total, uint32_t *pick, const SlotMap slot_of)
{
    const int tid = threadIdx.x;
    uint32_t prefix = 0u, need = (uint32_t)topk;
    int S = 32;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int width = pass < 2 ? 11 : 10;
        const int shift = S - width;
        const uint32_t dmask = (1u << width) - 1u;
        __syncthreads();
        for (int i = tid; i < kBins; i += NT) h[i] = 0u;
        __syncthreads();
        for (int i = tid; i < L; i += NT) {
            const uint32_t k = order_key(__ldcg(lg + i));
            if (S == 32 || (k >> S) == prefix) atomicAdd(&h[(k >> shift) & dmask], 1u);
        }
        __syncthreads();
        uint32_t c[kBins / NT];
        own_bins<NT>(h, c, dmask);
        pick_digit<NT>(c, need, warp_buf, total, pick);
        prefix = (S == 32 ? 0u : (prefix << width)) | pick[0];
        need = pick[1];
        S = shift;
        if (pick[2] == need) break;  // the whole bin is selected
    }
    // ordered pass: every key above the threshold, and the first `need` equal to it
    uint32_t gt_run = 0u, eq_run = 0u;
    for (int base = 0; base < L; base += 4 * NT) {
        const int i0 = base + 4 * tid;
        uint32_t cls[4], a_gt = 0u, a_eq = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            cls[j] = 0u;
            if (i0 + j < L) {
                const uint32_t v = order_key(__ldcg(lg + i0 + j)) >> S;
                cls[j] = v > prefix ? 2u : (v == prefix ? 1u : 0u);
            }
            a_gt += cls[j] == 2u;
            a_eq += cls[j] == 1u;
        }
        const uint32_t packed = a_gt | (a_eq << 16);
        const uint32_t incl = block_incl_scan(packed, warp_buf, total);
        uint32_t gt_before = gt_run + ((incl - packed) & 0xFFFFu);
        uint32_t eq_before = eq_run + ((incl - packed) >> 16);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (cls[j] == 2u) {
                out[gt_before + (eq_before < need ? eq_before : need)] = slot_of(i0 + j);
                ++gt_before;
            } else if (cls[j] == 1u) {
                if (eq_before < need) out[gt_before + eq_before] = slot_of(i0 + j);
                ++eq_before;
            }
        }
        gt_run += *total & 0xFFFFu;
        eq_run += *total >> 16;
        __syncthreads();  // *total is read before the next scan writes it
    }
}

// Keys of lg[0 .. n) into cache[0 .. n): 16-byte loads when aligned, all in flight at once.
template <int NT, int CAP>
__device__ __forceinline__ void fill_keys(const float *lg, int n, uint32_t *cache)
{
    constexpr int kV = CAP / (4 * NT);  // float4 per thread for a full row
    if ((((uintptr_t)lg) & 15) == 0) {
        const int nv = n >> 2;
        float4 v[kV];
#pragma unroll
        for (int u = 0; u < kV; ++u) {
            const int j = u * NT + (int)threadIdx.x;
            if (j < nv) v[u] = __ldg(reinterpret_cast<const float4 *>(lg) + j);
        }
#pragma unroll
        for (int u = 0; u < kV; ++u) {
            const int j = u * NT + (int)threadIdx.x;
            if (j < nv)
                reinterpret_cast<uint4 *>(cache)[j] =
                    make_uint4(order_key(v[u].x), order_key(v[u].y), order_key(v[u].z), order_key(v[u].w));
        }
        for (int i = (nv << 2) + (int)threadIdx.x; i < n; i += NT) cache[i] = order_key(lg[i]);
    } else {
        for (int i = threadIdx.x; i < n; i += NT) cache[i] = order_key(lg[i]);
    }
}

// Output slots of the selected positions sel[0 .. topk): the page-table reads of
// four slots per thread go out together.
template <int NT, class SlotOf>
__device__ __forceinline__ void write_slots(const uint32_t *sel, int topk, int32_t *out, SlotOf slot_of)
{
    for (int j0 = 0; j0 < topk; j0 += 4 * NT) {
        int32_t s[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = j0 + u * NT + (int)threadIdx.x;
            s[u] = j < topk ? slot_of((int)sel[j]) : 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = j0 + u * NT + (int)threadIdx.x;
            if (j < topk) out[j] = s[u];
        }
    }
}

template <int NT, int CAP>
__global__ void __launch_bounds__(NT, (NT < 1024 ? 3 : 1))
topk_row_kernel(const TopkArgs a)
{
    extern __shared__ __align__(16) uint32_t dyn[];
    uint32_t *h1 = dyn;                 // [kBins]; then, with cand, the selected positions
    uint32_t *cand = dyn + kBins;       // [kRowCand] positions in the threshold bin (kFlag: selected)
    uint32_t *cache = cand + kRowCand;  // [max_row_len] keys
    __shared__ uint32_t warp_buf[32];
    __shared__ uint32_t total;
    __shared__ uint32_t pick[3];

    pdl_trigger();
    pdl_wait();  // the scores (and the digit counts) come from the indexer
    const int r = blockIdx.x, tid = threadIdx.x;
    const int L = a.row_len[r];
    const int b = a.row_to_req[r];
    int32_t *out = a.indices + (int64_t)r * a.indices_ld;
    const SlotMap slot_of = slot_map(a, b);
    const float *lg = a.logits + (int64_t)r * a.logits_ld;

    // the indexer's digit counts of this row (a hint), read and cleared
    uint32_t *hrow = a.hist ? a.hist + (int64_t)r * kBins : nullptr;
    uint32_t hc[(kBins / NT)];
#pragma unroll
    for (int j = 0; j < (kBins / NT); ++j) {
        const int d = kBins - 1 - (kBins / NT) * tid - j;
        hc[j] = hrow ? hrow[d] : 0u;
        if (hrow) hrow[d] = 0u;
    }
    if (L < 0 || L > a.max_row_len || L <= a.topk) {
        const bool bad = L < 0 || L > a.max_row_len;
        if (bad && tid == 0) set_status(a.status, NSA_ERR_BOUNDS);
        for (int i = tid; i < a.topk; i += NT) out[i] = (!bad && i < L) ? slot_of(i) : -1;
        return;
    }
    fill_keys<NT, CAP>(lg, L, cache);

    const int C = 4 * (((L + 4 * NT - 1) / (4 * NT)) | 1);  // <= 44 positions a thread (CAP / NT <= 40)
    const int p0 = min(L, tid * C), p1 = min(L, p0 + C);
    bool have = false;
    if (hrow) {
        pick_digit<NT>(hc, (uint32_t)a.topk, warp_buf, &total, pick);
        have = total == (uint32_t)L && pick[2] != kNoDigit;  // uniform: shared values
    } else {
        __syncthreads();  // the cached keys are complete
    }
    bool done = false;
#pragma unroll 1
    for (int attempt = 0; attempt < 2 && !done; ++attempt) {
        if (!have) {
            for (int i = tid; i < kBins; i += NT) h1[i] = 0u;
            __syncthreads();
            for (int i4 = tid; i4 < (L >> 2); i4 += NT) {
                const uint4 k = reinterpret_cast<const uint4 *>(cache)[i4];
                atomicAdd(&h1[k.x >> kScoreDigitShift], 1u);
                atomicAdd(&h1[k.y >> kScoreDigitShift], 1u);
                atomicAdd(&h1[k.z >> kScoreDigitShift], 1u);
                atomicAdd(&h1[k.w >> kScoreDigitShift], 1u);
            }
            if (tid < (L & 3)) atomicAdd(&h1[cache[(L & ~3) + tid] >> kScoreDigitShift], 1u);
            __syncthreads();
            own_bins<NT>(h1, hc, kBins - 1);
            pick_digit<NT>(hc, (uint32_t)a.topk, warp_buf, &total, pick);
            have = true;
        }
        const uint32_t d1 = pick[0], need1 = pick[1], cnt1 = pick[2];
        // classify my run, four keys at a time (the last group may pass the row's end)
        uint64_t mgt = 0ull, meq = 0ull;
        for (int i = p0; i < p1; i += 4) {
            const uint4 v = *reinterpret_cast<const uint4 *>(cache + i);
            const uint32_t e0 = v.x >> kScoreDigitShift, e1 = v.y >> kScoreDigitShift;
            const uint32_t e2 = v.z >> kScoreDigitShift, e3 = v.w >> kScoreDigitShift;
            uint32_t g = (uint32_t)(e0 > d1) | ((uint32_t)(e1 > d1) << 1) | ((uint32_t)(e2 > d1) << 2) |
                         ((uint32_t)(e3 > d1) << 3);
            uint32_t q = (uint32_t)(e0 == d1) | ((uint32_t)(e1 == d1) << 1) | ((uint32_t)(e2 == d1) << 2) |
                         ((uint32_t)(e3 == d1) << 3);
            if (p1 - i < 4) {
                const uint32_t vm = (1u << (p1 - i)) - 1u;
                g &= vm;
                q &= vm;
            }
            mgt |= (uint64_t)g << (i - p0);
            meq |= (uint64_t)q << (i - p0);
        }
        const uint32_t n_gt = (uint32_t)__popcll(mgt), n_eq = (uint32_t)__popcll(meq);
        const uint32_t packed = n_gt | (n_eq << 16);  // L <= kRowCap: both fit 16 bits
        const uint32_t ex = block_incl_scan(packed, warp_buf, &total) - packed;
        const uint32_t tot_gt = total & 0xFFFFu, tot_eq = total >> 16;
        if (cnt1 == kNoDigit || tot_gt != (uint32_t)a.topk - need1 || tot_eq != cnt1) {
            have = false;  // the hint does not describe these scores: count them here
            continue;
        }
        uint64_t msel;
        if (tot_eq == need1) {
            msel = mgt | meq;  // the whole bin is selected
        } else if (tot_eq > (uint32_t)kRowCand) {
            break;  // a crowded bin: selected from the scores directly below
        } else {
            const uint32_t eq_before = ex >> 16;
            {
                uint32_t j = eq_before;
                for (uint64_t m = meq; m; m &= m - 1, ++j) cand[j] = (uint32_t)(p0 + __ffsll((long long)m) - 1);
            }
            resolve_candidates<NT>([&](int j) -> uint32_t { return cache[cand[j] & ~kFlag]; },
                               [&](int j) { cand[j] |= kFlag; }, (int)tot_eq, d1, need1, h1, warp_buf, &total, pick);
            uint64_t seq = 0ull;
            {
                uint32_t j = eq_before;
                for (uint64_t m = meq; m; m &= m - 1, ++j)
                    if (cand[j] & kFlag) seq |= m & (~m + 1ull);
            }
            msel = mgt | seq;
        }
        // ordered output: every selected position gets its slot in one scan
        const uint32_t n_sel = (uint32_t)__popcll(msel);
        uint32_t before = block_incl_scan(n_sel, warp_buf, &total) - n_sel;  // its barriers retire the reads above
        uint32_t *sel = dyn;  // [topk] over h1 and cand
        for (uint64_t m = msel; m; m &= m - 1) sel[before++] = (uint32_t)(p0 + __ffsll((long long)m) - 1);
        __syncthreads();
        write_slots<NT>(sel, a.topk, out, slot_of);
        done = true;
    }
    if (!done) select_row_directly<NT>(lg, L, a.topk, out, h1, warp_buf, &total, pick, slot_of);
}

// ---------------------------------------------------------------- chunks
// One CTA per 4096-position chunk: the threshold digit d1 from the row's counts,
// then every position of the chunk whose digit is above d1 (with its KV slot) or
// equal to it (a candidate, with its key) goes to the chunk's list, in order.
__global__ void __launch_bounds__(kThreads, 4)
topk_chunk_kernel(const TopkArgs a)
{
    __shared__ uint32_t warp_buf[32];
    __shared__ uint32_t total;
    __shared__ uint32_t pick[3];
    __shared__ uint32_t n_gt_s, n_eq_s;

    pdl_trigger();
    pdl_wait();  // the scores and the digit counts come from the previous kernels
    const int r = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
    const int L = a.row_len[r];
    if (L < 0 || L > a.max_row_len || L <= a.topk) return;  // written by the assemble kernel
    const int nch = (L + kChunk - 1) / kChunk;
    if (c >= nch) return;
    const int b = a.row_to_req[r];
    const SlotMap slot_of = slot_map(a, b);
    const float *lg = a.logits + (int64_t)r * a.logits_ld;
    const uint32_t *hrow = a.hist + (int64_t)r * kBins;

    const int s0 = c * kChunk, n = min(kChunk, L - s0);
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int i = (j >> 2) * kHalfChunk + 4 * tid + (j & 3);
        v[j] = i < n ? lg[s0 + i] : 0.f;
    }
    uint32_t hc[kBinsPerThread];
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) hc[j] = hrow[kBins - 1 - kBinsPerThread * tid - j];
    if (tid == 0) n_gt_s = n_eq_s = 0u;
    pick_digit<kThreads>(hc, (uint32_t)a.topk, warp_buf, &total, pick);
    const bool pick_ok = pick[2] != kNoDigit;
    const uint32_t d1 = pick[0];

    // classify: bit j of gt / eq for my key j (keys 0-3: first half, 4-7: second half)
    uint32_t gt = 0u, eq = 0u, key[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int i = (j >> 2) * kHalfChunk + 4 * tid + (j & 3);
        key[j] = order_key(v[j]);
        if (i < n && pick_ok) {
            const uint32_t d = key[j] >> kScoreDigitShift;
            if (d > d1) gt |= 1u << j;
            else if (d == d1) eq |= 1u << j;
        }
    }
    const uint32_t sel = gt | eq;
    // the KV slots of the positions selected for sure: their page-table reads go out together
    uint32_t w1[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int i = (j >> 2) * kHalfChunk + 4 * tid + (j & 3);
        w1[j] = ((gt >> j) & 1u) ? (uint32_t)slot_of(s0 + i) : key[j];
    }
    const uint32_t nA = (uint32_t)__popc(sel & 0xFu), nB = (uint32_t)__popc(sel >> 4);
    const uint32_t packed = nA | (nB << 16);
    const uint32_t ex = block_incl_scan(packed, warp_buf, &total) - packed;
    const uint32_t totA = total & 0xFFFFu;
    uint2 *list = a.lists + ((int64_t)r * a.nch_max + c) * kChunk;
    {
        uint32_t oA = ex & 0xFFFFu, oB = totA + (ex >> 16);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (!((sel >> j) & 1u)) continue;
            const int i = (j >> 2) * kHalfChunk + 4 * tid + (j & 3);
            const uint2 e = make_uint2((uint32_t)(s0 + i) | (((eq >> j) & 1u) ? kFlag : 0u), w1[j]);
            if (j < 4) list[oA++] = e;
            else list[oB++] = e;
        }
    }
    {
        uint32_t g = (uint32_t)__popc(gt), q = (uint32_t)__popc(eq);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, o);
            q += __shfl_xor_sync(0xffffffffu, q, o);
        }
        if ((tid & 31) == 0 && (g | q)) {
            atomicAdd(&n_gt_s, g);
            atomicAdd(&n_eq_s, q);
        }
    }
    __syncthreads();
    if (tid == 0) a.counts[(int64_t)r * a.nch_max + c] = n_gt_s | (n_eq_s << 16);
}

// ---------------------------------------------------------------- assemble
// One CTA per row: checks the chunks' counts against the digit counts, resolves
// the threshold bin on the candidates (one warp), and writes the ordered output
// from one scan over the concatenated lists, each thread holding its run of
// entries in registers.  Rows of at most topk positions are written here too.
__global__ void __launch_bounds__(kThreads, 1)
topk_assemble_kernel(const TopkArgs a)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    ChunkSmem &sm = *reinterpret_cast<ChunkSmem *>(smem_raw);
    __shared__ uint32_t warp_buf[32];
    __shared__ uint32_t total;
    __shared__ uint32_t pick[3];

    pdl_trigger();
    pdl_wait();  // the chunk lists come from the previous kernel
    const int r = blockIdx.x, tid = threadIdx.x;
    const int L = a.row_len[r];
    const int b = a.row_to_req[r];
    int32_t *out = a.indices + (int64_t)r * a.indices_ld;
    const SlotMap slot_of = slot_map(a, b);
    const float *lg = a.logits + (int64_t)r * a.logits_ld;

    // the row's digit counts, read and cleared for the next call
    uint32_t *hrow = a.hist + (int64_t)r * kBins;
    uint32_t hc[kBinsPerThread];
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) {
        const int d = kBins - 1 - kBinsPerThread * tid - j;
        hc[j] = hrow[d];
        hrow[d] = 0u;
    }
    if (L < 0 || L > a.max_row_len || L <= a.topk) {
        const bool bad = L < 0 || L > a.max_row_len;
        if (bad && tid == 0) set_status(a.status, NSA_ERR_BOUNDS);
        for (int i = tid; i < a.topk; i += kThreads) out[i] = (!bad && i < L) ? slot_of(i) : -1;
        return;
    }
    const int nch = (L + kChunk - 1) / kChunk;
    uint32_t cg = 0u, cq = 0u;
    if (tid < nch) {
        const uint32_t w = a.counts[(int64_t)r * a.nch_max + tid];
        cg = w & 0xFFFFu;
        cq = w >> 16;
    }
    pick_digit<kThreads>(hc, (uint32_t)a.topk, warp_buf, &total, pick);
    const bool pick_ok = pick[2] != kNoDigit;
    const uint32_t d1 = pick[0], need1 = pick[1], cnt1 = pick[2];
    // chunk offsets of the concatenated lists (chunk t's list after those of chunks < t)
    const uint32_t incl_len = block_incl_scan(cg + cq, warp_buf, &total);
    if (tid < nch) sm.chunk_off[tid] = incl_len - cg - cq;
    const uint32_t list_len = total;
    if (tid == 0) sm.chunk_off[nch] = list_len;
    block_incl_scan(cq, warp_buf, &total);
    const uint32_t tot_eq = total, tot_gt = list_len - tot_eq;
    const bool counts_ok = pick_ok && tot_gt == (uint32_t)a.topk - need1 && tot_eq == cnt1;
    if (!counts_ok || (tot_eq != need1 && tot_eq > (uint32_t)kCandCap)) {
        select_row_directly<kThreads>(lg, L, a.topk, out, sm.hist, warp_buf, &total, pick, slot_of);
        return;
    }
    // my contiguous run [i0, i1) of the concatenated list, in registers
    const uint32_t per = (list_len + kThreads - 1) / kThreads;  // <= kRun: list_len <= topk + kCandCap
    const uint32_t i0 = min(list_len, (uint32_t)tid * per), i1 = min(list_len, i0 + per);
    uint2 e[kRun];
    {
        int lo_c = 0, hi_c = nch - 1;  // the last chunk whose offset is <= i0
        while (lo_c < hi_c) {
            const int mid = (lo_c + hi_c + 1) >> 1;
            if (sm.chunk_off[mid] <= i0) lo_c = mid;
            else hi_c = mid - 1;
        }
        int chc = lo_c;
        const uint2 *lists_r = a.lists + (int64_t)r * a.nch_max * kChunk;
#pragma unroll
        for (int u = 0; u < kRun; ++u) {
            const uint32_t k = i0 + (uint32_t)u;
            e[u] = make_uint2(0u, 0u);
            if (k < i1) {
                while (k >= sm.chunk_off[chc + 1]) ++chc;
                e[u] = lists_r[(int64_t)chc * kChunk + (k - sm.chunk_off[chc])];
            }
        }
    }
    const int cnt = (int)(i1 - i0);
    if (tot_eq == need1) {
        // the whole threshold bin is selected: the lists are the output, in order
        int32_t v[kRun];
#pragma unroll
        for (int u = 0; u < kRun; ++u)
            v[u] = u < cnt ? ((e[u].x & kFlag) ? slot_of((int)(e[u].x & ~kFlag)) : (int32_t)e[u].y) : 0;
#pragma unroll
        for (int u = 0; u < kRun; ++u)
            if (u < cnt) out[i0 + u] = v[u];
        return;
    }
    // candidates, compacted in position order with their keys
    uint32_t nf = 0u;
#pragma unroll
    for (int u = 0; u < kRun; ++u) nf += (u < cnt) ? (e[u].x >> 31) : 0u;
    const uint32_t my_first = block_incl_scan(nf, warp_buf, &total) - nf;
    {
        uint32_t cb = my_first;
#pragma unroll
        for (int u = 0; u < kRun; ++u) {
            if (u < cnt && (e[u].x & kFlag)) {
                sm.cand_pos[cb] = e[u].x & ~kFlag;
                sm.cand_key[cb] = e[u].y;
                ++cb;
            }
        }
    }
    resolve_candidates<kThreads>([&](int j) -> uint32_t { return sm.cand_key[j]; }, [&](int j) { sm.cand_pos[j] |= kFlag; },
                       (int)tot_eq, d1, need1, sm.hist, warp_buf, &total, pick);
    // ordered output: above-d1 entries, and the selected candidates
    bool s[kRun];
    uint32_t nsel = 0u;
    {
        uint32_t cj = my_first;
#pragma unroll
        for (int u = 0; u < kRun; ++u) {
            s[u] = u < cnt;
            if (s[u] && (e[u].x & kFlag)) s[u] = (sm.cand_pos[cj++] >> 31) != 0u;
            nsel += s[u];
        }
    }
    uint32_t o = block_incl_scan(nsel, warp_buf, &total) - nsel;
    int32_t v[kRun];
#pragma unroll
    for (int u = 0; u < kRun; ++u)
        v[u] = s[u] ? ((e[u].x & kFlag) ? slot_of((int)(e[u].x & ~kFlag)) : (int32_t)e[u].y) : 0;
#pragma unroll
    for (int u = 0; u < kRun; ++u)
        if (s[u]) out[o++] = v[u];
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Which kernels select the rows: one 512-thread CTA per row up to kRowCap positions;
// one 1024-thread CTA per row up to kLongRowCap positions while the rows fit one wave
// (few long rows: the other SMs stay free for the next kernel's start); else chunks.
enum { kPathRow, kPathLongRow, kPathChunks };

int topk_path(int R, int max_row_len)
{
    if (max_row_len <= kRowCap) return kPathRow;
    const int sms = current_sm_count();
    if (max_row_len <= kLongRowCap && sms > 0 && R <= sms) return kPathLongRow;
    return kPathChunks;
}

struct WsLayout {
    size_t hist, counts, lists, bytes;
};

// Workspace of the chunked path: the digit counts [R][kBins] when the caller gives
// none, per-chunk counts [R][nch] and lists [R][nch * kChunk] of (position, slot|key).
WsLayout ws_layout(int R, int max_row_len, bool own_hist)
{
    const int64_t nch = std::max<int64_t>(1, ceil_div(max_row_len, kChunk));
    WsLayout w;
    w.hist = 0;
    w.counts = own_hist ? align256((size_t)R * kBins * sizeof(uint32_t)) : 0;
    w.lists = w.counts + align256((size_t)R * nch * sizeof(uint32_t));
    w.bytes = w.lists + align256((size_t)R * nch * kChunk * sizeof(uint2));
    return w;
}

nsa_status topk_launch(const float *logits_dev, int64_t logits_ld, const int32_t *row_len_dev,
                       const int32_t *row_to_req_dev, const int32_t *page_table_1_dev, int64_t pt_ld,
                       const int32_t *pt_rows_dev, int64_t pt_rows_limit, const int32_t *req_offset_dev, int R, int topk, int max_row_len, int32_t *indices_dev,
                       int64_t indices_ld, uint32_t *score_hist_dev, void *ws, size_t ws_bytes, int32_t *status_dev,
                       nsa_stream_t stream)
{
    if (R < 0 || topk < 1 || topk > 4096 || max_row_len < 0) return NSA_ERR_INVALID_ARG;
    if (indices_ld < topk || logits_ld < max_row_len || (page_table_1_dev && pt_ld < max_row_len))
        return NSA_ERR_INVALID_ARG;
    if (pt_rows_dev && (!page_table_1_dev || pt_rows_limit < 1)) return NSA_ERR_INVALID_ARG;
    if (ceil_div(max_row_len, kChunk) > kMaxChunks) return NSA_ERR_UNSUPPORTED;
    if (R == 0) return NSA_OK;
    if (!logits_dev || !row_len_dev || !row_to_req_dev || !indices_dev || (!page_table_1_dev && !req_offset_dev))
        return NSA_ERR_INVALID_ARG;
    const int nch = (int)std::max<int64_t>(1, ceil_div(max_row_len, kChunk));
    TopkArgs a;
    a.logits = logits_dev; a.logits_ld = logits_ld; a.row_len = row_len_dev; a.row_to_req = row_to_req_dev;
    a.pt = page_table_1_dev; a.pt_ld = pt_ld; a.req_offset = req_offset_dev;
    a.pt_rows = pt_rows_dev; a.pt_rows_limit = pt_rows_limit;
    a.topk = topk; a.max_row_len = max_row_len; a.nch_max = nch;
    a.indices = indices_dev; a.indices_ld = indices_ld;
    a.hist = score_hist_dev;
    a.counts = nullptr; a.lists = nullptr;
    a.status = status_dev;

    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = (cudaStream_t)stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int path = topk_path(R, max_row_len);
    if (path != kPathChunks) {
        // one CTA per row, the row cached whole (no workspace)
        const size_t smem = (size_t)(kBins + kRowCand + ((max_row_len + 3) & ~3)) * sizeof(uint32_t);
        auto kern = path == kPathRow ? topk_row_kernel<kThreads, kRowCap> : topk_row_kernel<1024, kLongRowCap>;
        NSA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        cfg.gridDim = dim3((unsigned)R);
        cfg.blockDim = dim3(path == kPathRow ? kThreads : 1024);
        cfg.dynamicSmemBytes = smem;
        NSA_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, a));
        return NSA_OK;
    }
    const bool own_hist = score_hist_dev == nullptr;
    const WsLayout w = ws_layout(R, max_row_len, own_hist);
    if (!ws || ws_bytes < w.bytes || ((uintptr_t)ws & 255)) return NSA_ERR_INVALID_ARG;
    uint8_t *base = (uint8_t *)ws;
    if (own_hist) a.hist = (uint32_t *)(base + w.hist);
    a.counts = (uint32_t *)(base + w.counts);
    a.lists = (uint2 *)(base + w.lists);
    cfg.gridDim = dim3((unsigned)R, (unsigned)nch);
    cfg.dynamicSmemBytes = 0;
    if (own_hist)
        NSA_CUDA_TRY(cudaLaunchKernelEx(&cfg, topk_hist_kernel, logits_dev, logits_ld, row_len_dev, topk, max_row_len,
                                        a.hist));
    NSA_CUDA_TRY(cudaLaunchKernelEx(&cfg, topk_chunk_kernel, a));
    NSA_CUDA_TRY(cudaFuncSetAttribute(topk_assemble_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)sizeof(ChunkSmem)));
    cfg.gridDim = dim3((unsigned)R);
    cfg.dynamicSmemBytes = sizeof(ChunkSmem);
    NSA_CUDA_TRY(cudaLaunchKernelEx(&cfg, topk_assemble_kernel, a));
    return NSA_OK;
}

}  // namespace
}  // namespace nsa

extern "C" size_t nsa_topk_workspace_bytes(int R, int max_row_len, int with_score_hist)
{
    if (R <= 0 || nsa::topk_path(R, max_row_len) != nsa::kPathChunks) return 0;
    return nsa::ws_layout(R, max_row_len, with_score_hist == 0).bytes;
}

extern "C" int nsa_topk_launches(int R, int max_row_len, int with_score_hist)
{
    if (R <= 0) return 0;
    if (nsa::topk_path(R, max_row_len) != nsa::kPathChunks) return 1;
    return with_score_hist ? 2 : 3;
}

extern "C" nsa_status nsa_topk_transform(const float *logits_dev, int64_t logits_ld,
                                         const int32_t *row_len_dev, const int32_t *row_to_req_dev,
                                         const int32_t *page_table_1_dev, int64_t pt_ld,
                                         const int32_t *pt_rows_dev, int64_t pt_rows_limit, int R,
                                         int topk, int max_row_len, int32_t *indices_dev,
                                         int64_t indices_ld, uint32_t *score_hist_dev, void *ws, size_t ws_bytes,
                                         int32_t *status_dev, nsa_stream_t stream)
{
    if (!page_table_1_dev && R > 0) return NSA_ERR_INVALID_ARG;
    return nsa::topk_launch(logits_dev, logits_ld, row_len_dev, row_to_req_dev, page_table_1_dev, pt_ld, pt_rows_dev,
                            pt_rows_limit, nullptr, R,
                            topk, max_row_len, indices_dev, indices_ld, score_hist_dev, ws, ws_bytes, status_dev,
                            stream);
}

extern "C" nsa_status nsa_topk_transform_ragged(const float *logits_dev, int64_t logits_ld,
                                                const int32_t *row_len_dev, const int32_t *row_to_req_dev,
                                                const int32_t *req_offset_dev, int R, int topk, int max_row_len,
                                                int32_t *indices_dev, int64_t indices_ld, uint32_t *score_hist_dev,
                                                void *ws, size_t ws_bytes, int32_t *status_dev, nsa_stream_t stream)
{
    if (!req_offset_dev && R > 0) return NSA_ERR_INVALID_ARG;
    return nsa::topk_launch(logits_dev, logits_ld, row_len_dev, row_to_req_dev, nullptr, 0, nullptr, 0, req_offset_dev,
                            R, topk,
                            max_row_len, indices_dev, indices_ld, score_hist_dev, ws, ws_bytes, status_dev, stream);
}
