// KV-cache write side: the rows the sparse attention and the indexer read.
//
// [NSA] / [DSA] set_mla_kv_buffer(layer, loc, k, k_rope) stores the new
// tokens' latent and rope parts at their KV slots; quantize_k_cache turns a
// bf16 cache into the fp8 layout; [DSA] dequantize_k_cache_paged gathers fp8
// rows back to bf16 through a flattened page table.  The indexer keys of the
// new tokens are stored as e4m3 with one fp32 scale per row.
//
// Quantisation of a block of values: scale = (largest magnitude) / 448 in fp32
// (1 for an all-zero block); code = e4m3(value / scale), round to nearest with
// ties to even, saturating.  The fp8 MLA row is 512 latent codes | 4 fp32
// scales (one per 128 latent values) | 64 bf16 rope values (656 bytes).
//
// One warp per row: lane l owns values 4l .. 4l+3 of every 128-value block
// (8-byte loads, 4-byte code stores), the block maximum comes from a warp
// reduction.  HBM-bound; every row is read and written once.
#include "nsa_internal.cuh"

namespace nsa {
namespace {

constexpr int kDl = 512;
constexpr int kDr = 64;
constexpr int kFp8Row = kDl + 4 * (kDl / 128) + 2 * kDr;  // 656
constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Four bf16 values (an 8-byte word) of a 128-value block -> four e4m3 codes and the
// block's scale (every lane of the warp calls it for its own four values).
__device__ __forceinline__ uint32_t quantize4(uint2 w, float &scale)
{
    const float v[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
    const float amax = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint32_t codes = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(v[j], scale), __NV_SATFINITE, __NV_E4M3);
        codes |= (uint32_t)c << (8 * j);
    }
    return codes;
}

// The fp8 row of one token: latent (512 bf16 at `lat`) and rope (64 bf16 at `rope`).
__device__ __forceinline__ void write_fp8_row(const uint16_t *lat, const uint16_t *rope, uint8_t *row, int lane)
{
#pragma unroll
    for (int b = 0; b < kDl / 128; ++b) {
        const uint2 w = *reinterpret_cast<const uint2 *>(lat + 128 * b + 4 * lane);
        float scale;
        const uint32_t codes = quantize4(w, scale);
        *reinterpret_cast<uint32_t *>(row + 128 * b + 4 * lane) = codes;
        if (lane == 0) *reinterpret_cast<float *>(row + kDl + 4 * b) = scale;
    }
    if (lane < 2 * kDr / 16)  // 128 bytes of rope in 16-byte pieces
        *reinterpret_cast<uint4 *>(row + kDl + 4 * (kDl / 128) + 16 * lane) =
            *reinterpret_cast<const uint4 *>(rope + 8 * lane);
}

// The bf16 row of one token (1152 bytes) in 8-byte pieces.
__device__ __forceinline__ void write_bf16_row(const uint16_t *lat, const uint16_t *rope, uint16_t *row, int lane)
{
#pragma unroll
    for (int b = 0; b < kDl / 128; ++b)
        *reinterpret_cast<uint2 *>(row + 128 * b + 4 * lane) = *reinterpret_cast<const uint2 *>(lat + 128 * b + 4 * lane);
    if (lane < kDr / 4)
        *reinterpret_cast<uint2 *>(row + kDl + 4 * lane) = *reinterpret_cast<const uint2 *>(rope + 4 * lane);
}

__global__ void __launch_bounds__(32 * kWarpsPerBlock)
set_mla_kv_kernel(bool fp8, const uint16_t *k_nope, int64_t nope_ld, const uint16_t *k_rope, int64_t rope_ld,
                  const int32_t *loc, int n, uint8_t *kv, int64_t num_slots, int32_t *status)
{
    const int lane = threadIdx.x & 31;
    for (int64_t i = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); i < n;
         i += (int64_t)gridDim.x * kWarpsPerBlock) {
        const int32_t slot = loc[i];
        if (slot < 0 || slot >= num_slots) {
            if (lane == 0) set_status(status, NSA_ERR_BOUNDS);
            continue;
        }
        const uint16_t *lat = k_nope + i * nope_ld, *rope = k_rope + i * rope_ld;
        if (fp8)
            write_fp8_row(lat, rope, kv + (int64_t)slot * kFp8Row, lane);
        else
            write_bf16_row(lat, rope, reinterpret_cast<uint16_t *>(kv) + (int64_t)slot * (kDl + kDr), lane);
    }
}

// A bf16 row held in registers: lane l has latent values 4l .. 4l+3 of each block and
// (lanes 0..7) 16 bytes of the rope.
struct RowRegs {
    uint2 lat[kDl / 128];
    uint4 rope;
};

__device__ __forceinline__ void load_row(const uint16_t *row, int lane, RowRegs &r)
{
#pragma unroll
    for (int b = 0; b < kDl / 128; ++b) r.lat[b] = __ldcs(reinterpret_cast<const uint2 *>(row + 128 * b + 4 * lane));
    if (lane < 2 * kDr / 16) r.rope = __ldcs(reinterpret_cast<const uint4 *>(row + kDl + 8 * lane));
}

__device__ __forceinline__ void store_fp8_row(const RowRegs &r, uint8_t *row, int lane)
{
#pragma unroll
    for (int b = 0; b < kDl / 128; ++b) {
        float scale;
        const uint32_t codes = quantize4(r.lat[b], scale);
        *reinterpret_cast<uint32_t *>(row + 128 * b + 4 * lane) = codes;
        if (lane == 0) *reinterpret_cast<float *>(row + kDl + 4 * b) = scale;
    }
    if (lane < 2 * kDr / 16) *reinterpret_cast<uint4 *>(row + kDl + 4 * (kDl / 128) + 16 * lane) = r.rope;
}

// The whole cache: each warp walks its rows with the next row's loads in flight
// while the current one is quantised and stored.
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
quantize_kv_cache_kernel(const uint16_t *src, int64_t num_slots, uint8_t *dst)
{
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerBlock;
    int64_t s = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (s >= num_slots) return;
    RowRegs cur, nxt;
    load_row(src + s * (kDl + kDr), lane, cur);
    for (; s < num_slots; s += stride) {
        const bool more = s + stride < num_slots;
        if (more) load_row(src + (s + stride) * (kDl + kDr), lane, nxt);
        store_fp8_row(cur, dst + s * kFp8Row, lane);
        if (more) cur = nxt;
    }
}

// Row i of the output = slot slots[i] of the fp8 cache, dequantised (code x scale
// in fp32, rounded to bf16); a negative slot gives a zero row.
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
dequantize_kv_paged_kernel(const uint8_t *kv, int64_t num_slots, const int32_t *slots, int64_t m, uint16_t *out,
                           int32_t *status)
{
    const int lane = threadIdx.x & 31;
    for (int64_t i = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); i < m;
         i += (int64_t)gridDim.x * kWarpsPerBlock) {
        const int32_t slot = slots[i];
        uint16_t *o = out + i * (kDl + kDr);
        if (slot < 0 || slot >= num_slots) {
            if (slot >= num_slots && lane == 0) set_status(status, NSA_ERR_BOUNDS);
#pragma unroll
            for (int b = 0; b < kDl / 128; ++b) *reinterpret_cast<uint2 *>(o + 128 * b + 4 * lane) = make_uint2(0u, 0u);
            if (lane < kDr / 4) *reinterpret_cast<uint2 *>(o + kDl + 4 * lane) = make_uint2(0u, 0u);
            continue;
        }
        const uint8_t *row = kv + (int64_t)slot * kFp8Row;
#pragma unroll
        for (int b = 0; b < kDl / 128; ++b) {
            const uint32_t codes = *reinterpret_cast<const uint32_t *>(row + 128 * b + 4 * lane);
            const float sc = *reinterpret_cast<const float *>(row + kDl + 4 * b);
            uint32_t packed[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)((codes >> (16 * j)) & 0xFFFFu);
                const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
                __nv_bfloat162 b2 = __floats2bfloat162_rn(f.x * sc, f.y * sc);
                packed[j] = *reinterpret_cast<uint32_t *>(&b2);
            }
            *reinterpret_cast<uint2 *>(o + 128 * b + 4 * lane) = make_uint2(packed[0], packed[1]);
        }
        if (lane < kDr / 4)
            *reinterpret_cast<uint2 *>(o + kDl + 4 * lane) =
                *reinterpret_cast<const uint2 *>(row + kDl + 4 * (kDl / 128) + 8 * lane);
    }
}

// Indexer keys: 128 bf16 -> 128 e4m3 codes at k_cache[slot] and one fp32 scale at k_scale[slot].
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
set_index_k_kernel(const uint16_t *k, int64_t k_ld, const int32_t *loc, int n, uint8_t *k_cache, float *k_scale,
                   int64_t num_slots, int32_t *status)
{
    const int lane = threadIdx.x & 31;
    for (int64_t i = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); i < n;
         i += (int64_t)gridDim.x * kWarpsPerBlock) {
        const int32_t slot = loc[i];
        if (slot < 0 || slot >= num_slots) {
            if (lane == 0) set_status(status, NSA_ERR_BOUNDS);
            continue;
        }
        const uint2 w = *reinterpret_cast<const uint2 *>(k + i * k_ld + 4 * lane);
        float scale;
        const uint32_t codes = quantize4(w, scale);
        *reinterpret_cast<uint32_t *>(k_cache + (int64_t)slot * 128 + 4 * lane) = codes;
        if (lane == 0) k_scale[slot] = scale;
    }
}

// Blocks for `rows` rows at one warp a row: up to 8 blocks of 8 warps per SM, the
// kernels grid-striding beyond; 0 when the device's SM count cannot be read.
unsigned rows_grid(int64_t rows)
{
    const int sms = current_sm_count();
    if (sms <= 0) return 0;
    const int64_t blocks = ceil_div(rows, kWarpsPerBlock);
    const int64_t cap = (int64_t)sms * 8;  // 8 blocks of 8 warps per SM, grid-stride beyond
    return (unsigned)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

}  // namespace
}  // namespace nsa

using namespace nsa;

extern "C" nsa_status nsa_set_mla_kv(nsa_dtype kv_dtype, const void *k_nope_dev, int64_t nope_ld,
                                     const void *k_rope_dev, int64_t rope_ld, const int32_t *loc_dev, int n,
                                     int d_latent, int d_rope, void *kv_dev, int64_t num_slots,
                                     int32_t *status_dev, nsa_stream_t stream)
{
    if (kv_dtype != NSA_DT_BF16 && kv_dtype != NSA_DT_E4M3) return NSA_ERR_UNSUPPORTED;
    if (d_latent != kDl || d_rope != kDr) return NSA_ERR_UNSUPPORTED;
    if (n < 0 || num_slots < 0 || nope_ld < kDl || rope_ld < kDr) return NSA_ERR_INVALID_ARG;
    if (n == 0) return NSA_OK;
    if (!k_nope_dev || !k_rope_dev || !loc_dev || !kv_dev) return NSA_ERR_INVALID_ARG;
    if (!aligned(k_nope_dev, 8) || !aligned(k_rope_dev, 16) || !aligned(kv_dev, 16) || nope_ld % 4 || rope_ld % 8)
        return NSA_ERR_INVALID_ARG;
    const unsigned grid = rows_grid(n);
    if (grid == 0) return NSA_ERR_CUDA;
    set_mla_kv_kernel<<<grid, 32 * kWarpsPerBlock, 0, (cudaStream_t)stream>>>(
        kv_dtype == NSA_DT_E4M3, (const uint16_t *)k_nope_dev, nope_ld, (const uint16_t *)k_rope_dev, rope_ld, loc_dev,
        n, (uint8_t *)kv_dev, num_slots, status_dev);
    return launch_status();
}

extern "C" nsa_status nsa_quantize_kv_cache(const void *kv_bf16_dev, int64_t num_slots, int d_latent, int d_rope,
                                            void *kv_fp8_dev, nsa_stream_t stream)
{
    if (d_latent != kDl || d_rope != kDr) return NSA_ERR_UNSUPPORTED;
    if (num_slots < 0) return NSA_ERR_INVALID_ARG;
    if (num_slots == 0) return NSA_OK;
    if (!kv_bf16_dev || !kv_fp8_dev || !aligned(kv_bf16_dev, 16) || !aligned(kv_fp8_dev, 16))
        return NSA_ERR_INVALID_ARG;
    const unsigned grid = rows_grid(num_slots);
    if (grid == 0) return NSA_ERR_CUDA;
    quantize_kv_cache_kernel<<<grid, 32 * kWarpsPerBlock, 0, (cudaStream_t)stream>>>(
        (const uint16_t *)kv_bf16_dev, num_slots, (uint8_t *)kv_fp8_dev);
    return launch_status();
}

extern "C" nsa_status nsa_dequantize_kv_paged(const void *kv_fp8_dev, int64_t num_slots, int d_latent, int d_rope,
                                              const int32_t *slots_dev, int64_t m, void *out_bf16_dev,
                                              int32_t *status_dev, nsa_stream_t stream)
{
    if (d_latent != kDl || d_rope != kDr) return NSA_ERR_UNSUPPORTED;
    if (num_slots < 0 || m < 0) return NSA_ERR_INVALID_ARG;
    if (m == 0) return NSA_OK;
    if (!kv_fp8_dev || !slots_dev || !out_bf16_dev || !aligned(kv_fp8_dev, 16) || !aligned(out_bf16_dev, 16))
        return NSA_ERR_INVALID_ARG;
    const unsigned grid = rows_grid(m);
    if (grid == 0) return NSA_ERR_CUDA;
    dequantize_kv_paged_kernel<<<grid, 32 * kWarpsPerBlock, 0, (cudaStream_t)stream>>>(
        (const uint8_t *)kv_fp8_dev, num_slots, slots_dev, m, (uint16_t *)out_bf16_dev, status_dev);
    return launch_status();
}

extern "C" nsa_status nsa_set_index_k(const void *k_dev, int64_t k_ld, const int32_t *loc_dev, int n, int Di,
                                      void *k_cache_dev, float *k_scale_dev, int64_t num_slots, int32_t *status_dev,
                                      nsa_stream_t stream)
{
    if (Di != 128) return NSA_ERR_UNSUPPORTED;
    if (n < 0 || num_slots < 0 || k_ld < Di) return NSA_ERR_INVALID_ARG;
    if (n == 0) return NSA_OK;
    if (!k_dev || !loc_dev || !k_cache_dev || !k_scale_dev || !aligned(k_dev, 8) || !aligned(k_cache_dev, 4) || k_ld % 4)
        return NSA_ERR_INVALID_ARG;
    const unsigned grid = rows_grid(n);
    if (grid == 0) return NSA_ERR_CUDA;
    set_index_k_kernel<<<grid, 32 * kWarpsPerBlock, 0, (cudaStream_t)stream>>>(
        (const uint16_t *)k_dev, k_ld, loc_dev, n, (uint8_t *)k_cache_dev, k_scale_dev, num_slots, status_dev);
    return launch_status();
}
