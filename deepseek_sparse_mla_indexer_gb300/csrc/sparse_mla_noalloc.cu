// nsa_sparse_mla_noalloc: nsa_sparse_mla for callers that cannot allocate
// device memory when they call in (for example a plug-in running inside a
// host framework that owns all device memory and hands it no allocator, or a
// serving loop that forbids allocation after start-up so its memory use stays
// fixed).  Instead of a caller workspace it uses one file-scope device array
// of fixed size for the split-KV partials.
//
// The array is part of this library's device image: every GPU that loads the
// library holds its kNoAllocScratchBytes until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; that first call should come before any stream
// capture.  All calls share the one array and it keeps the last call's
// contents: every element a call reads is written earlier in the same call,
// so nothing needs clearing, but calls that overlap on the GPU (two streams,
// or two threads) race on it and must be serialised by the caller.
#include <mutex>

#include "nsa_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_sparse_mla_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
nsa_status scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return NSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return NSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_sparse_mla_scratch) != cudaSuccess || !p) return NSA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return NSA_OK;
}

}  // namespace

extern "C" nsa_status nsa_sparse_mla_noalloc(nsa_dtype q_dtype, nsa_dtype kv_dtype, const void *q_nope_dev,
                                             int64_t nope_ld_r, int64_t nope_ld_h, const void *q_rope_dev,
                                             int64_t rope_ld_r, int64_t rope_ld_h, const void *kv_dev,
                                             int64_t num_slots, const int32_t *indices_dev, int64_t indices_ld,
                                             int R, int H, int d_latent, int d_rope, int topk, float sm_scale,
                                             void *out_dev, float *lse_dev, int32_t *status_dev,
                                             nsa_stream_t stream)
{
    const size_t need = nsa_sparse_mla_workspace_bytes(q_dtype, kv_dtype, R, H, d_latent, d_rope, topk);
    if (need > kNoAllocScratchBytes) return NSA_ERR_UNSUPPORTED;  // too large for the fixed scratch
    void *scratch = nullptr;
    const nsa_status st = scratch_for_current_device(&scratch);
    if (st != NSA_OK) return st;
    return nsa_sparse_mla(q_dtype, kv_dtype, q_nope_dev, nope_ld_r, nope_ld_h, q_rope_dev, rope_ld_r, rope_ld_h,
                          kv_dev, num_slots, indices_dev, indices_ld, R, H, d_latent, d_rope, topk, sm_scale,
                          out_dev, lse_dev, scratch, kNoAllocScratchBytes, status_dev, stream);
}
