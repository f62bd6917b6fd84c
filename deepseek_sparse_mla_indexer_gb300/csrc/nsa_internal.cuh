// Internal helpers shared by the CUDA sources of the library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/nsa.h"

#define NSA_CUDA_TRY(expr)                                   \
    do {                                                     \
        cudaError_t _e = (expr);                             \
        if (_e != cudaSuccess) return NSA_ERR_CUDA;          \
    } while (0)

namespace nsa {

// Record the first device-side error in the caller's status word (if any).
__device__ __forceinline__ void set_status(int32_t *status, int32_t code)
{
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float e4m3_to_float(uint8_t b)
{
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
    return __half2float(__half(h));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b)
{
    return __uint_as_float(((uint32_t)b) << 16);
}

// Order-preserving 32-bit key of a score: larger scores give larger keys, -0
// folds onto +0 and NaN ranks below every number.  The top-k selects on these
// keys; the indexer histograms their top kScoreDigitBits bits per row.
__device__ __forceinline__ uint32_t order_key(float x)
{
    uint32_t u = __float_as_uint(x);
    if (x != x) return 0u;       // NaN ranks lowest
    if ((u << 1) == 0u) u = 0u;  // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The per-row score histogram shared by the indexer and the top-k: counts of the
// keys' leading kScoreDigitBits bits (kScoreBins uint32 bins per row).
constexpr int kScoreDigitBits = 11;
constexpr int kScoreBins = 1 << kScoreDigitBits;
constexpr int kScoreDigitShift = 32 - kScoreDigitBits;

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Python floor division for the page-table transform (ids are non-negative
// in practice; negative ids keep the pages' `//` meaning).
__device__ __forceinline__ int32_t floor_div(int32_t a, int32_t b)
{
    int32_t q = a / b, r = a % b;
    return (r != 0 && ((r < 0) != (b < 0))) ? q - 1 : q;
}

// Programmatic dependent launch: the step's kernels are launched so that each
// may start while its predecessor on the stream finishes.  A kernel lets its
// dependents launch at entry (pdl_trigger) and, before it reads anything an
// earlier kernel wrote or writes anything an earlier kernel reads, waits for its
// predecessor to complete with its memory visible (pdl_wait).  Both are no-ops
// for a launch without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The launch attribute that allows the overlap.
inline cudaLaunchAttribute pdl_attribute()
{
    cudaLaunchAttribute a = {};
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

// Number of SMs of the current device (0 if it cannot be queried): grids are
// sized from it, never from a fixed count.
inline int current_sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n > 0 ? n : 0;
}

inline nsa_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_CUDA;
}

}  // namespace nsa
