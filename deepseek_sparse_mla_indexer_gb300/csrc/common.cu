// Status strings, ABI version and the status-word read-back.
#include "nsa_internal.cuh"

extern "C" const char *nsa_status_string(int status)
{
    switch (status) {
    case NSA_OK: return "ok";
    case NSA_ERR_INVALID_ARG: return "invalid argument";
    case NSA_ERR_UNSUPPORTED: return "unsupported dtype or shape";
    case NSA_ERR_CUDA: return "CUDA error";
    case NSA_ERR_BOUNDS: return "index, page id or length out of range (device-detected)";
    case NSA_ERR_TIMEOUT: return "bounded device wait timed out";
    default: return "unknown status";
    }
}

extern "C" int nsa_abi_version(void) { return 102; }

extern "C" nsa_status nsa_status_read(const int32_t *status_dev, int32_t *host_value, nsa_stream_t stream)
{
    if (!status_dev || !host_value) return NSA_ERR_INVALID_ARG;
    NSA_CUDA_TRY(cudaMemcpyAsync(host_value, status_dev, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                 (cudaStream_t)stream));
    NSA_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
    return NSA_OK;
}

// ---------------------------------------------------------------- several copies in one launch
namespace nsa {
namespace {

constexpr int kMaxCopies = 16;

// Device memory, managed memory, or pinned host memory mapped at the same address.
bool device_addressable(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return true;
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

struct CopyList {
    const uint8_t *src[kMaxCopies];
    uint8_t *dst[kMaxCopies];
    int64_t bytes[kMaxCopies];
    int64_t start[kMaxCopies + 1];  // running byte offsets: copy i covers [start[i], start[i+1])
    int n;
    int vec;  // every address and size a multiple of 16
};

// Grid-stride over the concatenated bytes of all copies, 16 bytes per thread and
// step when every buffer allows it.  Host pointers must be device-accessible
// (pinned, mapped into the unified address space).
__global__ void __launch_bounds__(256) copy_buffers_kernel(CopyList c)
{
    const int64_t total = c.start[c.n];
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    if (c.vec) {
        int i = 0;
        for (int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 16; g < total; g += step * 16) {
            while (g >= c.start[i + 1]) ++i;
            while (g < c.start[i]) --i;
            const int64_t o = g - c.start[i];
            *reinterpret_cast<uint4 *>(c.dst[i] + o) = *reinterpret_cast<const uint4 *>(c.src[i] + o);
        }
    } else {
        int i = 0;
        for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += step) {
            while (g >= c.start[i + 1]) ++i;
            while (g < c.start[i]) --i;
            const int64_t o = g - c.start[i];
            c.dst[i][o] = c.src[i][o];
        }
    }
}

}  // namespace
}  // namespace nsa

extern "C" nsa_status nsa_copy_buffers(int n, const void *const *src, void *const *dst, const int64_t *bytes,
                                       nsa_stream_t stream)
{
    using namespace nsa;
    if (n < 0 || n > kMaxCopies || (n > 0 && (!src || !dst || !bytes))) return NSA_ERR_INVALID_ARG;
    CopyList c = {};
    c.n = n;
    c.vec = 1;
    c.start[0] = 0;
    for (int i = 0; i < n; ++i) {
        if (bytes[i] < 0 || (bytes[i] > 0 && (!src[i] || !dst[i]))) return NSA_ERR_INVALID_ARG;
        if (bytes[i] > 0 && (!device_addressable(src[i]) || !device_addressable(dst[i]))) return NSA_ERR_INVALID_ARG;
        c.src[i] = (const uint8_t *)src[i];
        c.dst[i] = (uint8_t *)dst[i];
        c.bytes[i] = bytes[i];
        c.start[i + 1] = c.start[i] + bytes[i];
        if (((uintptr_t)src[i] | (uintptr_t)dst[i] | (uintptr_t)bytes[i]) & 15) c.vec = 0;
    }
    const int64_t total = c.start[n];
    if (total == 0) return NSA_OK;
    const int sms = current_sm_count();
    if (sms <= 0) return NSA_ERR_CUDA;
    const int64_t units = c.vec ? ceil_div(total, 16) : total;
    int64_t blocks = ceil_div(units, 256);
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    copy_buffers_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(c);
    return launch_status();
}
