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

extern "C" int nsa_abi_version(void) { return 100; }

extern "C" nsa_status nsa_status_read(const int32_t *status_dev, int32_t *host_value, nsa_stream_t stream)
{
    if (!status_dev || !host_value) return NSA_ERR_INVALID_ARG;
    NSA_CUDA_TRY(cudaMemcpyAsync(host_value, status_dev, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                 (cudaStream_t)stream));
    NSA_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
    return NSA_OK;
}
