// Library-wide state: the device error word, status strings and the device
// check every entry point runs before launching.
#include <cstdio>
#include <mutex>

#include <cudaTypedefs.h>

#include "fp8bs_device.cuh"
#include "fp8bs_host.h"

namespace fp8bs {

// Set by kernels (atomicOr of DEVERR_* bits); read and cleared by
// fp8bs_last_device_error. One word per device, zero at load time.
__device__ unsigned int g_device_error = 0;

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
unsigned int* g_err_ptr[kMaxDevices];
std::mutex g_info_mu;
}  // namespace

unsigned int* device_error_word()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_info_mu);
    if (g_err_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_err_ptr[dev] = static_cast<unsigned int*>(p);
    }
    return g_err_ptr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

bool current_device(DeviceInfo* out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lock(g_info_mu);
    DeviceInfo& d = g_info[dev];
    if (d.device < 0) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        d.device = dev;
        d.sm_count = prop.multiProcessorCount;
        d.major = prop.major;
        d.minor = prop.minor;
    }
    *out = d;
    return true;
}

fp8bs_status require_sm103(DeviceInfo* info)
{
    if (!current_device(info))
        return FP8BS_ERR_CUDA;
    if (info->major != 10 || info->minor != 3)
        return FP8BS_ERR_UNSUPPORTED;
    return FP8BS_OK;
}

}  // namespace fp8bs

extern "C" const char* fp8bs_status_string(fp8bs_status status)
{
    switch (status) {
    case FP8BS_OK: return "ok";
    case FP8BS_ERR_INVALID_ARG: return "invalid argument";
    case FP8BS_ERR_UNSUPPORTED: return "unsupported shape or device";
    case FP8BS_ERR_CUDA: return "CUDA error";
    case FP8BS_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

namespace {
// Clears exactly the bits that were read, so that a bit set by a kernel on
// another stream after the read is kept for the next call.
__global__ void clear_error_bits(unsigned int* word, unsigned int bits)
{
    atomicAnd(word, ~bits);
}
}  // namespace

extern "C" fp8bs_status fp8bs_last_device_error(fp8bs_stream_t stream)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    unsigned int* word_ptr = fp8bs::device_error_word();
    if (word_ptr == nullptr)
        return FP8BS_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, word_ptr, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    if (word == 0)
        return FP8BS_OK;
    clear_error_bits<<<1, 1, 0, s>>>(word_ptr, word);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    if (word & fp8bs::DEVERR_TIMEOUT)
        return FP8BS_ERR_TIMEOUT;
    return FP8BS_ERR_INVALID_ARG;
}
