// Host-side helpers shared by the library's entry points.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "fp8bs.h"

namespace fp8bs {

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int major = 0;
    int minor = 0;
};

// Current device's properties (cached per device). Returns false if the
// runtime cannot report them.
bool current_device(DeviceInfo* out);

// True when the current device is a compute-capability 10.3 GPU (B300), the
// only target this library is compiled for.
fp8bs_status require_sm103(DeviceInfo* info);

// Device address of the library's error word on the current device (cached
// per device); nullptr if the runtime cannot provide it.
unsigned int* device_error_word();

// The driver's tensor-map encoder (cuTensorMapEncodeTiled), looked up once;
// nullptr if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 get_encoder();

inline bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline fp8bs_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? FP8BS_OK : FP8BS_ERR_CUDA;
}

}  // namespace fp8bs
