// dtype_load.cuh -- exact widening of stored elements to fp32 on the device.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace lik {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ float load_f32(const T* p) {
    return to_f32(*p);
}

}  // namespace lik
