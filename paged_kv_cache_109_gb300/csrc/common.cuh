// common.cuh -- shared definitions of the decode/write kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa.h"

namespace pa {

// Device error word (PA_DEVERR_* bits).  One per library; kernels OR bits in,
// pa_last_device_error() reads and clears it.
__device__ unsigned int g_device_error;

__device__ __forceinline__ void raise_error(unsigned int bit) {
    atomicOr(&g_device_error, bit);
}

// Bound on any single pipeline wait, in SM clocks (about one second).
constexpr long long kWaitLimitCycles = 2000000000LL;

constexpr float kLog2e = 1.4426950408889634f;

template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static __device__ __forceinline__ float to_float(float x) { return x; }
    static __device__ __forceinline__ float from_float(float x) { return x; }
};

template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_float(__nv_bfloat16 x) {
        return __bfloat162float(x);
    }
    static __device__ __forceinline__ __nv_bfloat16 from_float(float x) {
        return __float2bfloat16_rn(x);
    }
};

}  // namespace pa
