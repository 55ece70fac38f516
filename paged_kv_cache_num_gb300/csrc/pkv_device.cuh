// pkv_device.cuh -- small device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {

// Programmatic dependent launch.  A kernel launched with
// launch_pdl may start while the previous kernel of its stream still runs:
// it must call griddep_wait() before touching any global memory that kernel
// may write, and calls griddep_launch_dependents() once the next kernel may
// be scheduled.  Both are no-ops for a normally launched kernel.
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;");
}

__device__ __forceinline__ void raise_err(int32_t *flag, int bits)
{
    if (flag) atomicOr(flag, bits);
}

// 2^x on the SFU (ex2.approx, flush-to-zero); exp(x) = 2^(x*log2 e).
__device__ __forceinline__ float exp2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16-bit element <-> float
template <int KIND> __device__ __forceinline__ float h2f(uint16_t v);
template <> __device__ __forceinline__ float h2f<kF16>(uint16_t v)
{
    return __half2float(__ushort_as_half(v));
}
template <> __device__ __forceinline__ float h2f<kBF16>(uint16_t v)
{
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

template <int KIND> __device__ __forceinline__ uint16_t f2h(float v);
template <> __device__ __forceinline__ uint16_t f2h<kF16>(float v)
{
    return __half_as_ushort(__float2half_rn(v));
}
template <> __device__ __forceinline__ uint16_t f2h<kBF16>(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// e4m3 byte -> float (exact), through the hardware fp8 -> f16 conversion.
__device__ __forceinline__ float e4m3_to_float(uint8_t c)
{
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
    return __half2float(__half(h));
}

// Two e4m3 bytes (low byte first) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two)
{
    __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    return __half22float2(__half2(h2));
}

// Two fp8 bytes of cache kind FP8 (kE4M3 / kE5M2) -> two floats (exact).
template <int FP8>
__device__ __forceinline__ float2 fp8x2_to_float2(uint16_t two)
{
    __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two),
                                                FP8 == kE4M3 ? __NV_E4M3 : __NV_E5M2);
    return __half22float2(__half2(h2));
}

}  // namespace pkv
