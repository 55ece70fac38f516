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

// Two fp8 codes of cache kind FP8 (kE4M3 / kE5M2), bytes 2HI and 2HI+1 of w
// (low byte first) -> two floats, exactly: cvt.rn.f16x2 on the 16-bit half
// of the register, then the f16 -> f32 widening.
template <int FP8, int HI>
__device__ __forceinline__ float2 fp8x2_to_float2(uint32_t w)
{
    uint32_t h;
    if constexpr (FP8 == kE4M3) {
        if constexpr (HI)
            asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}" : "=r"(h) : "r"(w));
        else
            asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.rn.f16x2.e4m3x2 %0, l;\n}" : "=r"(h) : "r"(w));
    } else {
        if constexpr (HI)
            asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.rn.f16x2.e5m2x2 %0, h;\n}" : "=r"(h) : "r"(w));
        else
            asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.rn.f16x2.e5m2x2 %0, l;\n}" : "=r"(h) : "r"(w));
    }
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

}  // namespace pkv
