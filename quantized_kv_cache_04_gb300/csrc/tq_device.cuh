// Device helpers shared by the TurboQuant CUDA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace tq {

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int m = 16; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

__device__ __forceinline__ float warp_min(float v)
{
#pragma unroll
    for (int m = 16; m; m >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// Unnormalised Walsh-Hadamard transform (natural/Sylvester order) of a
// 128-vector held 4 consecutive elements per lane: element 4*lane + i is v[i].
// Element index bits 0-1 live inside the lane, bits 2-6 are the lane bits.
// Each butterfly maps (x_lo, x_hi) -> (x_lo + x_hi, x_lo - x_hi).
__device__ __forceinline__ void fwht128_warp(float (&v)[4], int lane)
{
    float a = v[0] + v[1], b = v[0] - v[1], c = v[2] + v[3], d = v[2] - v[3];
    v[0] = a + c; v[2] = a - c; v[1] = b + d; v[3] = b - d;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = lane & m;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float p = __shfl_xor_sync(0xffffffffu, v[i], m);
            v[i] = upper ? (p - v[i]) : (v[i] + p);
        }
    }
}

// Unnormalised Sylvester Walsh-Hadamard transform of a 128-vector held 8
// consecutive elements per lane of a half-warp (element 8l + i is v[i]):
// index bits 0-2 inside the lane, bits 3-6 across lanes.  Each butterfly
// maps (x_lo, x_hi) -> (x_lo + x_hi, x_lo - x_hi); across lanes the upper
// partner computes fma(x, -1, p) = p - x and the lower fma(x, 1, p) = x + p.
__device__ __forceinline__ void fwht128_half(float (&v)[8], int l)
{
#pragma unroll
    for (int b = 1; b < 8; b <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (!(i & b)) {
                const float x = v[i], y = v[i + b];
                v[i] = x + y;
                v[i + b] = x - y;
            }
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) {
        const float sg = (l & m) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float p = __shfl_xor_sync(0xffffffffu, v[i], m);
            v[i] = __fmaf_rn(v[i], sg, p);
        }
    }
}

__device__ __forceinline__ uint16_t ld_u16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }

}  // namespace tq
