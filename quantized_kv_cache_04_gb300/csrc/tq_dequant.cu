// Dequantisation of cached slots back to K and V in the original space.
//
// The inverse of the store for the slots a slot mapping names: FP8 keys are
// decoded as they are; MSE keys are k_hat = k_norm * s . (H c[idx]) with H
// the orthonormal Sylvester Hadamard matrix (the transform is its own
// inverse, so the rotation is undone by the same fast transform the store
// applies, then the sign flips); values are code * v_scale + v_zero.
//
// Method sources: "vllm.v1.attention.backends.turboquant_attn" API page,
// "_continuation_prefill" (the full dequantisation of the cached prefix,
// whose MSE keys are rotated back before attention); "turboquant-plus.md",
// "Background" (the randomized Hadamard rotation and its inverse).
#include "tq.h"
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

struct DqArgs {
    const uint8_t* cache;
    long long nslots;                 // num_blocks * block_size
    int Hk, num_tokens;
    const int64_t* slot_mapping;
    const int8_t* signs;
    const float* centroids;
    void* kout;
    void* vout;
    long long k_stride, v_stride;     // elements per token row of the outputs
    SlotGeom g;
};

constexpr int kDqWarps = 8;           // (token, kv head) pairs per CTA

// Codes of dims 4 lane .. 4 lane + 3 from packed data p (2-byte aligned).
// 4-bit: low nibble first.  3-bit: groups of 32 codes in 12 bytes read as
// words W0..W2; code 8w + i sits in bits 4i..4i+2 of Ww, and bit w of code
// 24 + i in bit 4i + 3 of Ww.
template <int BITS>
__device__ __forceinline__ void lane_codes(const uint8_t* p, int lane, int (&c)[4])
{
    if constexpr (BITS == 4) {
        const uint32_t x = ld_u16(p + 2 * lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = (x >> (4 * i)) & 15;
    } else {
        const uint8_t* grp = p + 12 * (lane >> 3);
        uint32_t W[3];
#pragma unroll
        for (int w = 0; w < 3; ++w) W[w] = uint32_t(ld_u16(grp + 4 * w)) | (uint32_t(ld_u16(grp + 4 * w + 2)) << 16);
        const int j0 = 4 * (lane & 7);          // first code of the lane within its group
        if (j0 < 24) {
            const uint32_t x = W[j0 >> 3] >> (4 * (j0 & 7));
#pragma unroll
            for (int i = 0; i < 4; ++i) c[i] = (x >> (4 * i)) & 7;
        } else {
            const int sh = 4 * (j0 - 24) + 3;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                c[i] = int(((W[0] >> (sh + 4 * i)) & 1) | (((W[1] >> (sh + 4 * i)) & 1) << 1) |
                           (((W[2] >> (sh + 4 * i)) & 1) << 2));
        }
    }
}

template <typename TO>
__device__ __forceinline__ void store4(TO* p, const float (&x)[4])
{
    if constexpr (sizeof(TO) == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    } else {
        TO t[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) t[i] = from_f32<TO>(x[i]);
        *reinterpret_cast<uint2*>(p) = *reinterpret_cast<const uint2*>(t);
    }
}

// One warp per (token, kv head); lane l holds dims 4l .. 4l+3.
// KBITS: 0 = FP8 keys, 3 or 4 = Lloyd-Max keys.  VBITS: 3 or 4.
template <typename TO, int KBITS, int VBITS>
__global__ void __launch_bounds__(32 * kDqWarps) dequant_kernel(DqArgs a)
{
    const int lane = threadIdx.x & 31;
    const long long pair = (long long)blockIdx.x * kDqWarps + (threadIdx.x >> 5);
    if (pair >= (long long)a.num_tokens * a.Hk) return;
    const long long n = pair / a.Hk;
    const int h = int(pair - n * a.Hk);
    TO* ko = static_cast<TO*>(a.kout) + n * a.k_stride + h * kHeadDim + 4 * lane;
    TO* vo = static_cast<TO*>(a.vout) + n * a.v_stride + h * kHeadDim + 4 * lane;
    const long long slot = a.slot_mapping[n];
    float k[4] = {0.f, 0.f, 0.f, 0.f}, v[4] = {0.f, 0.f, 0.f, 0.f};
    if (slot < 0 || slot >= a.nslots) {        // padding: zero rows, nothing read
        store4(ko, k);
        store4(vo, v);
        return;
    }
    const uint8_t* s = a.cache + (slot * a.Hk + h) * a.g.slot;

    if constexpr (KBITS == 0) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(s + 4 * lane);   // slot 196: 4-byte aligned
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>((w >> (8 * i)) & 0xFF),
                                                          __NV_E4M3);
            k[i] = __half2float(__half(hr));
        }
    } else {
        // centroid table in registers: lane j < 2^KBITS holds c[j]
        const float cl = lane < (1 << KBITS) ? a.centroids[lane] : 0.f;
        int c[4];
        lane_codes<KBITS>(s, lane, c);
#pragma unroll
        for (int i = 0; i < 4; ++i) k[i] = __shfl_sync(0xffffffffu, cl, c[i]);
        fwht128_warp(k, lane);                   // H c up to the 1/sqrt(D) factor
        const float norm = __half2float(__ushort_as_half(ld_u16(s + a.g.off_k_norm)));
        const float f = norm * 0.08838834764831845f;
#pragma unroll
        for (int i = 0; i < 4; ++i) k[i] = k[i] * f * float(a.signs[4 * lane + i]);
    }

    {
        const float sc = __half2float(__ushort_as_half(ld_u16(s + a.g.off_v_scale)));
        const float z = __half2float(__ushort_as_half(ld_u16(s + a.g.off_v_zero)));
        int c[4];
        lane_codes<VBITS>(s + a.g.off_v_data, lane, c);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = fmaf(float(c[i]), sc, z);   // code * scale is exact in fp32
    }
    store4(ko, k);
    store4(vo, v);
}

template <typename TO>
cudaError_t launch_dq(const DqArgs& a, unsigned grid, cudaStream_t st)
{
    if (a.g.key_fp8) dequant_kernel<TO, 0, 4><<<grid, 32 * kDqWarps, 0, st>>>(a);
    else if (a.g.key_bits == 4) dequant_kernel<TO, 4, 4><<<grid, 32 * kDqWarps, 0, st>>>(a);
    else if (a.g.value_bits == 4) dequant_kernel<TO, 3, 4><<<grid, 32 * kDqWarps, 0, st>>>(a);
    else dequant_kernel<TO, 3, 3><<<grid, 32 * kDqWarps, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace
}  // namespace tq

extern "C" int tq_dequant(int preset, int head_dim, int num_tokens, int num_kv_heads, int block_size,
                          const uint8_t* kv_cache, long long num_blocks, const int64_t* slot_mapping,
                          const int8_t* signs, const float* centroids, void* key_out, void* value_out,
                          int out_dtype, long long key_stride_tok, long long value_stride_tok,
                          void* stream)
{
    using namespace tq;
    tq_layout L;
    const int rc = fill_layout(preset, head_dim, &L);
    if (rc) return rc;
    if (head_dim != kHeadDim || !block_size_ok(block_size) || !out_dtype_ok(out_dtype))
        return TQ_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 0) return TQ_ERR_INVALID_ARG;
    if (num_tokens == 0) return TQ_OK;
    if (!kv_cache || !slot_mapping || !key_out || !value_out) return TQ_ERR_INVALID_ARG;
    if (!L.key_fp8 && (!signs || !centroids)) return TQ_ERR_INVALID_ARG;
    const long long row = (long long)num_kv_heads * head_dim;
    if (key_stride_tok < row || value_stride_tok < row || key_stride_tok % 8 || value_stride_tok % 8)
        return TQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(key_out) | reinterpret_cast<uintptr_t>(value_out) |
         reinterpret_cast<uintptr_t>(kv_cache)) & 15)
        return TQ_ERR_INVALID_ARG;

    DqArgs a;
    a.cache = kv_cache;
    a.nslots = num_blocks * block_size;
    a.Hk = num_kv_heads;
    a.num_tokens = num_tokens;
    a.slot_mapping = slot_mapping;
    a.signs = signs;
    a.centroids = centroids;
    a.kout = key_out;
    a.vout = value_out;
    a.k_stride = key_stride_tok;
    a.v_stride = value_stride_tok;
    a.g = geom_of(L);
    const long long pairs = (long long)num_tokens * num_kv_heads;
    const long long grid = (pairs + kDqWarps - 1) / kDqWarps;
    if (grid > 0x7fffffffLL) return TQ_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = out_dtype == TQ_F32 ? launch_dq<float>(a, unsigned(grid), st)
                          : out_dtype == TQ_F16 ? launch_dq<__half>(a, unsigned(grid), st)
                                                : launch_dq<__nv_bfloat16>(a, unsigned(grid), st);
    return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
