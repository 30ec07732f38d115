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
    int Hk, num_tokens, bs;
    const int64_t* slot_mapping;
    const int8_t* signs;
    const float* centroids;
    void* kout;
    void* vout;
    long long k_stride, v_stride;     // elements per token row of the outputs
    SlotGeom g;
};

constexpr int kDqWarps = 8;           // warps per CTA, one token at a time each

// ---------------------------------------------------------------------------
// Two kv heads per warp at a time: the half-warp hw = lane >> 4 takes heads
// of its parity and lane l = lane & 15 their dims 8l .. 8l + 7, so the
// transform takes 4 shuffle stages for two heads at once and every output
// row is one 16-byte (fp16 / bf16) or two (fp32) stores per lane.

template <typename TO>
__device__ __forceinline__ void store8(TO* p, const float (&x)[8])
{
    if constexpr (sizeof(TO) == 4) {
        reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
    } else {
        TO t[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = from_f32<TO>(x[i]);
        *reinterpret_cast<uint4*>(p) = *reinterpret_cast<const uint4*>(t);
    }
}

// The slot bytes a lane needs for its 8 dims of one (token, kv head):
// loaded for two heads per half-warp before either is decoded.
template <int KBITS, int VBITS>
struct Raw8 {
    uint32_t k0, k1;              // key bytes: FP8 8 bytes, else the 16-32 code bits (k0)
    uint32_t v;                   // value code bits
    uint16_t norm, scale, zero;
};

template <int BITS>
__device__ __forceinline__ uint32_t bits8(const uint8_t* p, int l)
{
    if constexpr (BITS == 4) {
        const uint16_t* q = reinterpret_cast<const uint16_t*>(p + 4 * l);
        return uint32_t(q[0]) | (uint32_t(q[1]) << 16);
    } else if constexpr (BITS == 2) {
        return ld_u16(p + 2 * l);
    } else {
        static_assert(BITS == 3, "2, 3 or 4 bits");
        const uint8_t* q = p + 3 * l;
        return uint32_t(q[0]) | (uint32_t(q[1]) << 8) | (uint32_t(q[2]) << 16);
    }
}

template <int KBITS, int VBITS>
__device__ __forceinline__ void load8(const DqArgs& a, const uint8_t* dp, const uint8_t* mp, int l,
                                      Raw8<KBITS, VBITS>& r)
{
    if constexpr (KBITS == 0) {
        const uint16_t* q = reinterpret_cast<const uint16_t*>(dp + 8 * l);
        r.k0 = uint32_t(q[0]) | (uint32_t(q[1]) << 16);
        r.k1 = uint32_t(q[2]) | (uint32_t(q[3]) << 16);
    } else {
        r.k0 = bits8<KBITS>(dp, l);
        r.norm = ld_u16(mp + a.g.m_norm);
    }
    r.v = bits8<VBITS>(dp + a.g.v_off, l);
    r.scale = ld_u16(mp + a.g.m_scale);
    r.zero = ld_u16(mp + a.g.m_zero);
}

template <typename TO, int KBITS, int VBITS>
__device__ __forceinline__ void decode8(const Raw8<KBITS, VBITS>& r, int l, float cl, const float (&sg)[8],
                                        TO* kr, TO* vr, bool live)
{
    float k[8], v[8];
    if constexpr (KBITS == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w = i < 4 ? r.k0 : r.k1;
            const __half_raw hr = __nv_cvt_fp8_to_halfraw(
                static_cast<__nv_fp8_storage_t>((w >> (8 * (i & 3))) & 0xFF), __NV_E4M3);
            k[i] = __half2float(__half(hr));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            k[i] = __shfl_sync(0xffffffffu, cl, (r.k0 >> (KBITS * i)) & ((1u << KBITS) - 1));
        fwht128_half(k, l);                      // H c up to the 1/sqrt(D) factor
        const float f = __half2float(__ushort_as_half(r.norm)) * 0.08838834764831845f;
#pragma unroll
        for (int i = 0; i < 8; ++i) k[i] = k[i] * f * sg[i];
    }
    const float sc = __half2float(__ushort_as_half(r.scale));
    const float z = __half2float(__ushort_as_half(r.zero));
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = fmaf(float((r.v >> (VBITS * i)) & ((1u << VBITS) - 1)), sc, z);   // code * scale is exact in fp32
    if (live) {
        store8(kr, k);
        store8(vr, v);
    }
}

// A warp per token (grid-stride over tokens), two head pairs per step with
// the slot loads of both issued before either is decoded.
template <typename TO, int KBITS, int VBITS>
__global__ void __launch_bounds__(32 * kDqWarps) dequant2_kernel(DqArgs a)
{
    const int lane = threadIdx.x & 31, hw = lane >> 4, l = lane & 15;
    // centroid table in registers: lane j of each half holds c[j]; the lane's signs
    const float cl = (KBITS > 0 && l < (1 << KBITS)) ? a.centroids[l] : 0.f;
    float sg[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sg[i] = KBITS > 0 ? float(a.signs[8 * l + i]) : 1.f;
    const int Hk = a.Hk;
    const int lgbs = 31 - __clz(a.bs);
    const long long nw = (long long)gridDim.x * kDqWarps;
    for (long long n = (long long)blockIdx.x * kDqWarps + (threadIdx.x >> 5); n < a.num_tokens; n += nw) {
        const long long slot = a.slot_mapping[n];
        TO* kbase = static_cast<TO*>(a.kout) + n * a.k_stride + 8 * l;
        TO* vbase = static_cast<TO*>(a.vout) + n * a.v_stride + 8 * l;
        if (slot < 0 || slot >= a.nslots) {       // padding: zero rows, nothing read
            const float zr[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int h = hw; h < Hk; h += 2) {
                store8(kbase + h * kHeadDim, zr);
                store8(vbase + h * kHeadDim, zr);
            }
            continue;
        }
        // (block sizes are powers of two: no division per token)
        const long long page = slot >> lgbs;
        const int off = int(slot & (a.bs - 1));
        for (int h0 = 0; h0 < Hk; h0 += 4) {
            const int ha = h0 + hw, hb = h0 + 2 + hw;      // this half-warp's two heads
            const bool la = ha < Hk, lb = hb < Hk;        // an odd count leaves halves idle
            const uint8_t *dpa, *mpa, *dpb, *mpb;
            slot_ptrs(a.g, a.cache, page, off, la ? ha : 0, a.bs, Hk, dpa, mpa);
            slot_ptrs(a.g, a.cache, page, off, lb ? hb : 0, a.bs, Hk, dpb, mpb);
            Raw8<KBITS, VBITS> ra, rb;
            load8(a, dpa, mpa, l, ra);
            load8(a, dpb, mpb, l, rb);
            decode8<TO>(ra, l, cl, sg, kbase + ha * kHeadDim, vbase + ha * kHeadDim, la);
            decode8<TO>(rb, l, cl, sg, kbase + hb * kHeadDim, vbase + hb * kHeadDim, lb);
        }
    }
}

// One wave of resident CTAs (occupancy of this instantiation on the current
// device, asked once), or fewer when there are fewer tokens.
template <typename TO, int KBITS, int VBITS>
cudaError_t launch_one(const DqArgs& a, long long tokens, cudaStream_t st)
{
    static int resident[64];                 // per device: CTAs per SM x SMs, 0 until asked
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int* res = dev >= 0 && dev < 64 ? &resident[dev] : nullptr;
    int n = res ? *res : 0;
    if (n <= 0) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dequant2_kernel<TO, KBITS, VBITS>,
                                                              32 * kDqWarps, 0);
        if (e != cudaSuccess) return e;
        n = per_sm > 0 && sms > 0 ? per_sm * sms : 1;
        if (res) *res = n;                   // the same value from any thread
    }
    long long grid = (tokens + kDqWarps - 1) / kDqWarps;
    if (grid > n) grid = n;
    dequant2_kernel<TO, KBITS, VBITS><<<unsigned(grid), 32 * kDqWarps, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename TO>
cudaError_t launch_dq(const DqArgs& a, long long tokens, cudaStream_t st)
{
    if (a.g.key_fp8) return launch_one<TO, 0, 4>(a, tokens, st);
    if (a.g.key_bits == 4) return launch_one<TO, 4, 4>(a, tokens, st);
    if (a.g.key_bits == 2) return launch_one<TO, 2, 2>(a, tokens, st);
    if (a.g.value_bits == 4) return launch_one<TO, 3, 4>(a, tokens, st);
    return launch_one<TO, 3, 3>(a, tokens, st);
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
    a.bs = block_size;
    a.g = geom_of(L, is_soa(preset));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = out_dtype == TQ_F32 ? launch_dq<float>(a, num_tokens, st)
                          : out_dtype == TQ_F16 ? launch_dq<__half>(a, num_tokens, st)
                                                : launch_dq<__nv_bfloat16>(a, num_tokens, st);
    return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
