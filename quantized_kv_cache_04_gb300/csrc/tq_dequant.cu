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

// Raw packed codes of the lane's 4 dims (every width an LSB-first
// bitstream): 4-bit: one 16-bit word; 2-bit: one byte; 3-bit: the 16 bits
// from byte 3*lane/2, whose low 12 (lane even) or high 12 (lane odd) bits
// are the lane's codes.  Loaded in a first phase so that the loads of
// several pairs are in flight together.
template <int BITS>
struct RawCodes {
    uint32_t w[1];
};

template <int BITS>
__device__ __forceinline__ void load_codes(const uint8_t* p, int lane, RawCodes<BITS>& r)
{
    if constexpr (BITS == 2) {
        r.w[0] = p[lane];
    } else if constexpr (BITS == 4) {
        r.w[0] = ld_u16(p + 2 * lane);
    } else {
        const uint8_t* q = p + ((3 * lane) >> 1);
        r.w[0] = uint32_t(q[0]) | (uint32_t(q[1]) << 8);
    }
}

// Codes of dims 4 lane .. 4 lane + 3.
template <int BITS>
__device__ __forceinline__ void lane_codes(const RawCodes<BITS>& r, int lane, int (&c)[4])
{
    if constexpr (BITS == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = (r.w[0] >> (2 * i)) & 3;
    } else if constexpr (BITS == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = (r.w[0] >> (4 * i)) & 15;
    } else {
        const uint32_t x = r.w[0] >> (4 * (lane & 1));
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = (x >> (3 * i)) & 7;
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

// The slot bytes one lane needs for its 4 dims of one (token, kv head).
// KBITS: 0 = FP8 keys, 2, 3 or 4 = Lloyd-Max keys.  VBITS: 2, 3 or 4.
template <int KBITS, int VBITS>
struct PairRaw {
    uint32_t kw;                  // FP8 keys: the lane's 4 key bytes
    RawCodes<KBITS == 0 ? 4 : KBITS> kc;
    RawCodes<VBITS> vc;
    uint16_t norm, scale, zero;
};

// s: the record's data (key data at 0, value data at v_off); m: its metadata
// (the slot itself for AoS).
template <int KBITS, int VBITS>
__device__ __forceinline__ void load_pair(const DqArgs& a, const uint8_t* s, const uint8_t* m, int lane,
                                          PairRaw<KBITS, VBITS>& r)
{
    if constexpr (KBITS == 0) {
        r.kw = *reinterpret_cast<const uint32_t*>(s + 4 * lane);   // slot 196 / record 192: 4-byte aligned
    } else {
        load_codes<KBITS>(s, lane, r.kc);
        r.norm = ld_u16(m + a.g.m_norm);
    }
    load_codes<VBITS>(s + a.g.v_off, lane, r.vc);
    r.scale = ld_u16(m + a.g.m_scale);
    r.zero = ld_u16(m + a.g.m_zero);
}

// Lane l of the warp writes dims 4l .. 4l+3 of one kv head's K and V rows.
template <typename TO, int KBITS, int VBITS>
__device__ __forceinline__ void finish_pair(const DqArgs& a, TO* ko, TO* vo, int lane, float cl,
                                            const float (&sg4)[4], const PairRaw<KBITS, VBITS>& r)
{
    float k[4], v[4];
    if constexpr (KBITS == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half_raw hr = __nv_cvt_fp8_to_halfraw(
                static_cast<__nv_fp8_storage_t>((r.kw >> (8 * i)) & 0xFF), __NV_E4M3);
            k[i] = __half2float(__half(hr));
        }
    } else {
        int c[4];
        lane_codes<KBITS>(r.kc, lane, c);
#pragma unroll
        for (int i = 0; i < 4; ++i) k[i] = __shfl_sync(0xffffffffu, cl, c[i]);
        fwht128_warp(k, lane);                   // H c up to the 1/sqrt(D) factor
        const float f = __half2float(__ushort_as_half(r.norm)) * 0.08838834764831845f;
#pragma unroll
        for (int i = 0; i < 4; ++i) k[i] = k[i] * f * sg4[i];
    }
    {
        const float sc = __half2float(__ushort_as_half(r.scale));
        const float z = __half2float(__ushort_as_half(r.zero));
        int c[4];
        lane_codes<VBITS>(r.vc, lane, c);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = fmaf(float(c[i]), sc, z);   // code * scale is exact in fp32
    }
    store4(ko + 4 * lane, k);
    store4(vo + 4 * lane, v);
}

// Warps stride over tokens; a warp does every kv head of its token, two
// heads per step with the slot loads of both issued before either is decoded.
template <typename TO, int KBITS, int VBITS>
__global__ void __launch_bounds__(32 * kDqWarps) dequant_kernel(DqArgs a)
{
    const int lane = threadIdx.x & 31;
    const long long nw = (long long)gridDim.x * kDqWarps;
    // centroid table in registers: lane j < 2^KBITS holds c[j]; the lane's signs
    const float cl = (KBITS > 0 && lane < (1 << KBITS)) ? a.centroids[lane] : 0.f;
    float sg4[4] = {1.f, 1.f, 1.f, 1.f};
    if constexpr (KBITS > 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) sg4[i] = float(a.signs[4 * lane + i]);
    }
    const int Hk = a.Hk, S = a.g.slot;
    for (long long n = (long long)blockIdx.x * kDqWarps + (threadIdx.x >> 5); n < a.num_tokens; n += nw) {
        const long long slot = a.slot_mapping[n];
        TO* kr = static_cast<TO*>(a.kout) + n * a.k_stride;
        TO* vr = static_cast<TO*>(a.vout) + n * a.v_stride;
        if (slot < 0 || slot >= a.nslots) {     // padding: zero rows, nothing read
            const float z[4] = {0.f, 0.f, 0.f, 0.f};
            for (int h = 0; h < Hk; ++h) {
                store4(kr + h * kHeadDim + 4 * lane, z);
                store4(vr + h * kHeadDim + 4 * lane, z);
            }
            continue;
        }
        // the token's records: data at dbase + h * ds, metadata at mbase + h * ms
        const uint8_t *dbase, *mbase;
        slot_ptrs(a.g, a.cache, slot / a.bs, int(slot % a.bs), 0, a.bs, Hk, dbase, mbase);
        const int ds = a.g.soa ? a.g.data_bytes : S, ms = a.g.soa ? a.g.meta_bytes : S;
        int h = 0;
        for (; h + 1 < Hk; h += 2) {
            PairRaw<KBITS, VBITS> r0, r1;
            load_pair(a, dbase + h * ds, mbase + h * ms, lane, r0);
            load_pair(a, dbase + (h + 1) * ds, mbase + (h + 1) * ms, lane, r1);
            finish_pair<TO>(a, kr + h * kHeadDim, vr + h * kHeadDim, lane, cl, sg4, r0);
            finish_pair<TO>(a, kr + (h + 1) * kHeadDim, vr + (h + 1) * kHeadDim, lane, cl, sg4, r1);
        }
        if (h < Hk) {
            PairRaw<KBITS, VBITS> r0;
            load_pair(a, dbase + h * ds, mbase + h * ms, lane, r0);
            finish_pair<TO>(a, kr + h * kHeadDim, vr + h * kHeadDim, lane, cl, sg4, r0);
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
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dequant_kernel<TO, KBITS, VBITS>,
                                                              32 * kDqWarps, 0);
        if (e != cudaSuccess) return e;
        n = per_sm > 0 && sms > 0 ? per_sm * sms : 1;
        if (res) *res = n;                   // the same value from any thread
    }
    long long grid = (tokens + kDqWarps - 1) / kDqWarps;
    if (grid > n) grid = n;
    dequant_kernel<TO, KBITS, VBITS><<<unsigned(grid), 32 * kDqWarps, 0, st>>>(a);
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
