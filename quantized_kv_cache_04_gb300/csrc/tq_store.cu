// Fused quantising store of new K/V tokens into the combined paged cache.
//
// Method: "turboquant-plus.md" (Atlas TQ+), section "Background" (randomised
// Hadamard rotation, Lloyd-Max codebook, matched-norm L2 scale, 3-bit packing
// of 8 codes per 3 bytes; every code stream is LSB-first);
// "vllm.v1.attention.backends.turboquant_attn" API page, sections "_store_kv"
// and "do_kv_cache_update" (fused store of K and V into one slot per (block,
// token, kv head)).
//
// Mapping: one CTA per token (grid-stride), one warp per kv head, 4 consecutive
// coordinates per lane.  The rotation is a warp-shuffle Walsh-Hadamard
// transform in registers; the bucketize is a branch-free binary search over
// midpoints in shared memory; each warp writes its slot straight into the
// cache (the SoA convention stages the token's slots in shared memory and
// scatters their data and metadata records).  Warps of a CTA do not wait
// for each other in the AoS form.
// The value path uses explicitly rounded fp32 operations so the stored bytes
// are reproducible bit for bit.
#include "tq.h"
#include "tq_device.cuh"
#include "tq_internal.h"

#include <atomic>
#include <type_traits>

namespace tq {
namespace {

struct StoreArgs {
    const void* key;
    const void* value;
    long long key_stride, value_stride;   // elements between tokens
    const int64_t* slot_mapping;
    uint8_t* cache;
    long long num_slots;                  // num_blocks * block_size
    const int8_t* signs;
    const float* centroids;
    const float* midpoints;
    int num_tokens, num_kv_heads;
    int slot_size;                        // unpadded
    int bs;                               // block_size (SoA record positions)
    int vec;                              // 1: K and V rows of a head are 8-byte aligned
    SlotGeom g;
};

// The 4 input elements of lane `lane` for (token n, head h): one 8-byte load
// when the rows are 8-byte aligned, else four 2-byte loads.
template <typename T>
__device__ __forceinline__ uint2 load4(const T* base, long long stride, int n, int h, int lane, bool vec)
{
    const T* p = base + n * stride + (long long)h * kHeadDim + 4 * lane;
    if (vec) return *reinterpret_cast<const uint2*>(p);
    const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
    return make_uint2(uint32_t(q[0]) | uint32_t(q[1]) << 16, uint32_t(q[2]) | uint32_t(q[3]) << 16);
}

template <typename T>
__device__ __forceinline__ void unpack4(uint2 r, float (&x)[4])
{
    const uint16_t u[4] = {uint16_t(r.x), uint16_t(r.x >> 16), uint16_t(r.y), uint16_t(r.y >> 16)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (std::is_same<T, __half>::value) x[i] = __half2float(__ushort_as_half(u[i]));
        else x[i] = __bfloat162float(__ushort_as_bfloat16(u[i]));
    }
}

// Pack the 4 codes of every lane (code 4*lane+i = c[i]) as a BITS-wide
// LSB-first bitstream starting at dst (2-byte aligned).  All lanes of the warp
// take part.  Every shared-memory write is an aligned 16-bit store.
template <int BITS>
__device__ __forceinline__ void pack_codes(uint8_t* dst, const int (&c)[4], int lane)
{
    const uint32_t w = uint32_t(c[0]) | uint32_t(c[1]) << BITS | uint32_t(c[2]) << (2 * BITS) |
                       uint32_t(c[3]) << (3 * BITS);
    uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
    if constexpr (BITS == 4) {
        d16[lane] = uint16_t(w);
    } else if constexpr (BITS == 2) {   // lane pairs form 16 bits
        const uint32_t hi = __shfl_down_sync(0xffffffffu, w, 1);
        if (!(lane & 1)) d16[lane >> 1] = uint16_t(w | (hi << 8));
    } else {
        // 3 bits: lanes 4g..4g+3 hold codes 16g..16g+15, 48 bits = three
        // aligned 16-bit words at word 3g; lane 4g+j (j < 3) writes word j,
        // bits [16j, 16j+16) of the group, from its own 12 bits and the next
        // lane's
        static_assert(BITS == 3, "2, 3 or 4 bits");
        const uint32_t nxt = __shfl_down_sync(0xffffffffu, w, 1);
        const int j = lane & 3;
        if (j < 3) d16[3 * (lane >> 2) + j] = uint16_t((w >> (4 * j)) | (nxt << (12 - 4 * j)));
    }
}

__device__ __forceinline__ void put_u16(uint8_t* p, uint16_t v)
{
    *reinterpret_cast<uint16_t*>(p) = v;   // p is 2-byte aligned: slots and fields are even
}

template <typename T, bool KEY_FP8, int KBITS, int VBITS, bool NORM_CORR>
__global__ void __launch_bounds__(1024) store_kernel(StoreArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float s_cent[16], s_mid[16];
    // a decode launched next as a programmatic dependent may start its
    // prologue now; it waits for this grid's completion before reading memory
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31, h = threadIdx.x >> 5;
    const int S = a.g.slot;
    const int row_bytes = a.num_kv_heads * S;

    if constexpr (!KEY_FP8) {
        constexpr int NC = 1 << KBITS;
        if (threadIdx.x < NC) s_cent[threadIdx.x] = a.centroids[threadIdx.x];
        if (threadIdx.x < NC - 1) s_mid[threadIdx.x] = a.midpoints[threadIdx.x];
    }
    float sgn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sgn[i] = float(a.signs[4 * lane + i]);
    __syncthreads();

    const T* K = static_cast<const T*>(a.key);
    const T* V = static_cast<const T*>(a.value);
    const bool vec = a.vec != 0;

    // The inputs and slots of the next two tokens are in flight while this
    // one is encoded.
    int n = blockIdx.x;
    uint2 kr[2], vr[2];
    long long sl[2] = {-1, -1};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int m = n + u * gridDim.x;
        kr[u] = vr[u] = make_uint2(0u, 0u);
        if (m < a.num_tokens) {
            kr[u] = load4(K, a.key_stride, m, h, lane, vec);
            vr[u] = load4(V, a.value_stride, m, h, lane, vec);
            sl[u] = a.slot_mapping[m];
        }
    }
    for (; n < a.num_tokens; n += gridDim.x) {
        const long long slot_idx = sl[0];
        float k[4], v[4];
        unpack4<T>(kr[0], k);
        unpack4<T>(vr[0], v);
        kr[0] = kr[1];
        vr[0] = vr[1];
        sl[0] = sl[1];
        const int nn = n + 2 * gridDim.x;
        if (nn < a.num_tokens) {
            kr[1] = load4(K, a.key_stride, nn, h, lane, vec);
            vr[1] = load4(V, a.value_stride, nn, h, lane, vec);
            sl[1] = a.slot_mapping[nn];
        }
        if (slot_idx < 0 || slot_idx >= a.num_slots) continue;   // uniform across the CTA
        // AoS: each warp writes its slot straight to the cache (the token's
        // Hk slots are one contiguous row); SoA: slots are staged in shared
        // memory and scattered by the CTA
        const bool soa = a.g.soa;
        uint8_t* row = smem;
        uint8_t* dst = soa ? row + h * S : a.cache + slot_idx * (long long)row_bytes + h * S;

        // ---------------- keys
        if constexpr (KEY_FP8) {
            uint32_t b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) b[i] = __nv_cvt_float_to_fp8(k[i], __NV_SATFINITE, __NV_E4M3);
            uint16_t* d16 = reinterpret_cast<uint16_t*>(dst + 4 * lane);
            d16[0] = uint16_t(b[0] | (b[1] << 8));
            d16[1] = uint16_t(b[2] | (b[3] << 8));
        } else {
            const float n2 = warp_sum(k[0] * k[0] + k[1] * k[1] + k[2] * k[2] + k[3] * k[3]);
            const float nrm = __fsqrt_rn(n2);
            float x[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = sgn[i] * k[i];
            fwht128_warp(x, lane);
            // y = H(s.k)/||k|| with H = Sylvester / sqrt(128)
            const float inv = nrm > 0.f ? __fdiv_rn(0.08838834764831845f, nrm) : 0.f;
            int idx[4];
            float cn = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float y = x[i] * inv;
                int j = 0;
#pragma unroll
                for (int step = 1 << (KBITS - 1); step; step >>= 1)
                    if (y > s_mid[j + step - 1]) j += step;
                idx[i] = j;
                const float c = s_cent[j];
                cn += c * c;
            }
            cn = warp_sum(cn);
            const float stored = NORM_CORR ? __fdiv_rn(nrm, __fsqrt_rn(cn)) : nrm;
            pack_codes<KBITS>(dst, idx, lane);
            if (lane == 0) put_u16(dst + a.g.off_k_norm, __half_as_ushort(__float2half_rn(stored)));
        }

        // ---------------- values: asymmetric min/max uniform codes
        {
            constexpr int QMAX = (1 << VBITS) - 1;
            const float lo = warp_min(fminf(fminf(v[0], v[1]), fminf(v[2], v[3])));
            const float hi = warp_max(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])));
            const __half scale16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), float(QMAX)));
            const __half zero16 = __float2half_rn(lo);
            const float sc = __half2float(scale16), z = __half2float(zero16);
            // code = rint((v - z) / sc) with the division correctly rounded.
            // For quotients below 16, t * fl(1/sc) is within 2^-19 of the
            // correctly rounded one (three roundings of at most 2^-24
            // relative), so both take the same rint unless t * fl(1/sc) lies
            // within 2^-16 of a half-integer, where the exact division
            // decides; larger quotients clamp to QMAX either way.
            const float rsc = sc > 0.f ? __frcp_rn(sc) : 0.f;
            int code[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float r = 0.f;
                if (sc > 0.f) {
                    const float t = __fsub_rn(v[i], z);
                    float q = __fmul_rn(t, rsc);
                    if (fabsf(q - (floorf(q) + 0.5f)) < 0x1p-16f) q = __fdiv_rn(t, sc);
                    r = fminf(fmaxf(rintf(q), 0.f), float(QMAX));
                }
                code[i] = int(r);
            }
            pack_codes<VBITS>(dst + a.g.off_v_data, code, lane);
            if (lane == 0) {
                put_u16(dst + a.g.off_v_scale, __half_as_ushort(scale16));
                put_u16(dst + a.g.off_v_zero, __half_as_ushort(zero16));
                if (a.slot_size < S) dst[S - 1] = 0;
            }
        }
        if (!soa) continue;
        __syncthreads();

        // ---------------- SoA: the token's Hk data records and Hk metadata
        // records from the staged slots
        {
            const int Hk = a.num_kv_heads, kd = a.g.key_data_bytes;
            const long long page = slot_idx >> (31 - __clz(a.bs));    // block sizes are powers of two
            const int off = int(slot_idx & (a.bs - 1));
            uint8_t* blk = a.cache + page * a.bs * (long long)row_bytes;
            uint16_t* dd = reinterpret_cast<uint16_t*>(blk + (long long)off * Hk * a.g.data_bytes);
            uint16_t* md = reinterpret_cast<uint16_t*>(blk + (long long)a.bs * Hk * a.g.data_bytes +
                                                       (long long)off * Hk * a.g.meta_bytes);
            // warp hh moves head hh's records (one warp per kv head)
            const int dh = a.g.data_bytes / 2, mh = a.g.meta_bytes / 2;
            const int hh = threadIdx.x >> 5, ln = threadIdx.x & 31;
            for (int i = ln; i < dh; i += 32) {
                const int j = 2 * i;
                const int src = hh * S + (j < kd ? j : a.g.off_v_data + (j - kd));
                dd[hh * dh + i] = *reinterpret_cast<const uint16_t*>(row + src);
            }
            if (ln < mh) {
                const int f = ln;
                const int fo = a.g.key_fp8 ? (f == 0 ? a.g.off_v_scale : a.g.off_v_zero)
                                           : (f == 0 ? a.g.off_k_norm : f == 1 ? a.g.off_v_scale : a.g.off_v_zero);
                md[hh * mh + f] = *reinterpret_cast<const uint16_t*>(row + hh * S + fo);
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// The AoS store with two kv heads per warp (even kv-head counts): half-warp
// hw = lane >> 4 takes head 2 * warp + hw, lane l = lane & 15 its dims
// 8l .. 8l + 7.  Against a warp per head this halves the reductions' and the
// scalar steps' instructions per head (one instruction serves both halves)
// and takes the transform in 3 local and 4 shuffle stages instead of 2 and 5.

// Sum / min / max over the 16 lanes of a half-warp.
__device__ __forceinline__ float half_sum(float v)
{
#pragma unroll
    for (int m = 8; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}
__device__ __forceinline__ float half_min(float v)
{
#pragma unroll
    for (int m = 8; m; m >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}
__device__ __forceinline__ float half_max(float v)
{
#pragma unroll
    for (int m = 8; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// The 8 input elements of lane l of half-warp head h for token n: 16-byte
// loads when rows are 16-byte aligned (vec 2), 8-byte (vec 1), else 2-byte.
template <typename T>
__device__ __forceinline__ uint4 load8(const T* base, long long stride, int n, int h, int l, int vec)
{
    const T* p = base + n * stride + (long long)h * kHeadDim + 8 * l;
    if (vec == 2) return *reinterpret_cast<const uint4*>(p);
    if (vec == 1) {
        const uint2 a = reinterpret_cast<const uint2*>(p)[0], b = reinterpret_cast<const uint2*>(p)[1];
        return make_uint4(a.x, a.y, b.x, b.y);
    }
    const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
    return make_uint4(uint32_t(q[0]) | uint32_t(q[1]) << 16, uint32_t(q[2]) | uint32_t(q[3]) << 16,
                      uint32_t(q[4]) | uint32_t(q[5]) << 16, uint32_t(q[6]) | uint32_t(q[7]) << 16);
}

template <typename T>
__device__ __forceinline__ void unpack8(uint4 r, float (&x)[8])
{
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint16_t u = uint16_t(w[i >> 1] >> (16 * (i & 1)));
        if constexpr (std::is_same<T, __half>::value) x[i] = __half2float(__ushort_as_half(u));
        else x[i] = __bfloat162float(__ushort_as_bfloat16(u));
    }
}

// The 8 codes of lane l (code 8l + i = c[i]) as a BITS-wide LSB-first
// bitstream at dst (2-byte aligned); all 16 lanes of the half take part.
template <int BITS>
__device__ __forceinline__ void pack8(uint8_t* dst, const int (&c)[8], int l)
{
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) w |= uint32_t(c[i]) << (BITS * i);
    uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
    if constexpr (BITS == 4) {
        d16[2 * l] = uint16_t(w);
        d16[2 * l + 1] = uint16_t(w >> 16);
    } else if constexpr (BITS == 2) {
        d16[l] = uint16_t(w);
    } else {
        // lanes 2m, 2m + 1: 48 bits = three aligned 16-bit words at word 3m
        static_assert(BITS == 3, "2, 3 or 4 bits");
        const uint32_t nxt = __shfl_down_sync(0xffffffffu, w, 1);
        if (!(l & 1)) {
            d16[3 * (l >> 1)] = uint16_t(w);
            d16[3 * (l >> 1) + 1] = uint16_t((w >> 16) | (nxt << 8));
        } else {
            d16[3 * (l >> 1) + 2] = uint16_t(w >> 8);
        }
    }
}

template <typename T, bool KEY_FP8, int KBITS, int VBITS, bool NORM_CORR>
__global__ void __launch_bounds__(512) store2_kernel(StoreArgs a)
{
    __shared__ float s_cent[16], s_mid[16];
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31, hw = lane >> 4, l = lane & 15;
    const int h = 2 * (threadIdx.x >> 5) + hw;
    const int S = a.g.slot;
    const int row_bytes = a.num_kv_heads * S;

    if constexpr (!KEY_FP8) {
        constexpr int NC = 1 << KBITS;
        if (threadIdx.x < NC) s_cent[threadIdx.x] = a.centroids[threadIdx.x];
        if (threadIdx.x < NC - 1) s_mid[threadIdx.x] = a.midpoints[threadIdx.x];
    }
    float sgn[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sgn[i] = float(a.signs[8 * l + i]);
    __syncthreads();

    const T* K = static_cast<const T*>(a.key);
    const T* V = static_cast<const T*>(a.value);
    const int vec = a.vec;

    // the inputs and slots of the next two tokens are in flight while this
    // one is encoded
    int n = blockIdx.x;
    uint4 kr[2], vr[2];
    long long sl[2] = {-1, -1};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int m = n + u * gridDim.x;
        kr[u] = vr[u] = make_uint4(0u, 0u, 0u, 0u);
        if (m < a.num_tokens) {
            kr[u] = load8(K, a.key_stride, m, h, l, vec);
            vr[u] = load8(V, a.value_stride, m, h, l, vec);
            sl[u] = a.slot_mapping[m];
        }
    }
    for (; n < a.num_tokens; n += gridDim.x) {
        const long long slot_idx = sl[0];
        float k[8], v[8];
        unpack8<T>(kr[0], k);
        unpack8<T>(vr[0], v);
        kr[0] = kr[1];
        vr[0] = vr[1];
        sl[0] = sl[1];
        const int nn = n + 2 * gridDim.x;
        if (nn < a.num_tokens) {
            kr[1] = load8(K, a.key_stride, nn, h, l, vec);
            vr[1] = load8(V, a.value_stride, nn, h, l, vec);
            sl[1] = a.slot_mapping[nn];
        }
        if (slot_idx < 0 || slot_idx >= a.num_slots) continue;   // uniform across the CTA
        uint8_t* dst = a.cache + slot_idx * (long long)row_bytes + h * S;

        // ---------------- keys
        if constexpr (KEY_FP8) {
            uint32_t b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) b[i] = __nv_cvt_float_to_fp8(k[i], __NV_SATFINITE, __NV_E4M3);
            uint16_t* d16 = reinterpret_cast<uint16_t*>(dst + 8 * l);
#pragma unroll
            for (int i = 0; i < 4; ++i) d16[i] = uint16_t(b[2 * i] | (b[2 * i + 1] << 8));
        } else {
            float n2 = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) n2 = __fmaf_rn(k[i], k[i], n2);
            n2 = half_sum(n2);
            float x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = sgn[i] * k[i];
            fwht128_half(x, l);
            // y = H(s.k)/||k|| with H = Sylvester / sqrt(128).  The scales
            // use rsqrtf (within 2 ulp): a relative error of ~2^-22 moves y
            // far less than the 1e-5 a code may flip within, and the stored
            // norm far less than its fp16 ulp
            const float rn = n2 > 0.f ? rsqrtf(n2) : 0.f;
            const float inv = 0.08838834764831845f * rn;
            int idx[8];
            float cn = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float y = x[i] * inv;
                int j = 0;
#pragma unroll
                for (int step = 1 << (KBITS - 1); step; step >>= 1) j = y > s_mid[j + step - 1] ? j + step : j;
                idx[i] = j;
                const float c = s_cent[j];
                cn = __fmaf_rn(c, c, cn);
            }
            cn = half_sum(cn);
            // ||k|| / ||c[idx]|| = n2 * rsqrt(n2) * rsqrt(cn)
            const float stored = NORM_CORR ? n2 * rn * rsqrtf(cn) : n2 * rn;
            pack8<KBITS>(dst, idx, l);
            if (l == 0) put_u16(dst + a.g.off_k_norm, __half_as_ushort(__float2half_rn(stored)));
        }

        // ---------------- values: asymmetric min/max uniform codes
        {
            constexpr int QMAX = (1 << VBITS) - 1;
            float lo = v[0], hi = v[0];
#pragma unroll
            for (int i = 1; i < 8; ++i) { lo = fminf(lo, v[i]); hi = fmaxf(hi, v[i]); }
            lo = half_min(lo);
            hi = half_max(hi);
            const __half scale16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), float(QMAX)));
            const __half zero16 = __float2half_rn(lo);
            const float sc = __half2float(scale16), z = __half2float(zero16);
            // code = rint((v - z) / sc) with the division correctly rounded.
            // m = fma(t, fl(1/sc), 1.5 * 2^23) rounds the exact product
            // t * fl(1/sc) to an integer r (half to even), which is its bits
            // minus those of 1.5 * 2^23.  For quotients below 16 that product
            // is within 2^-19 of the correctly rounded quotient, so both
            // round alike unless d = t * fl(1/sc) - r is within 2^-16 of
            // +-1/2, where the exact division decides; larger quotients clamp
            // to QMAX either way.  sc = 0 gives fl(1/sc) := 0 and code 0.
            const float rsc = sc > 0.f ? __frcp_rn(sc) : 0.f;
            int code[8];
            bool near[8], any_near = false;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float t = __fsub_rn(v[i], z);
                const float m = __fmaf_rn(t, rsc, 12582912.f);
                const float r = __fsub_rn(m, 12582912.f);
                const float d = __fmaf_rn(t, rsc, -r);
                code[i] = __float_as_int(m) - 0x4B400000;
                near[i] = fabsf(d) > 0.5f - 0x1p-16f;
                any_near |= near[i];
            }
            // near a half-integer (rare): the exact quotient decides; one
            // warp-uniform test instead of a branch per code
            if (__any_sync(0xffffffffu, any_near)) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (near[i]) code[i] = int(rintf(__fdiv_rn(__fsub_rn(v[i], z), sc)));
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) code[i] = min(max(code[i], 0), QMAX);
            pack8<VBITS>(dst + a.g.off_v_data, code, l);
            if (l == 0) {
                put_u16(dst + a.g.off_v_scale, __half_as_ushort(scale16));
                put_u16(dst + a.g.off_v_zero, __half_as_ushort(zero16));
                if (a.slot_size < S) dst[S - 1] = 0;
            }
        }
    }
}

// Grid of the grid-stride store: every CTA takes the same number of tokens,
// so the grid is the CTAs that fit on the device at once (one wave; a second
// partial wave would finish last with a whole share each).  Resident CTAs
// per SM are asked once per (instantiation, device, kv heads) and kept: the
// instantiations differ in registers and so in CTAs per SM.
template <typename T, bool KEY_FP8, int KBITS, int VBITS, bool NORM_CORR>
cudaError_t launch_one(const StoreArgs& a, cudaStream_t st)
{
    // two kv heads per warp for AoS caches with an even kv-head count; a
    // warp per head otherwise (SoA stages the token's slots in shared memory)
    const bool pairs = !a.g.soa && a.num_kv_heads % 2 == 0;
    auto kernel = pairs ? store2_kernel<T, KEY_FP8, KBITS, VBITS, NORM_CORR>
                        : store_kernel<T, KEY_FP8, KBITS, VBITS, NORM_CORR>;
    static std::atomic<int> cache[2][16][33];  // kernel x devices x kv heads: resident CTAs on the device
    const int threads = pairs ? 16 * a.num_kv_heads : 32 * a.num_kv_heads;
    const size_t smem = pairs ? 0 : size_t(a.num_kv_heads) * a.g.slot;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); dev = 0; }
    const bool keep = dev >= 0 && dev < 16;
    int n = keep ? cache[pairs][dev][a.num_kv_heads].load(std::memory_order_relaxed) : 0;
    if (n <= 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = kNumSMs;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm <= 0)
            per_sm = 4;
        cudaGetLastError();
        n = sms * per_sm;
        if (keep) cache[pairs][dev][a.num_kv_heads].store(n, std::memory_order_relaxed);
    }
    kernel<<<a.num_tokens < n ? a.num_tokens : n, threads, smem, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_store_t(int preset, const StoreArgs& a, cudaStream_t st)
{
    switch (preset & 0xFF) {
    case TQ_K8V4:    return launch_one<T, true, 4, 4, false>(a, st);
    case TQ_4BIT_NC: return launch_one<T, false, 4, 4, true>(a, st);
    case TQ_K3V4_NC: return launch_one<T, false, 3, 4, true>(a, st);
    case TQ_3BIT_NC: return launch_one<T, false, 3, 3, true>(a, st);
    case TQ_2BIT_NC: return launch_one<T, false, 2, 2, true>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace tq

extern "C" int tq_store(int preset, int head_dim, int num_tokens, int num_kv_heads, int block_size,
                        int in_dtype, const void* key, const void* value,
                        long long key_stride_tok, long long value_stride_tok,
                        const int64_t* slot_mapping, uint8_t* kv_cache, long long num_blocks,
                        const int8_t* signs, const float* centroids, const float* midpoints,
                        void* stream)
{
    using namespace tq;
    tq_layout L;
    int rc = fill_layout(preset, head_dim, &L);
    if (rc) return rc;
    if (head_dim != kHeadDim || !block_size_ok(block_size) || !in_dtype_ok(in_dtype))
        return TQ_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_kv_heads < 1 || num_kv_heads > 32 || num_blocks < 0)
        return TQ_ERR_INVALID_ARG;
    if (num_tokens == 0) return TQ_OK;
    if (!key || !value || !slot_mapping || !kv_cache || !signs) return TQ_ERR_INVALID_ARG;
    if (!L.key_fp8 && (!centroids || !midpoints)) return TQ_ERR_INVALID_ARG;
    if (key_stride_tok < (long long)num_kv_heads * head_dim ||
        value_stride_tok < (long long)num_kv_heads * head_dim)
        return TQ_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(kv_cache) & 15) return TQ_ERR_INVALID_ARG;

    StoreArgs a;
    a.key = key;
    a.value = value;
    a.key_stride = key_stride_tok;
    a.value_stride = value_stride_tok;
    a.slot_mapping = slot_mapping;
    a.cache = kv_cache;
    a.num_slots = num_blocks * (long long)block_size;
    a.signs = signs;
    a.centroids = centroids;
    a.midpoints = midpoints;
    a.num_tokens = num_tokens;
    a.num_kv_heads = num_kv_heads;
    a.slot_size = L.slot_size;
    a.bs = block_size;
    a.g = geom_of(L, is_soa(preset));
    // 8-byte input loads need 8-byte aligned rows: both bases, and strides of
    // a multiple of 4 elements
    // (the two-heads-per-warp kernel takes 16-byte loads when the rows are
    // 16-byte aligned: vec = 2)
    const uintptr_t base = reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value);
    a.vec = (base & 7) == 0 && key_stride_tok % 4 == 0 && value_stride_tok % 4 == 0;
    if (a.vec && (base & 15) == 0 && key_stride_tok % 8 == 0 && value_stride_tok % 8 == 0) a.vec = 2;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = in_dtype == TQ_F16 ? launch_store_t<__half>(preset, a, st)
                                       : launch_store_t<__nv_bfloat16>(preset, a, st);
    return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
