// Split-K decode attention read straight from the compressed paged cache.
//
// Method: "vllm-project/vllm pull 38479" digest, implementation item 4 (stage 1
// scores from the compressed cache and accumulates values per split, stage 2
// merges splits by log-sum-exp); "vllm.v1.attention.backends.turboquant_attn"
// API page, section "_decode_attention" (GQA grouping, fixed split count,
// shared mid_o / lse scratch); "turboquant-plus.md", "weight pre-rotation"
// note (<Q H, H K> = <Q, K>, so q is rotated once and keys stay rotated).
//
// This file holds the host entry point, stage 2 (the log-sum-exp merge) and
// the CUDA-core stage 1 used for shapes the tensor-core stage 1
// (tq_decode_mma.cu) does not serve: one CTA per (split, kv head, sequence),
// four warps striding over the split's tokens, 4 coordinates per lane, fp32
// scores and online softmax, partials merged across warps in shared memory.
#include "tq.h"
#include "tq_device.cuh"
#include "tq_internal.h"

#include <cmath>
#include <mutex>
#include <vector>

namespace tq {

namespace {

struct DecodeArgs {
    const void* query;
    const uint8_t* cache;
    long long num_blocks;
    const int32_t* block_table;
    int bt_stride;
    const int32_t* seq_lens;
    float scale;
    int num_splits;
    const int8_t* signs;
    const float* centroids;
    float* mid;          // (B, Hq, S, D+1)
    void* out;
    float* lse;
    int B, Hq, Hk, G, bs;
    float vthr;          // sparse V: rows with p <= vthr skip the value sum (0: off)
    SlotGeom g;
};

constexpr int kWarps = 4;

// Codes 4*lane .. 4*lane+3 of a packed code stream starting at p (2-byte
// aligned).  Every width is an LSB-first bitstream: 4 bits low nibble first,
// 2 bits four per byte, 3 bits 8 codes per 3 bytes (the lane's 12 bits start
// at bit 12*lane, i.e. byte 3*lane/2 plus 0 or 4 bits).
template <int BITS>
__device__ __forceinline__ void load_codes(const uint8_t* p, int lane, int (&c)[4])
{
    if constexpr (BITS == 2) {
        const uint32_t w = p[lane];
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = (w >> (2 * i)) & 3u;
    } else if constexpr (BITS == 4) {
        const uint32_t w = ld_u16(p + 2 * lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = (w >> (4 * i)) & 15u;
    } else {
        static_assert(BITS == 3, "2, 3 or 4 bits");
        const uint8_t* q = p + ((3 * lane) >> 1);
        const uint32_t w = (uint32_t(q[0]) | uint32_t(q[1]) << 8) >> (4 * (lane & 1));
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = (w >> (3 * i)) & 7u;
    }
}

template <typename TQ, bool KEY_FP8, int KBITS, int VBITS, int GM>
__global__ void __launch_bounds__(kWarps * 32) stage1_kernel(DecodeArgs a)
{
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.G, S = a.num_splits;
    const int L = a.seq_lens[b];
    const int chunk = (L + S - 1) / S;
    const int t0 = split * chunk;
    const int t1 = min(L, t0 + chunk);

    __shared__ float s_cent[16];
    __shared__ float s_m[kWarps][GM], s_l[kWarps][GM];
    __shared__ float s_acc[kWarps][GM][kHeadDim];

    if (t0 >= t1) {   // empty split: lse = -inf, zero partial output
        for (int i = threadIdx.x; i < G * (kHeadDim + 1); i += blockDim.x) {
            const int g = i / (kHeadDim + 1), d = i % (kHeadDim + 1);
            float* m = a.mid + (((long long)b * a.Hq + h * G + g) * S + split) * (kHeadDim + 1);
            m[d] = d == kHeadDim ? -INFINITY : 0.f;
        }
        return;
    }
    __shared__ int s_bad;        // a block-table entry outside [0, num_blocks) was met
    if (threadIdx.x == 0) s_bad = 0;
    if constexpr (!KEY_FP8) {
        if (threadIdx.x < (1 << KBITS)) s_cent[threadIdx.x] = a.centroids[threadIdx.x];
    }

    // q (rotated once for MSE keys), pre-multiplied by the softmax scale
    float qv[GM][4];
    const TQ* Q = static_cast<const TQ*>(a.query);
    float sgn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sgn[i] = KEY_FP8 ? 1.f : float(a.signs[4 * lane + i]);
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        if (g < G) {
            const TQ* qp = Q + ((long long)b * a.Hq + h * G + g) * kHeadDim + 4 * lane;
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[g][i] = sgn[i] * to_f32(qp[i]);
            if constexpr (!KEY_FP8) {
                fwht128_warp(qv[g], lane);
#pragma unroll
                for (int i = 0; i < 4; ++i) qv[g][i] *= 0.08838834764831845f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[g][i] *= a.scale;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[g][i] = 0.f;
        }
    }
    __syncthreads();

    float m[GM], l[GM], acc[GM][4];
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[g][i] = 0.f;
    }

    const int32_t* bt = a.block_table + (long long)b * a.bt_stride;
    const int lgbs = 31 - __clz(a.bs);       // block sizes are powers of two
    bool bad = false;
    for (int t = t0 + warp; t < t1; t += kWarps) {
        const long long page = bt[t >> lgbs];
        if (page < 0 || page >= a.num_blocks) { bad = true; continue; }   // not read; the rows become NaN
        const uint8_t *sp, *mp;              // data and metadata of the record
        slot_ptrs(a.g, a.cache, page, t & (a.bs - 1), h, a.bs, a.Hk, sp, mp);

        float kv[4];
        float knorm = 1.f;
        if constexpr (KEY_FP8) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                __half_raw hr = __nv_cvt_fp8_to_halfraw(sp[4 * lane + i], __NV_E4M3);
                kv[i] = __half2float(__half(hr));
            }
        } else {
            int c[4];
            load_codes<KBITS>(sp, lane, c);
#pragma unroll
            for (int i = 0; i < 4; ++i) kv[i] = s_cent[c[i]];
            knorm = __half2float(__ushort_as_half(ld_u16(mp + a.g.m_norm)));
        }
        float s[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g)
            s[g] = warp_sum(qv[g][0] * kv[0] + qv[g][1] * kv[1] + qv[g][2] * kv[2] + qv[g][3] * kv[3]) * knorm;

        // online softmax; sparse V: a row whose p is at most vthr keeps its
        // weight in l but adds nothing to the value sum, and the value codes
        // are not read when no head keeps the row (s is warp-uniform)
        float al[GM], pv[GM];
        bool anyv = false;
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            const float mn = fmaxf(m[g], s[g]);
            const float p = expf(s[g] - mn);
            al[g] = expf(m[g] - mn);
            l[g] = l[g] * al[g] + p;
            m[g] = mn;
            pv[g] = p > a.vthr ? p : 0.f;
            anyv |= g < G && pv[g] > 0.f;
        }
        float vv[4] = {0.f, 0.f, 0.f, 0.f};
        if (anyv) {
            int vc[4];
            load_codes<VBITS>(sp + a.g.v_off, lane, vc);
            const float vs = __half2float(__ushort_as_half(ld_u16(mp + a.g.m_scale)));
            const float vz = __half2float(__ushort_as_half(ld_u16(mp + a.g.m_zero)));
#pragma unroll
            for (int i = 0; i < 4; ++i) vv[i] = float(vc[i]) * vs + vz;
        }
#pragma unroll
        for (int g = 0; g < GM; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[g][i] = acc[g][i] * al[g] + pv[g] * vv[i];
    }

    // merge the four warps' partials
    if (bad && lane == 0) s_bad = 1;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        if (lane == 0) { s_m[warp][g] = m[g]; s_l[warp][g] = l[g]; }
#pragma unroll
        for (int i = 0; i < 4; ++i) s_acc[warp][g][4 * lane + i] = acc[g][i];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * kHeadDim; i += blockDim.x) {
        const int g = i / kHeadDim, d = i % kHeadDim;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][g]);
        float lsum = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = s_m[w][g] == -INFINITY ? 0.f : expf(s_m[w][g] - M);
            lsum += s_l[w][g] * f;
            o += s_acc[w][g][d] * f;
        }
        float* mp = a.mid + (((long long)b * a.Hq + h * G + g) * S + split) * (kHeadDim + 1);
        mp[d] = o / lsum;
        if (d == 0) mp[kHeadDim] = s_bad ? __int_as_float(0x7fc00000) : M + logf(lsum);
    }
}

// Stage 2: the log-sum-exp merge of the split partials.  A row (sequence,
// query head) takes R = ceil(S / 16) warps (at most 8), each merging every
// R-th split in rounds of 16 with every load of a round issued before any
// arithmetic; lane l owns dims 4l..4l+3.  The R partial merges (running max
// M, weight sum W, weighted output) are combined through shared memory by
// the row's first warp.  A NaN lse (a split that gave up waiting for its
// data, or met a block-table entry outside the cache) makes the row NaN.
constexpr int kStage2Warps = 8;

template <typename TO>
__global__ void __launch_bounds__(32 * kStage2Warps) stage2_kernel(DecodeArgs a, int R)
{
    __shared__ float s_part[kStage2Warps][kHeadDim + 2];
    // launched as a programmatic dependent of stage 1: wait until its
    // partials are complete and visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rows_per_cta = kStage2Warps / R;
    const int r = warp % R;                                    // this warp's share of the splits
    const long long bh = (long long)blockIdx.x * rows_per_cta + warp / R;   // b * Hq + hq
    const bool live = bh < (long long)a.B * a.Hq;
    const int S = a.num_splits;
    constexpr int kRound = 16;
    float M = -INFINITY, W = 0.f;
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    if (live) {
        const float* mp = a.mid + bh * S * (kHeadDim + 1);
        for (int s0 = r; s0 < S; s0 += kRound * R) {
            float ls[kRound], x[kRound][4];
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
                const int sp = s0 + u * R;
                const float* row = mp + min(sp, S - 1) * (kHeadDim + 1);
                ls[u] = sp < S ? row[kHeadDim] : -INFINITY;
#pragma unroll
                for (int i = 0; i < 4; ++i) x[u][i] = row[4 * lane + i];
            }
            float mc = M;
            bool nan = false;
#pragma unroll
            for (int u = 0; u < kRound; ++u) { mc = fmaxf(mc, ls[u]); nan |= ls[u] != ls[u]; }
            if (nan) { M = W = __int_as_float(0x7fc00000); break; }
            if (mc == -INFINITY) continue;            // only empty splits so far
            const float sc = expf(M - mc);            // 0 while M = -inf
            W *= sc;
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] *= sc;
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
                const float w = expf(ls[u] - mc);     // 0 for empty and padding splits
                W += w;
                if (w != 0.f) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] += w * x[u][i];
                }
            }
            M = mc;
        }
    }
    if (R > 1) {                                     // uniform per launch
        float* sp = s_part[warp];
#pragma unroll
        for (int i = 0; i < 4; ++i) sp[4 * lane + i] = o[i];
        if (lane == 0) { sp[kHeadDim] = M; sp[kHeadDim + 1] = W; }
        __syncthreads();
        if (r != 0) return;
        M = -INFINITY;
        bool nan = false;
        for (int j = 0; j < R; ++j) {
            const float mj = s_part[warp + j][kHeadDim];
            nan |= mj != mj;
            M = fmaxf(M, mj);
        }
        W = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = 0.f;
        if (nan) {
            M = W = __int_as_float(0x7fc00000);
        } else if (M != -INFINITY) {
            for (int j = 0; j < R; ++j) {
                const float* pj = s_part[warp + j];
                const float f = pj[kHeadDim] == -INFINITY ? 0.f : expf(pj[kHeadDim] - M);
                W += pj[kHeadDim + 1] * f;
#pragma unroll
                for (int i = 0; i < 4; ++i) o[i] += pj[4 * lane + i] * f;
            }
        }
    }
    if (!live) return;
    if (M != -INFINITY) {
        const float inv = 1.f / W;
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] *= inv;
    }
    TO* out = static_cast<TO*>(a.out) + bh * kHeadDim + 4 * lane;
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = from_f32<TO>(o[i]);
    if (lane == 0 && a.lse) a.lse[bh] = M == -INFINITY ? -INFINITY : M + logf(W);
}

template <typename TO>
cudaError_t launch_stage2(const DecodeArgs& a, cudaStream_t st)
{
    int R = (a.num_splits + 15) / 16;                 // warps per row: at most 16 splits each
    R = R <= 1 ? 1 : R <= 2 ? 2 : R <= 4 ? 4 : 8;     // a divisor of kStage2Warps
    const unsigned rows = unsigned(a.B) * a.Hq, rows_per_cta = kStage2Warps / R;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows + rows_per_cta - 1) / rows_per_cta);
    cfg.blockDim = dim3(32 * kStage2Warps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stage2_kernel<TO>, a, R);
}

template <typename TQ, bool FP8, int KB, int VB>
cudaError_t launch_stage1_g(const DecodeArgs& a, cudaStream_t st)
{
    dim3 grid(a.num_splits, a.Hk, a.B);
    if (a.G <= 1) stage1_kernel<TQ, FP8, KB, VB, 1><<<grid, kWarps * 32, 0, st>>>(a);
    else if (a.G <= 2) stage1_kernel<TQ, FP8, KB, VB, 2><<<grid, kWarps * 32, 0, st>>>(a);
    else if (a.G <= 4) stage1_kernel<TQ, FP8, KB, VB, 4><<<grid, kWarps * 32, 0, st>>>(a);
    else if (a.G <= 8) stage1_kernel<TQ, FP8, KB, VB, 8><<<grid, kWarps * 32, 0, st>>>(a);
    else stage1_kernel<TQ, FP8, KB, VB, 16><<<grid, kWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename TQ>
cudaError_t launch_stage1(int preset, const DecodeArgs& a, cudaStream_t st)
{
    switch (preset & 0xFF) {
    case TQ_K8V4:    return launch_stage1_g<TQ, true, 4, 4>(a, st);
    case TQ_4BIT_NC: return launch_stage1_g<TQ, false, 4, 4>(a, st);
    case TQ_K3V4_NC: return launch_stage1_g<TQ, false, 3, 4>(a, st);
    case TQ_3BIT_NC: return launch_stage1_g<TQ, false, 3, 3>(a, st);
    case TQ_2BIT_NC: return launch_stage1_g<TQ, false, 2, 2>(a, st);
    }
    return cudaErrorInvalidValue;
}

template <bool FP8, int KB, int VB>
int v1_slots(int G, int num_sms)
{
    int per_sm = 0;
    cudaError_t e;
    if (G <= 1) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stage1_kernel<__nv_bfloat16, FP8, KB, VB, 1>, kWarps * 32, 0);
    else if (G <= 2) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stage1_kernel<__nv_bfloat16, FP8, KB, VB, 2>, kWarps * 32, 0);
    else if (G <= 4) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stage1_kernel<__nv_bfloat16, FP8, KB, VB, 4>, kWarps * 32, 0);
    else if (G <= 8) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stage1_kernel<__nv_bfloat16, FP8, KB, VB, 8>, kWarps * 32, 0);
    else e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stage1_kernel<__nv_bfloat16, FP8, KB, VB, 16>, kWarps * 32, 0);
    return e == cudaSuccess ? per_sm * num_sms : 0;
}

// (CTAs per split, resident CTA slots) of the stage-1 kernel for a shape,
// cached per device.
void stage1_shape(const tq_layout& L, bool soa, int Hk, int G, int* cps, int* slots)
{
    struct Entry { int dev, kf8, kb, vb, soa, hk, g, cps, slots; };
    static std::mutex mu;
    static std::vector<Entry> cache;
    int dev = -1, num_sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();        // no device: clear the error, use the defaults below
        dev = -1;
        num_sms = 0;
    }
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry& e : cache)
            if (e.dev == dev && e.kf8 == L.key_fp8 && e.kb == L.key_bits && e.vb == L.value_bits &&
                e.soa == int(soa) && e.hk == Hk && e.g == G) {
                *cps = e.cps;
                *slots = e.slots;
                return;
            }
    }
    int c = Hk, n = 0;
    if (mma_stage1_supported(L, soa, Hk, G)) {
        mma_stage1_shape(L, soa, Hk, G, num_sms, &c, &n);
    } else if (num_sms > 0) {
        c = Hk;                    // grid (splits, kv heads, batch)
        if (L.key_fp8) n = v1_slots<true, 4, 4>(G, num_sms);
        else if (L.key_bits == 2) n = v1_slots<false, 2, 2>(G, num_sms);
        else if (L.key_bits == 4) n = v1_slots<false, 4, 4>(G, num_sms);
        else if (L.value_bits == 4) n = v1_slots<false, 3, 4>(G, num_sms);
        else n = v1_slots<false, 3, 3>(G, num_sms);
    }
    if (n <= 0) {
        cudaGetLastError();
        n = 2 * kNumSMs;           // no device to ask: two CTAs per SM of a GB300
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() < 256) cache.push_back({dev, L.key_fp8, L.key_bits, L.value_bits, int(soa), Hk, G, c, n});
    *cps = c;
    *slots = n;
}

}  // namespace

int pick_splits(const tq_layout& L, bool soa, int batch, int num_q_heads, int num_kv_heads, int max_seq_len)
{
    if (batch <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || max_seq_len <= 0) return 1;
    int cps = 1, slots = 1;
    stage1_shape(L, soa, num_kv_heads, num_q_heads / num_kv_heads, &cps, &slots);
    // Critical path of stage 1 in 32-token tiles: the CTAs of all splits run
    // in ceil(CTAs / slots) waves, each as long as one split's tiles plus a
    // fixed start-up (q preparation, first copy latency, epilogue) worth about
    // kStartTiles tiles.  Splits shorter than 128 tokens are not used.
    constexpr double kStartTiles = 3.0;
    long long max_s = (max_seq_len + 127) / 128;
    if (max_s > TQ_MAX_SPLITS) max_s = TQ_MAX_SPLITS;
    if (max_s < 1) max_s = 1;
    int best = 1;
    double best_cost = 0.0;
    for (long long s = 1; s <= max_s; ++s) {
        const long long ctas = (long long)batch * s * cps;
        const long long waves = (ctas + slots - 1) / slots;
        const long long chunk = (max_seq_len + s - 1) / s;
        const long long tiles = (chunk + 31) / 32;
        const double cost = double(waves) * (double(tiles) + kStartTiles);
        if (s == 1 || cost < best_cost * (1.0 - 1e-9)) { best = int(s); best_cost = cost; }
    }
    return best;
}

}  // namespace tq

namespace tq {
namespace {

// Argument checks, split choice and the launches of both stages; stuck_tile
// >= 0 (the wait-expiry test) needs the tensor-core stage 1.
int decode_impl(int preset, int head_dim, int batch, int num_q_heads, int num_kv_heads, int block_size,
                int q_dtype, const void* query, const uint8_t* kv_cache, long long num_blocks,
                const int32_t* block_table, int block_table_stride, const int32_t* seq_lens,
                int max_seq_len, float softmax_scale, int num_splits, const int8_t* signs,
                const float* centroids, void* out, int out_dtype, float* lse, void* workspace,
                size_t workspace_bytes, float v_threshold, int stuck_tile, uint32_t wait_polls,
                void* stream)
{
    tq_layout L;
    int rc = fill_layout(preset, head_dim, &L);
    if (rc) return rc;
    if (head_dim != kHeadDim || !block_size_ok(block_size) || !in_dtype_ok(q_dtype) ||
        !out_dtype_ok(out_dtype))
        return TQ_ERR_UNSUPPORTED;
    if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads ||
        num_blocks < 0 || block_table_stride < 0 || max_seq_len < 0 || num_splits < 0 ||
        num_splits > TQ_MAX_SPLITS || !(v_threshold >= 0.f && v_threshold < 1.f))
        return TQ_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > kMaxGroup) return TQ_ERR_UNSUPPORTED;
    if (batch == 0) return TQ_OK;
    if (!query || !kv_cache || !block_table || !seq_lens || !out || !workspace)
        return TQ_ERR_INVALID_ARG;
    if (!L.key_fp8 && (!signs || !centroids)) return TQ_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 15) return TQ_ERR_INVALID_ARG;
    const bool soa = is_soa(preset);
    const int S = num_splits ? num_splits : pick_splits(L, soa, batch, num_q_heads, num_kv_heads, max_seq_len);
    if (workspace_bytes < tq_decode_workspace_bytes(batch, num_q_heads, S, head_dim))
        return TQ_ERR_WORKSPACE;

    DecodeArgs a;
    a.query = query;
    a.cache = kv_cache;
    a.num_blocks = num_blocks;
    a.block_table = block_table;
    a.bt_stride = block_table_stride;
    a.seq_lens = seq_lens;
    a.scale = softmax_scale;
    a.num_splits = S;
    a.signs = signs;
    a.centroids = centroids;
    a.mid = static_cast<float*>(workspace);
    a.out = out;
    a.lse = lse;
    a.B = batch;
    a.Hq = num_q_heads;
    a.Hk = num_kv_heads;
    a.G = num_q_heads / num_kv_heads;
    a.bs = block_size;
    a.vthr = v_threshold;
    a.g = geom_of(L, soa);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    const bool mma = mma_stage1_supported(L, soa, num_kv_heads, a.G);
    if (stuck_tile >= 0 && !mma) return TQ_ERR_UNSUPPORTED;
    if (mma) {
        rc = launch_mma_stage1(L, soa, q_dtype, query, kv_cache, num_blocks, block_table, block_table_stride, seq_lens,
                               softmax_scale, S, signs, centroids, a.mid, batch, num_q_heads,
                               num_kv_heads, block_size, v_threshold, st, stuck_tile,
                               wait_polls);
        if (rc) return rc;
    } else {
        cudaError_t e = q_dtype == TQ_F16 ? launch_stage1<__half>(preset, a, st)
                                          : launch_stage1<__nv_bfloat16>(preset, a, st);
        if (e != cudaSuccess) return TQ_ERR_CUDA;
    }
    const cudaError_t e2 = out_dtype == TQ_F32 ? launch_stage2<float>(a, st)
                           : out_dtype == TQ_F16 ? launch_stage2<__half>(a, st)
                                                 : launch_stage2<__nv_bfloat16>(a, st);
    return e2 == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace
}  // namespace tq

extern "C" int tq_decode_attention_sparse_v(int preset, int head_dim, int batch, int num_q_heads,
                                            int num_kv_heads, int block_size, int q_dtype,
                                            const void* query, const uint8_t* kv_cache,
                                            long long num_blocks, const int32_t* block_table,
                                            int block_table_stride, const int32_t* seq_lens,
                                            int max_seq_len, float softmax_scale, int num_splits,
                                            const int8_t* signs, const float* centroids, void* out,
                                            int out_dtype, float* lse, void* workspace,
                                            size_t workspace_bytes, float v_threshold, void* stream)
{
    return tq::decode_impl(preset, head_dim, batch, num_q_heads, num_kv_heads, block_size, q_dtype, query,
                           kv_cache, num_blocks, block_table, block_table_stride, seq_lens, max_seq_len,
                           softmax_scale, num_splits, signs, centroids, out, out_dtype, lse, workspace,
                           workspace_bytes, v_threshold, -1, tq::kWaitPolls, stream);
}

extern "C" int tq_test_decode_wait_expiry(int preset, int head_dim, int batch, int num_q_heads,
                                          int num_kv_heads, int block_size, int q_dtype,
                                          const void* query, const uint8_t* kv_cache,
                                          long long num_blocks, const int32_t* block_table,
                                          int block_table_stride, const int32_t* seq_lens,
                                          int max_seq_len, float softmax_scale, int num_splits,
                                          const int8_t* signs, const float* centroids, void* out,
                                          int out_dtype, float* lse, void* workspace,
                                          size_t workspace_bytes, int stuck_tile,
                                          unsigned int wait_polls, void* stream)
{
    if (stuck_tile < 0 || wait_polls < 1) return TQ_ERR_INVALID_ARG;
    return tq::decode_impl(preset, head_dim, batch, num_q_heads, num_kv_heads, block_size, q_dtype, query,
                           kv_cache, num_blocks, block_table, block_table_stride, seq_lens, max_seq_len,
                           softmax_scale, num_splits, signs, centroids, out, out_dtype, lse, workspace,
                           workspace_bytes, 0.f, stuck_tile, wait_polls, stream);
}

extern "C" int tq_decode_attention(int preset, int head_dim, int batch, int num_q_heads,
                                   int num_kv_heads, int block_size, int q_dtype, const void* query,
                                   const uint8_t* kv_cache, long long num_blocks,
                                   const int32_t* block_table, int block_table_stride,
                                   const int32_t* seq_lens, int max_seq_len,
                                   float softmax_scale, int num_splits,
                                   const int8_t* signs, const float* centroids,
                                   void* out, int out_dtype, float* lse,
                                   void* workspace, size_t workspace_bytes, void* stream)
{
    return tq_decode_attention_sparse_v(preset, head_dim, batch, num_q_heads, num_kv_heads, block_size,
                                        q_dtype, query, kv_cache, num_blocks, block_table,
                                        block_table_stride, seq_lens, max_seq_len, softmax_scale,
                                        num_splits, signs, centroids, out, out_dtype, lse, workspace,
                                        workspace_bytes, 0.f, stream);
}

extern "C" int tq_decode_kernel_kind(int preset, int head_dim, int num_q_heads, int num_kv_heads)
{
    using namespace tq;
    tq_layout L;
    if (fill_layout(preset, head_dim, &L) || head_dim != kHeadDim || num_kv_heads < 1 ||
        num_q_heads < 1 || num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > kMaxGroup)
        return -1;                  // the shapes tq_decode_attention rejects
    return mma_stage1_supported(L, is_soa(preset), num_kv_heads, num_q_heads / num_kv_heads) ? 1 : 0;
}
