// Decode stage 1 on tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate).
//
// Same partials as the CUDA-core stage 1 (per split: o_s and lse_s in the
// fp32 workspace), computed per CTA = (split, sequence, kv-head group): one
// warp per kv head, 32-token tiles streamed into a shared-memory ring by
// bulk (TMA) copies of whole token rows (Hk contiguous slots each; FP8 keys:
// 2-D tensor copies of 4 heads' part of each row) whose completion is
// tracked by mbarriers with bounded waits; warps only wait for data, never
// for each other (the last warp done with a stage refills it).
//
// Per tile and warp, with G query heads sharing the kv head:
//   scores  S[t, g] = sum_d K^[t, d] Q[g, d]      A = K^ (16 tokens x 16 dims),
//                                                B = q columns (16 dims x 8)
//   values  O[d, g] += sum_t V^[t, d] P'[t, g]    A = V codes (16 dims x 16 tokens),
//                                                B = P' columns (16 tokens x 8)
// The grouped-query tiles are dense after unpacking, so they run as MMAs.
// Precision: fp16 operands carry 11 bits, so every fp32 quantity that is not
// exactly representable is split into hi = fp16(x) and lo = fp16(x - hi):
// q (all presets), the Lloyd-Max centroids of 3- and 4-bit keys, and P' (for
// G = 4 the spare 4 columns carry the lo parts; for G = 8 a second MMA does).
// 2-bit centroids are scaled by a factor that makes them fp16-exact (no lo
// part).  FP8 keys and integer value codes are exact in fp16.  The value
// path uses P' = p * v_scale and adds sum_t p_t v_zero_t separately
// (v_hat = code * scale + zero).  With 3- or 4-bit keys and G = 8, q's lo
// part meets only the keys' hi words, and the q fragments live in tensor
// memory (tcgen05.st / tcgen05.ld), which leaves the shared memory to the
// ring.
// Centroid lookups: 3- and 4-bit keys read code pairs from a shared-memory
// table (one 8-byte load per pair: both centroids, hi and lo); 2-bit keys
// select bytes of register tables with PRMT.
//
// Launch chain: stage 1 is a programmatic dependent of the previous kernel
// in the stream and waits for it before its first global read; stage 2 is a
// programmatic dependent of stage 1.
//
// Method sources: "vllm-project/vllm pull 38479" digest, implementation item 4
// (split-K stage 1 / stage 2); "vllm.v1.attention.backends.turboquant_attn" API
// page, "_decode_attention" (GQA grouping, fixed split count);
// "turboquant-plus.md", weight pre-rotation note (<Q H, H K> = <Q, K>).
#include "tq.h"
#include "tq_device.cuh"
#include "tq_internal.h"

#include <cuda.h>

#include <cmath>
#include <type_traits>

namespace tq {

struct MmaArgs {
    // CTAs that take part of each token row (FP8 keys, 4 of 8+ kv heads):
    // a 2-D map of the cache as rows of 32-bit words (inner: the row, outer:
    // block * bs + offset), boxes of the CTA's copy_bytes x one page segment
    CUtensorMap tmap;
    int use_tmap;            // 1: page segments by tensor copies through tmap
    const void* query;
    const uint8_t* cache;
    long long num_blocks;    // block-table entries outside [0, num_blocks) are caller errors
    const int32_t* block_table;
    int bt_stride;
    const int32_t* seq_lens;
    float qscale;            // softmax_scale * log2(e): scores in log2 units
    int num_splits;
    const int8_t* signs;
    const float* centroids;
    float* mid;              // (B, Hq, S, D+1)
    int Hq, Hk, G, bs, bs_log2;
    int row_bytes;           // global token row: Hk * slot
    int hpc;                 // kv heads per CTA (Hk, or 4 for FP8 keys)
    int nqg;                 // query-head groups per kv head: CTAs of up to 8 of its G query heads
    int copy_bytes;          // AoS: hpc * slot; SoA: hpc * data record (the data part a CTA copies)
    int smem_row;            // copy_bytes padded to 16 mod 32 bytes
    int meta_bytes;          // SoA: hpc * metadata record per token (0 for AoS)
    int nstages;
    float vthr;              // sparse V: rows with p <= vthr skip the value sum (0: off)
    int lpt;                 // 1: CTA row y takes the y-th longest sequence (seq_of_rank)
    float key_alpha;         // 2-bit keys: centroid scale making alpha * c_k fp16-exact (0: none)
    uint32_t wait_polls;     // mbarrier polls before a stage wait gives up
    int stuck_tile;          // test hook: this tile of split 0, sequence 0, head group 0 is
                             // expected 16 bytes more than its copies bring (-1: none)
    SlotGeom g;
};

// Stage 1 with the value sum of every row (dense) or with the sparse-V gate;
// each is instantiated in its own translation unit.
cudaError_t launch_mma_dense(const MmaArgs& a, int q_dtype, int B, size_t smem, cudaStream_t st);
cudaError_t launch_mma_sparse(const MmaArgs& a, int q_dtype, int B, size_t smem, cudaStream_t st);

namespace {

constexpr int kTile = 32;   // tokens per pipeline stage (two 16-row MMA tiles)

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// hi/lo fp16 split of x: x ~= hi + lo with |x - hi - lo| ~ 2^-22 |x|
__device__ __forceinline__ void split_f16(float x, float& hi, float& lo)
{
    hi = __half2float(__float2half_rn(x));
    lo = x - hi;
}

// ---- bulk (TMA) copies into shared memory, completion tracked by mbarriers
__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 20000;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity, giving up after `limit` polls;
// each poll suspends the thread until the phase completes or 20 us pass.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit)
{
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// One box of a 2-D tensor map (x: 32-bit words within a row, y: row) into
// shared memory, completing on the mbarrier.  x * 4 is a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void fence_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Tensor memory (TMEM): a CTA's allocation is 128 lanes x ncols columns of
// 32-bit cells; warp w reaches lanes 32 (w mod 4) .. 32 (w mod 4) + 31, one
// per thread, at the address (lane << 16) + column.  Allocation and
// deallocation are per warp (all lanes); the allocated address is written to
// shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Four consecutive columns of this thread's lane (all lanes of the warp).
// TMEM is not memory the compiler tracks: these carry no memory clobber, so
// shared-memory loads may move across them; the volatile statements keep
// their order among themselves (and with the MMAs that use the registers).
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint4& v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w));
}
__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;");
}
// the registers are valid after tmem_wait_ld()
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint4& v)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;");
}

// n little-endian 32-bit words starting at the 2-byte aligned shared address p.
// `mis` (0 or 2, uniform per warp) is p mod 4.  MIS = 0 or 2 fixes it at
// compile time (the tile loop is instantiated per warp misalignment: a
// branch in the loop costs more than the loads); MIS = -1 reads `mis`.
template <int N, int MIS = -1>
__device__ __forceinline__ void lds_words(const uint8_t* p, int mis, uint32_t (&w)[N])
{
    if (MIS == 0 || (MIS < 0 && mis == 0)) {
        const uint32_t* q = reinterpret_cast<const uint32_t*>(p);
#pragma unroll
        for (int i = 0; i < N; ++i) w[i] = q[i];
    } else {
        const uint32_t* q = reinterpret_cast<const uint32_t*>(p - mis);
        uint32_t r[N + 1];
#pragma unroll
        for (int i = 0; i <= N; ++i) r[i] = q[i];
#pragma unroll
        for (int i = 0; i < N; ++i) w[i] = __funnelshift_r(r[i], r[i + 1], 16);
    }
}

__device__ __forceinline__ float lds_f16(const uint8_t* p)
{
    return __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(p)));
}

// Eight 3-bit codes (bits 0..23 of x, code i at bit 3i) spread to a nibble
// word (code i in bits [4i, 4i+3), every nibble's top bit clear).  Each
// step moves the upper part of every field up with a masked multiply-add:
// a + (2^k - 1) * (a & m) = (a & ~m) + 2^k (a & m).
__device__ __forceinline__ uint32_t spread3(uint32_t x)
{
    uint32_t a = x & 0x00FFFFFFu;
    a += 15u * (a & 0x00FFF000u);     // codes 4..7 to bits 16..27
    a += 3u * (a & 0x0FC00FC0u);      // codes 2, 3 (6, 7) up by 2 bits: two codes per byte
    a += a & 0x38383838u;             // odd codes up by 1 bit
    return a;
}

// 3-bit keys: a code pair (codes 2p, 2p + 1 of a 32-code group, the 6-bit
// field at bit 6p of the group's 96-bit LSB-first stream w[0..2]) indexes a
// shared table of 64 entries, each the pair's (hi, lo) fp16x2 centroids.
// Entries are 128 bytes apart and hold one copy per half-warp lane (lane
// & 15 at byte 8 (lane & 15)), so the 16 lanes of each half of an 8-byte
// load touch 16 distinct bank pairs whatever codes they read.  The field is
// shifted to bits [7, 13), the entry offset.
constexpr int kLut3Entries = 64 * 16;

__device__ __forceinline__ uint32_t pair_off(const uint32_t (&w)[3], int bit)
{
    const int wi = bit >> 5, b = bit & 31;
    uint32_t x;
    if (b + 6 > 32)  x = __funnelshift_r(w[wi], w[wi + 1], b - 7);
    else if (b >= 7) x = w[wi] >> (b - 7);
    else             x = w[wi] << (7 - b);
    return x & 0x1F80u;
}

// 4-bit keys: the code pair of byte p of the group's 16 bytes (codes 2p in
// the low nibble, 2p + 1 in the high one) indexes a 256-entry table laid out
// like the 3-bit one (entries 128 bytes apart, a copy per half-warp lane):
// the byte is shifted to bits [7, 15).
constexpr int kLut4Entries = 256 * 16;

__device__ __forceinline__ uint32_t pair_off(const uint32_t (&w)[4], int p)
{
    const uint32_t x = w[p >> 2];
    const int b = 8 * (p & 3);
    return (b >= 7 ? x >> (b - 7) : x << (7 - b)) & 0x7F80u;
}

// the (hi, lo) entry of code pair p of a 3-bit (N = 3) or 4-bit (N = 4) group
template <int N>
__device__ __forceinline__ uint2 lut_pair(const uint2* lut, const uint32_t (&w)[N], int p, uint32_t l8)
{
    uint32_t off;
    if constexpr (N == 3) off = pair_off(w, 6 * p);
    else                  off = pair_off(w, p);
    return *reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(lut) + (off | l8));
}

// Longest-first dispatch: CTA row y (blockIdx.y) takes the sequence of rank y
// when the batch is ordered by decreasing length (ties by index), so the
// block scheduler starts the longest sequences' splits first and the short
// ones fill the tail of the grid.  O(B) per thread for B <= 512; `sl` is
// (B + 1) ints of shared memory; all threads of the block call it.
__device__ __forceinline__ int seq_of_rank(const int32_t* seq_lens, int B, int r, int* sl)
{
    for (int i = threadIdx.x; i < B; i += blockDim.x) sl[i] = seq_lens[i];
    __syncthreads();
    for (int c = threadIdx.x; c < B; c += blockDim.x) {
        const int Lc = sl[c];
        int rank = 0;
        for (int j = 0; j < B; ++j) {
            const int Lj = sl[j];
            rank += (Lj > Lc) || (Lj == Lc && j < c);
        }
        if (rank == r) sl[B] = c;        // the ranks are a permutation: one writer
    }
    __syncthreads();
    const int b = sl[B];
    __syncthreads();                     // the area is reused afterwards
    return b;
}

// Token order inside a 16-row tile: the MMAs' own.  QK row r is token r
// (thread gid: tokens gid and gid + 8); value k index k is token k (thread
// tig: tokens 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9, held by the QK threads
// gid = 2 tig and 2 tig + 1).  With a shared row stride of 4 mod 8 words,
// the key loads of a warp (8 rows, 12-16 bytes per lane) and its value loads
// (4 rows 2 tig + c, 8 bytes per lane) touch distinct banks.

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// two E4M3 pairs (low and high half of w) -> two f16x2
__device__ __forceinline__ void cvt_e4m3x4(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Scores of one 16-row MMA tile for the thread's rows (r0: row gid, r1:
// row gid+8), FP8 or 2-bit keys.  Returns the raw accumulators: G = 4 -> sc
// (cols head x {hi,lo}); G = 8 -> sc (q hi), scl (q lo).  2-bit keys with
// G = 8 read their q fragments from tensor memory (tq: this thread's columns
// of k-step 0, four per k-step: q hi and q lo words).
template <int KMODE, int G, bool KGEN, int KM, int NT>
__device__ __forceinline__ void qk_tile(const uint8_t* r0, const uint8_t* r1, int tig, int kmis,
                                        const uint32_t (&bq)[8][2], const uint32_t (&bql)[8][2],
                                        uint32_t tq, const uint32_t (&T)[NT][2], const uint2* lut,
                                        uint32_t l8, float (&out)[4], float (&outl)[4])
{
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float scl[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if constexpr (KMODE == 8) {
        const uint32_t* k0p = reinterpret_cast<const uint32_t*>(r0 + 4 * tig);
        const uint32_t* k1p = reinterpret_cast<const uint32_t*>(r1 + 4 * tig);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t A[4];
            cvt_e4m3x4(k0p[4 * kk], A[0], A[2]);
            cvt_e4m3x4(k1p[4 * kk], A[1], A[3]);
            mma16816(sc[kk & 1], A, bq[kk][0], bq[kk][1]);
            if constexpr (G == 8) mma16816(scl[kk & 1], A, bql[kk][0], bql[kk][1]);
        }
    } else {
        // 2-bit keys: one 32-code group (8 bytes) of each row per thread.
        // The 32 codes = two words; the even codes of a word go to one
        // nibble word and the odd codes to another (code 2i / 2i + 1 of the
        // word in nibble i), so k-step kk covers dims with stride 2
        uint32_t c0[4], c1[4];
        {
            uint32_t w0[2], w1[2];
            lds_words<2, KM>(r0 + 8 * tig, kmis, w0);
            lds_words<2, KM>(r1 + 8 * tig, kmis, w1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                c0[2 * i] = w0[i] & 0x33333333u;
                c0[2 * i + 1] = (w0[i] >> 2) & 0x33333333u;
                c1[2 * i] = w1[i] & 0x33333333u;
                c1[2 * i + 1] = (w1[i] >> 2) & 0x33333333u;
            }
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t s0 = c0[kk >> 1] >> (16 * (kk & 1));
            const uint32_t s1 = c1[kk >> 1] >> (16 * (kk & 1));
            uint32_t Ahi[4], Alo[4] = {0u, 0u, 0u, 0u};
            constexpr bool use_lo = KGEN;     // fp16-exact alpha * c_k: no lo part
            {
                // one lookup per byte plane, then interleave the low and
                // high bytes into half2 registers
                const uint32_t p0 = prmt(T[0][0], T[0][1], s0), p1 = prmt(T[1][0], T[1][1], s0);
                const uint32_t q0 = prmt(T[0][0], T[0][1], s1), q1 = prmt(T[1][0], T[1][1], s1);
                Ahi[0] = prmt(p0, p1, 0x5140u);
                Ahi[2] = prmt(p0, p1, 0x7362u);
                Ahi[1] = prmt(q0, q1, 0x5140u);
                Ahi[3] = prmt(q0, q1, 0x7362u);
                if constexpr (use_lo) {
                    const uint32_t u0 = prmt(T[2][0], T[2][1], s0), u1 = prmt(T[3][0], T[3][1], s0);
                    const uint32_t v0 = prmt(T[2][0], T[2][1], s1), v1 = prmt(T[3][0], T[3][1], s1);
                    Alo[0] = prmt(u0, u1, 0x5140u);
                    Alo[2] = prmt(u0, u1, 0x7362u);
                    Alo[1] = prmt(v0, v1, 0x5140u);
                    Alo[3] = prmt(v0, v1, 0x7362u);
                }
            }
            if constexpr (G == 4) {
                if constexpr (use_lo) {
                    mma16816(sc[0], Ahi, bq[kk][0], bq[kk][1]);
                    mma16816(sc[1], Alo, bq[kk][0], bq[kk][1]);
                } else {
                    mma16816(sc[kk & 1], Ahi, bq[kk][0], bq[kk][1]);
                }
            } else {
                uint4 qf;                           // q hi (x, y) and lo (z, w) of this k-step
                tmem_ld4(tq + 4 * kk, qf);
                tmem_wait_ld();
                mma16816(sc[kk & 1], Ahi, qf.x, qf.y);
                mma16816(scl[0], Ahi, qf.z, qf.w);
                if constexpr (use_lo) mma16816(scl[1], Alo, qf.x, qf.y);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[i] = sc[0][i] + sc[1][i];
        outl[i] = scl[0][i] + scl[1][i];
    }
}

// 3- and 4-bit keys (KB bits per code) through the pair table: the MMA's
// 16 rows are 8 tokens x {hi, lo}: row gid holds token gid's fp16 centroids
// and row gid + 8 their fp16 residuals, so one table load (a code pair's hi
// and lo words) is A registers a0 / a1 (pair 2 kk, columns 2 tig, 2 tig + 1)
// or a2 / a3 (pair 2 kk + 1, columns 2 tig + 8, 2 tig + 9) as loaded, and a
// token's score is the sum of its hi and lo rows.  The thread's 32 codes of
// a token (dims 32 tig .. 32 tig + 31) are 4 KB bytes (12 or 16).  Both 16-row tiles
// at once: the thread's four tokens (rows r[0..3] = tokens gid, gid + 8 of
// tile 0, then of tile 1) share one k-step loop, so the lookups and MMAs of
// the two tiles interleave.  out[rt]: G = 4 -> columns head x {q hi, q lo};
// G = 8 -> q hi (out) and q lo (outl) of 8 heads; [0] / [1] = token gid,
// columns 2 tig / 2 tig + 1; [2] / [3] = token gid + 8.
template <int KB, int G, int KM>
__device__ __forceinline__ void qk_pairs(const uint8_t* const (&r)[4], int tig, int kmis,
                                         const uint32_t (&bq)[8][2], uint32_t tq, const uint2* lut,
                                         uint32_t l8, float (&out)[2][4], float (&outl)[2][4])
{
    uint32_t w[4][KB];
#pragma unroll
    for (int i = 0; i < 4; ++i) lds_words<KB, KM>(r[i] + 4 * KB * tig, kmis, w[i]);
    // G = 8: the q lo part meets only the keys' hi words, as one MMA over
    // the 16 tokens of a row tile (rows = tokens gid, gid + 8); the term it
    // leaves out, k lo . q lo, is below 2^-22 of |k| |q|
    float c[4][4] = {}, d[2][4] = {};
    // G = 8: q fragments of k-step kk + 1 are read from tensor memory while
    // k-step kk runs
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint4 qf;
        if constexpr (G == 8) {
            tmem_ld4(tq + 4 * kk, qf);
            tmem_wait_ld();
        }
        uint2 e0[4], e1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            e0[i] = lut_pair(lut, w[i], 2 * kk, l8);
            e1[i] = lut_pair(lut, w[i], 2 * kk + 1, l8);
            const uint32_t A[4] = {e0[i].x, e0[i].y, e1[i].x, e1[i].y};
            if constexpr (G == 4) mma16816(c[i], A, bq[kk][0], bq[kk][1]);
            else                  mma16816(c[i], A, qf.x, qf.y);
        }
        if constexpr (G == 8) {
#pragma unroll
            for (int rt = 0; rt < 2; ++rt) {
                const uint32_t A[4] = {e0[2 * rt].x, e0[2 * rt + 1].x, e1[2 * rt].x, e1[2 * rt + 1].x};
                mma16816(d[rt], A, qf.z, qf.w);
            }
        }
    }
#pragma unroll
    for (int rt = 0; rt < 2; ++rt) {
        const float (&c0)[4] = c[2 * rt], (&c1)[4] = c[2 * rt + 1];
        out[rt][0] = c0[0] + c0[2];
        out[rt][1] = c0[1] + c0[3];
        out[rt][2] = c1[0] + c1[2];
        out[rt][3] = c1[1] + c1[3];
#pragma unroll
        for (int i = 0; i < 4; ++i) outl[rt][i] = d[rt][i];
    }
}

// P' of one 16-row tile to the B layout of the value MMA: thread (gid, tig)
// feeds column gid for tokens 2 tig, 2 tig + 1 (b0) and 2 tig + 8, 2 tig + 9
// (b1), which QK threads with gid 2 tig and 2 tig + 1 hold (rows gid, gid + 8).
// pp[j][r]: P' of the thread's head j (G = 8: heads 2 tig, 2 tig + 1), row r.
template <int G>
__device__ __forceinline__ void p_to_b(const float (&pp)[G == 8 ? 2 : 1][2], int gid, int tig,
                                       uint32_t (&pb)[2][2])
{
    uint32_t Xh, Yh, Xl, Yl;
    if constexpr (G == 4) {
        float h0, l0, h1, l1;
        split_f16(pp[0][0], h0, l0);
        split_f16(pp[0][1], h1, l1);
        Xh = pack_half2(h0, h1);        // column (head, hi)
        Yh = pack_half2(l0, l1);        // column (head, lo)
        Xl = Yl = 0u;
    } else {
        float h0, l0, h1, l1, h2, l2, h3, l3;
        split_f16(pp[0][0], h0, l0);
        split_f16(pp[0][1], h1, l1);
        split_f16(pp[1][0], h2, l2);
        split_f16(pp[1][1], h3, l3);
        Xh = pack_half2(h0, h1);
        Yh = pack_half2(h2, h3);
        Xl = pack_half2(l0, l1);
        Yl = pack_half2(l2, l3);
    }
    const int src_tig = gid >> 1;
    const bool take_y = gid & 1;
    const int srcA = 4 * (2 * tig) + src_tig, srcB = 4 * (2 * tig + 1) + src_tig;
    constexpr int NP = G == 4 ? 1 : 2;
#pragma unroll
    for (int part = 0; part < NP; ++part) {
        const uint32_t X = part ? Xl : Xh, Y = part ? Yl : Yh;
        const uint32_t ax = __shfl_sync(0xffffffffu, X, srcA), ay = __shfl_sync(0xffffffffu, Y, srcA);
        const uint32_t bx = __shfl_sync(0xffffffffu, X, srcB), by = __shfl_sync(0xffffffffu, Y, srcB);
        const uint32_t XA = take_y ? ay : ax, XB = take_y ? by : bx;
        pb[part][0] = prmt(XA, XB, 0x5410u);
        pb[part][1] = prmt(XA, XB, 0x7632u);
    }
}

// Value MMAs of one 16-row tile: tokens 2 tig + (j & 1) + 8 (j >> 1), dims 16 gid + 2i (+1).
// A value code n (0..15) placed alone in a byte and read as FP8 E4M3 is
// exactly n * 2^-9 (subnormal for n < 8, normal above), and that is a normal
// fp16 number: one conversion instruction turns two such bytes into the
// half2 of an A register.  The accumulators therefore hold 2^-9 of the value
// sums; the epilogue scales them back by 512 (exact).
template <int VBITS, int G, int VM>
__device__ __forceinline__ void pv_tile(const uint8_t* tile_v, int rs, int gid, int tig, int vmis,
                                        const uint32_t (&pb)[2][2], float (&acc)[8][4])
{
    uint32_t vw[4][2];   // per token j of the thread: nibble words of dims 16 gid .. 16 gid + 15
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint8_t* rv = tile_v + (2 * tig + (j & 1) + 8 * (j >> 1)) * rs;
        if constexpr (VBITS == 4) {
            lds_words<2, VM>(rv + 8 * gid, vmis, vw[j]);
        } else if constexpr (VBITS == 2) {
            uint32_t w[1];
            lds_words<1, VM>(rv + 4 * gid, vmis, w);
            vw[j][0] = w[0];
            vw[j][1] = 0u;
        } else {
            // 3 bits: dims 16 gid .. 16 gid + 15 are the 48 bits from byte
            // 6 gid, inside the two aligned words from 6 gid - m (m = its
            // misalignment, 0 or 2); spread to two nibble words
            const int m = ((VM >= 0 ? VM : vmis) + 2 * (gid & 1)) & 2;
            const uint32_t* q = reinterpret_cast<const uint32_t*>(rv + 6 * gid - m);
            const uint32_t x0 = q[0], x1 = q[1];
            const uint32_t lo = __funnelshift_r(x0, x1, 8 * m), hi = x1 >> (8 * m);
            vw[j][0] = spread3(lo);
            vw[j][1] = spread3(__funnelshift_r(lo, hi, 24));
        }
    }
    // MMAs i and i + 1 (dims 16 gid + 2i .. 2i + 3) share one byte gather:
    // ab = [A_i, B_i, A_i+1, B_i+1] with A, B the tokens of k = 2 tig, 2 tig + 1
    // (cd likewise for tokens 2 tig + 8, + 9); its low nibbles give row gid
    // (even dims), its high nibbles row gid + 8 (odd dims).
    if constexpr (VBITS == 2) {
        // byte b of a token's word holds dims 16 gid + 4b .. 4b + 3 (two bits
        // each): ab = [A_b, B_b, A_b+1, B_b+1] feeds MMAs 2b .. 2b + 3
#pragma unroll
        for (int i = 0; i < 8; i += 4) {
            const uint32_t c = uint32_t(i >> 1);
            const uint32_t sel = c | ((c + 4) << 4) | ((c + 1) << 8) | ((c + 5) << 12);
            const uint32_t ab = prmt(vw[0][0], vw[1][0], sel);
            const uint32_t cd = prmt(vw[2][0], vw[3][0], sel);
            uint32_t A[4][4];            // MMAs i .. i + 3
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // two-bit field q of each byte: dim 2i + q (+4 in the high half)
                const uint32_t m = 0x03030303u;
                const int mma = (q >> 1), row = q & 1;
                cvt_e4m3x4((ab >> (2 * q)) & m, A[mma][row], A[mma + 2][row]);
                cvt_e4m3x4((cd >> (2 * q)) & m, A[mma][row + 2], A[mma + 2][row + 2]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                mma16816(acc[i + u], A[u], pb[0][0], pb[0][1]);
                if constexpr (G == 8) mma16816(acc[i + u], A[u], pb[1][0], pb[1][1]);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const uint32_t c = uint32_t(i & 3);
            const uint32_t sel = c | ((c + 4) << 4) | ((c + 1) << 8) | ((c + 5) << 12);
            const uint32_t ab = prmt(vw[0][i >> 2], vw[1][i >> 2], sel);
            const uint32_t cd = prmt(vw[2][i >> 2], vw[3][i >> 2], sel);
            uint32_t A0[4], A1[4];
            cvt_e4m3x4(ab & 0x0F0F0F0Fu, A0[0], A1[0]);
            cvt_e4m3x4((ab >> 4) & 0x0F0F0F0Fu, A0[1], A1[1]);
            cvt_e4m3x4(cd & 0x0F0F0F0Fu, A0[2], A1[2]);
            cvt_e4m3x4((cd >> 4) & 0x0F0F0F0Fu, A0[3], A1[3]);
            mma16816(acc[i], A0, pb[0][0], pb[0][1]);
            if constexpr (G == 8) mma16816(acc[i], A0, pb[1][0], pb[1][1]);
            mma16816(acc[i + 1], A1, pb[0][0], pb[0][1]);
            if constexpr (G == 8) mma16816(acc[i + 1], A1, pb[1][0], pb[1][1]);
        }
    }
}

// KMODE: 8 = FP8 E4M3 keys, 2 / 3 / 4 = 2- / 3- / 4-bit Lloyd-Max keys.
// VBITS: 2, 3 or 4.
// G: 4 (columns = 4 heads x {hi, lo}) or 8 (columns = 8 heads).
// One CTA = (split, sequence); warp w = kv head w; each iteration consumes a
// 32-token tile (two 16-row MMA tiles) with one softmax update.
template <typename TQ, int KMODE, int VBITS, int G, bool SOA, bool SPARSE>
__global__ void __launch_bounds__(512) stage1_mma_kernel(const __grid_constant__ MmaArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    // 3-bit keys: the code-pair centroid table (8 KB; one element elsewhere)
    __shared__ __align__(16) uint2 key_lut[KMODE == 3 ? kLut3Entries : KMODE == 4 ? kLut4Entries : 1];
    // launched as a programmatic dependent of the previous kernel in the
    // stream (typically the store of the step's new tokens): wait for it to
    // complete before the first read of global memory
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // blockIdx.x = (split * nqg + qg) * (Hk / hpc) + kv-head group: the
    // CTAs that read the parts of the same token rows (kv-head groups) and
    // the same pages (query-head groups) are neighbours in launch order, so
    // they run together (DRAM pages and L2 lines are used once)
    const int ngroups = a.Hk / a.hpc;
    const int kvg = blockIdx.x % ngroups;     // which hpc kv heads
    const int qg = (blockIdx.x / ngroups) % a.nqg;   // which 8 query heads of each kv head (G > 8)
    const int split = blockIdx.x / ngroups / a.nqg;
    const int b = a.lpt ? seq_of_rank(a.seq_lens, gridDim.y, blockIdx.y, reinterpret_cast<int*>(smem))
                        : blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int h0 = kvg * a.hpc;               // first kv head of this CTA
    const int h = h0 + warp;                   // this warp's kv head
    // query heads of this CTA per kv head: Greal of them from qh0 (all G
    // when G <= 8); query head of (kv head hh, column g) = hh * Gall + qh0 + g
    const int S = a.num_splits, Hq = a.Hq, Gall = a.G;
    const int qh0 = 8 * qg;
    const int Greal = a.nqg > 1 ? min(8, Gall - qh0) : Gall;
    const int Hc = a.hpc;
    const int nwarps = blockDim.x >> 5;

    const int L = a.seq_lens[b];
    int chunk = (L + S - 1) / S;
    chunk = (chunk + kTile - 1) / kTile * kTile;
    const int t_begin = split * chunk;
    const int t_end = min(L, t_begin + chunk);

    if (t_begin >= t_end || a.num_blocks <= 0) {
        // empty split: lse = -inf and a zero partial; tokens but no cache
        // block to read them from: a NaN lse
        const float lse0 = t_begin >= t_end ? -INFINITY : __int_as_float(0x7fc00000);
        for (int i = threadIdx.x; i < Hc * Greal * (kHeadDim + 1); i += blockDim.x) {
            const int r = i / (kHeadDim + 1), d = i % (kHeadDim + 1);
            const int hq = (h0 + r / Greal) * Gall + qh0 + r % Greal;
            float* m = a.mid + (((long long)b * Hq + hq) * S + split) * (kHeadDim + 1);
            m[d] = d == kHeadDim ? lse0 : 0.f;
        }
        return;
    }

    // ---------------- shared-memory ring of 32 token rows (the CTA's kv
    // heads), filled by bulk (TMA) copies.  Rows of one page are contiguous in
    // global memory: one copy per page segment when the CTA takes whole rows
    // and the shared row stride equals the global one, else one copy per row
    // (issued by the 32 lanes of one warp).
    const int row_bytes = a.row_bytes;        // global token row (Hk slots)
    const int cb = a.copy_bytes;              // bytes of it this CTA copies (SoA: data part)
    const int rs = a.smem_row;                // shared row stride: 16 mod 32 bytes
    const int mb = SOA ? a.meta_bytes : 0;    // SoA: metadata part per token, rows after the data rows
    const int stage_bytes = kTile * (rs + mb);
    const int NST = a.nstages;
    const int ntiles = (t_end - t_begin + kTile - 1) / kTile;
    const int32_t* bt = a.block_table + (long long)b * a.bt_stride;
    const int lg = a.bs_log2;
    const int seg_rows = kTile < (1 << lg) ? kTile : (1 << lg);   // rows per page segment
    const int seg_lg = lg < 5 ? lg : 5;                                  // log2(seg_rows)
    // Per stage: `full` completes when the stage's bytes have landed; `done`
    // counts the warps finished with it.  The warp that finishes a stage last
    // refills it, so warps never wait on each other, only on data.
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * stage_bytes);
    int* done = reinterpret_cast<int*>(full + NST);
    int* bad_pages = done + NST;               // a block-table entry outside the cache was met
    int* finished = bad_pages + 1;             // warps past their epilogue
    // MSE keys with G = 8 keep their q fragments (hi and lo, 32 words per
    // thread) in tensor memory: 32 columns per group of 4 warps, the address
    // written by the allocation to the word after the stage counters
    constexpr bool kQt = KMODE != 8 && G == 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + NST * stage_bytes + 16 * NST);
    const uint32_t q_cols = nwarps <= 4 ? 32u : nwarps <= 8 ? 64u : 128u;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) { mbar_init(&full[i], 1); done[i] = 0; }
        *bad_pages = 0;
        *finished = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (kQt) {
        if (warp == 0) tmem_alloc(tmem_slot, q_cols);
        tmem_fence_before_sync();
    }
    __syncthreads();
    uint32_t tq = 0;                           // this thread's q columns (k-step 0)
    if constexpr (kQt) {
        tmem_fence_after_sync();
        tq = *reinterpret_cast<volatile uint32_t*>(tmem_slot) + ((32u * uint32_t(warp & 3)) << 16) +
             32u * uint32_t(warp >> 2);
    }
    // Only rows of tokens < L are copied: block-table entries past the
    // sequence's last page are never read.  Skipped rows keep stale bytes and
    // are masked out of the softmax.
    // SoA blocks: the token rows' data parts and metadata parts lie in two
    // regions of the block; each row (or page segment) takes one copy per
    // region, the metadata landing in rows of mb bytes after the data rows.
    constexpr bool soa = SOA;                  // the block convention (a.g.soa), fixed per instantiation
    const long long hs_g = soa ? a.g.data_bytes : a.g.slot;    // head stride in a global data row
    const long long drow = soa ? (long long)a.Hk * a.g.data_bytes : row_bytes;
    bool bad_seen = false;                     // this lane replaced a page outside the cache
    // tensor copies land on 128-byte aligned stage and segment offsets
    // (stage_bytes and the segment size are multiples of 128 for these
    // rows); a ring base that is not would take the per-row copies
    // (FP8 keys only: the other instantiations carry no tensor-copy code)
    const bool use_tm = KMODE == 8 && !soa && a.use_tmap && (smem_u32(smem) & 127u) == 0;
    auto issue = [&](int tile, int stage) {   // called by all lanes of one warp
        if (tile >= ntiles) return;
        uint8_t* dst = smem + stage * stage_bytes;
        uint64_t* bar = &full[stage];
        const int tbase = t_begin + tile * kTile;
        // data rows: one copy per page segment when the CTA takes whole rows
        // and the shared stride equals the global one, or through the tensor
        // map (a box of the CTA's part of a segment's rows), else one per
        // row; SoA metadata rows (unpadded in shared memory): one copy per
        // page segment when the CTA takes every kv head
        const bool seg_d = (rs == drow && cb == drow) || use_tm;
        const bool seg_m = soa && mb == a.Hk * a.g.meta_bytes;
        const int len_d = seg_d ? seg_rows : 1, len_m = seg_m ? seg_rows : 1;   // rows per copy
        const int lg_d = seg_d ? seg_lg : 0, lg_m = seg_m ? seg_lg : 0;      // (powers of two)
        const int nd = min(kTile >> lg_d, (L - tbase + len_d - 1) >> lg_d);
        const int nm = soa ? min(kTile >> lg_m, (L - tbase + len_m - 1) >> lg_m) : 0;
        if (lane == 0) {
            fence_async_shared();             // prior generic reads of this stage before the async writes
            // the test hook's tile expects 16 bytes that no copy brings: its
            // stage never completes and the bounded waits run out
            const uint32_t extra =
                (tile == a.stuck_tile && split == 0 && qg == 0 && b == 0 && kvg == 0) ? 16u : 0u;
            mbar_expect_tx(bar, uint32_t(nd * len_d * cb + nm * len_m * mb) + extra);
        }
        __syncwarp();
        const bool same = !soa || len_d == len_m;     // one address computation for both copies
        // a block-table entry outside [0, num_blocks) is replaced by page 0,
        // so nothing outside the cache is read, and noted: the CTA's rows
        // come out NaN (see the end of the kernel)
        if (lane < nd) {
            const int t = tbase + lane * len_d;
            long long page = bt[t >> lg];
            if ((unsigned long long)page >= (unsigned long long)a.num_blocks) { page = 0; bad_seen = true; }
            const int off = t & ((1 << lg) - 1);
            const uint8_t* blk = a.cache + (page << lg) * (long long)row_bytes;
            if (KMODE == 8 && !soa && use_tm) {
                tma_load_2d(dst + lane * len_d * rs, &a.tmap, int(h0 * hs_g) >> 2, int((page << lg) + off), bar);
            } else {
                const uint8_t* src =
                    soa ? blk + off * drow + h0 * hs_g : blk + off * (long long)row_bytes + h0 * hs_g;
                bulk_g2s(dst + lane * len_d * rs, src, uint32_t(len_d * cb), bar);
            }
            if (soa && same) {
                const uint8_t* meta = blk + (1LL << lg) * drow + ((long long)off * a.Hk + h0) * a.g.meta_bytes;
                bulk_g2s(dst + kTile * rs + lane * len_m * mb, meta, uint32_t(len_m * mb), bar);
            }
        }
        if (!same && lane < nm) {
            const int t = tbase + lane * len_m;
            long long page = bt[t >> lg];
            if ((unsigned long long)page >= (unsigned long long)a.num_blocks) { page = 0; bad_seen = true; }
            const int off = t & ((1 << lg) - 1);
            const uint8_t* blk = a.cache + (page << lg) * (long long)row_bytes;
            const uint8_t* meta = blk + (1LL << lg) * drow + ((long long)off * a.Hk + h0) * a.g.meta_bytes;
            bulk_g2s(dst + kTile * rs + lane * len_m * mb, meta, uint32_t(len_m * mb), bar);
        }
    };
    // The q staging area (hpc x (4 or 8) heads x 512 B) sits at the end of the
    // ring: the tiles whose stages lie wholly before it are requested first,
    // so their latency overlaps the preparation of q.
    const int q_base = NST * stage_bytes - Hc * G * kHeadDim * 4;
    const int s_q = q_base / stage_bytes;
    if (warp == 0)
        for (int i = 0; i < s_q; ++i) issue(i, i);

    // ---------------- q columns: B operand of the score MMA.  Each warp
    // rotates (MSE keys) and scales its G query heads with lane l holding dims
    // 4l..4l+3, parks them in the staging area, and every thread reads back
    // the 32 values of its column.  The k index of k-step kk and thread tig
    // maps to dims
    //   FP8 keys:   16 kk + 4 tig + j   one key word per k-step, bank-conflict
    //               free across the warp
    //   3-bit keys: 32 tig + 4 kk + j   12 bytes (32 codes) per thread and row
    //   4-bit keys: the same, 16 bytes per thread
    //   2-bit keys: 32 tig + 16 (kk >> 2) + 8 (kk & 1) + ((kk >> 1) & 1) + 2 j
    //               (8 bytes per thread; see qk_tile)
    // 2-bit keys: the host passes a scale alpha that makes every alpha * c_k
    // of the library's codebook an fp16 value to 5e-7 relative.  If that holds
    // for the centroids given (the same test in every thread), the keys use
    // fp16(alpha c_k) alone and q carries 1 / alpha: no lo lookups or MMAs.
    float key_alpha = 1.f;
    bool key_lo = KMODE != 8;
    if constexpr (KMODE == 2) {
        const float al = a.key_alpha;
        float err = (al >= 1.f && al < 2.f) ? 0.f : INFINITY;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float x = al * a.centroids[k];
            const float d = fabsf(x - __half2float(__float2half_rn(x)));
            err = fmaxf(err, x != 0.f ? d / fabsf(x) : d);
        }
        if (err <= 5e-7f) { key_alpha = al; key_lo = false; }
    }

    // 3- and 4-bit keys: entry e (codes e mod 2^bits and e >> bits) of the
    // pair table holds fp16x2 (hi) and fp16x2 (lo) of the two centroids, once
    // per half-warp lane; the barrier after the q staging below orders it
    // before any use
    if constexpr (KMODE == 3 || KMODE == 4) {
        // one (entry, two copies) per step: a 16-byte store of the entry twice
        constexpr int NE = KMODE == 3 ? kLut3Entries : kLut4Entries;
        for (int i = threadIdx.x; i < NE / 2; i += blockDim.x) {
            const int e = i >> 3;
            float h0, l0, h1, l1;
            split_f16(a.centroids[e & ((1 << KMODE) - 1)], h0, l0);
            split_f16(a.centroids[e >> KMODE], h1, l1);
            const uint32_t x = pack_half2(h0, h1), y = pack_half2(l0, l1);
            reinterpret_cast<uint4*>(key_lut)[i] = make_uint4(x, y, x, y);
        }
    }

    // MSE keys with G = 8 keep their q fragments in tensor memory (read once
    // per k-step) instead of 32 registers (the register file is the limit of
    // that instantiation) or 4 KB of shared memory per warp (which a third
    // ring stage needs).
    uint32_t bq[8][2], bql[8][2];
    {
        float* sq = reinterpret_cast<float*>(smem + q_base) + warp * G * kHeadDim;
        float sgn[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sgn[i] = KMODE == 8 ? 1.f : float(a.signs[4 * lane + i]);
        const TQ* Q = static_cast<const TQ*>(a.query);
        for (int g = 0; g < G; ++g) {
            float qv[4] = {0.f, 0.f, 0.f, 0.f};
            if (g < Greal) {        // warp-uniform
                const TQ* qp = Q + ((long long)b * Hq + h * Gall + qh0 + g) * kHeadDim + 4 * lane;
#pragma unroll
                for (int i = 0; i < 4; ++i) qv[i] = sgn[i] * to_f32(qp[i]);
                if constexpr (KMODE != 8) {
                    fwht128_warp(qv, lane);
#pragma unroll
                    for (int i = 0; i < 4; ++i) qv[i] *= 0.08838834764831845f;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) qv[i] *= a.qscale / key_alpha;
            }
            reinterpret_cast<float4*>(sq + g * kHeadDim)[lane] = make_float4(qv[0], qv[1], qv[2], qv[3]);
        }
        __syncwarp();
        const int col_head = G == 4 ? (gid >> 1) : gid;
        const bool col_lo = G == 4 && (gid & 1);
        const float* qc = sq + col_head * kHeadDim;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            float4 x;
            if constexpr (KMODE == 2) {
                // dims 32 tig + 16 (kk >> 2) + 8 (kk & 1) + ((kk >> 1) & 1) + 2 j
                const float* qd = qc + 32 * tig + 16 * (kk >> 2) + 8 * (kk & 1) + ((kk >> 1) & 1);
                x = make_float4(qd[0], qd[2], qd[4], qd[6]);
            } else {
                x = reinterpret_cast<const float4*>(qc + (KMODE == 8 ? 16 * kk + 4 * tig : 32 * tig + 4 * kk))[0];
            }
            float hi[4], lo[4];
            split_f16(x.x, hi[0], lo[0]);
            split_f16(x.y, hi[1], lo[1]);
            split_f16(x.z, hi[2], lo[2]);
            split_f16(x.w, hi[3], lo[3]);
            if (G == 4) {
                bq[kk][0] = col_lo ? pack_half2(lo[0], lo[1]) : pack_half2(hi[0], hi[1]);
                bq[kk][1] = col_lo ? pack_half2(lo[2], lo[3]) : pack_half2(hi[2], hi[3]);
                bql[kk][0] = bql[kk][1] = 0u;
            } else {
                bq[kk][0] = pack_half2(hi[0], hi[1]);
                bq[kk][1] = pack_half2(hi[2], hi[3]);
                bql[kk][0] = pack_half2(lo[0], lo[1]);
                bql[kk][1] = pack_half2(lo[2], lo[3]);
                if constexpr (kQt) {
                    tmem_st4(tq + 4 * kk, make_uint4(bq[kk][0], bq[kk][1], bql[kk][0], bql[kk][1]));
                    bq[kk][0] = bq[kk][1] = bql[kk][0] = bql[kk][1] = 0u;
                }
            }
        }
        if constexpr (kQt) tmem_wait_st();
        __syncthreads();            // every warp is done with the staging area
    }
    if (warp == 0)
        for (int i = s_q; i < NST; ++i) issue(i, i);

    // ---------------- centroid byte planes for the PRMT lookup (2-bit keys):
    // plane 0/1 = low/high byte of fp16(c), plane 2/3 = low/high byte of the
    // fp16 residual c - fp16(c), with c = key_alpha * c_k; T[p][0] holds the
    // four codes' bytes of plane p
    uint32_t T[4][2] = {};
    if constexpr (KMODE == 2) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float c = key_alpha * a.centroids[k];
            const __half chi = __float2half_rn(c);
            const __half clo = __float2half_rn(c - __half2float(chi));
            const uint32_t hb = __half_as_ushort(chi), lb = __half_as_ushort(clo);
            const int sh = 8 * k;
            T[0][0] |= (hb & 0xFFu) << sh;
            T[1][0] |= (hb >> 8) << sh;
            T[2][0] |= (lb & 0xFFu) << sh;
            T[3][0] |= (lb >> 8) << sh;
        }
    }

    constexpr int NH = G == 8 ? 2 : 1;        // query heads per thread (softmax state)
    float m_run[NH], l_run[NH], z_run[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) { m_run[j] = -INFINITY; l_run[j] = 0.f; z_run[j] = 0.f; }
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    const int tau0 = gid, tau1 = gid + 8;      // this thread's QK rows
    const uint32_t l8 = uint32_t(lane & 15) * 8;   // this lane's copy in a pair-table entry
    const int hoff = warp * int(hs_g);         // this warp's slot (SoA: data record) in a shared row
    const int kmis = hoff & 2;
    const int vmis = (hoff + a.g.v_off) & 2;
    // metadata rows: AoS = the data rows (fields inside the slot); SoA = the
    // rows after the data rows, mb bytes each
    const int mrs = soa ? mb : rs;
    const int moff = soa ? kTile * rs + warp * a.g.meta_bytes : hoff;

    // One 32-token tile in stage memory st (this warp's slot at offset 0).
    // PARTIAL: some of its tokens lie at or past t_end and are masked.
    // KGEN: the general key path; false: 2-bit keys without the lo part
    // (key_alpha)
    // KM / VM: the key / value misalignment of this warp's slot (0 or 2)
    auto tile = [&](const uint8_t* st, const uint8_t* sm, int t0, auto partial_tag, auto lo_tag,
                    auto km_tag, auto vm_tag) {
        constexpr bool PARTIAL = decltype(partial_tag)::value;
        [[maybe_unused]] constexpr bool KGEN = decltype(lo_tag)::value;
        constexpr int KM = decltype(km_tag)::value, VM = decltype(vm_tag)::value;
        // ---- scores of both 16-row tiles
        float s[NH][2][2], vs[2][2], vz[2][2];
        bool ok[2][2];
        [[maybe_unused]] float sc2[2][4], scl2[2][4];
        if constexpr (KMODE == 3 || KMODE == 4) {
            const uint8_t* const rr[4] = {st + tau0 * rs, st + tau1 * rs, st + (16 + tau0) * rs,
                                          st + (16 + tau1) * rs};
            qk_pairs<KMODE, G, KM>(rr, tig, kmis, bq, tq, key_lut, l8, sc2, scl2);
        }
#pragma unroll
        for (int rt = 0; rt < 2; ++rt) {
            [[maybe_unused]] const uint8_t* r0 = st + (16 * rt + tau0) * rs;
            [[maybe_unused]] const uint8_t* r1 = st + (16 * rt + tau1) * rs;
            const uint8_t* m0 = sm + (16 * rt + tau0) * mrs;
            const uint8_t* m1 = sm + (16 * rt + tau1) * mrs;
            float sc[4], scl[4];
            if constexpr (KMODE == 3 || KMODE == 4) {
#pragma unroll
                for (int i = 0; i < 4; ++i) { sc[i] = sc2[rt][i]; scl[i] = scl2[rt][i]; }
            } else {
                qk_tile<KMODE, G, KGEN, KM>(r0, r1, tig, kmis, bq, bql, tq, T, key_lut, l8, sc, scl);
            }
            float n0 = 1.f, n1 = 1.f;
            if constexpr (KMODE != 8) { n0 = lds_f16(m0 + a.g.m_norm); n1 = lds_f16(m1 + a.g.m_norm); }
            vs[rt][0] = lds_f16(m0 + a.g.m_scale);
            vz[rt][0] = lds_f16(m0 + a.g.m_zero);
            vs[rt][1] = lds_f16(m1 + a.g.m_scale);
            vz[rt][1] = lds_f16(m1 + a.g.m_zero);
            ok[rt][0] = !PARTIAL || t0 + 16 * rt + tau0 < t_end;
            ok[rt][1] = !PARTIAL || t0 + 16 * rt + tau1 < t_end;
            if constexpr (G == 4) {
                s[0][rt][0] = (sc[0] + sc[1]) * n0;
                s[0][rt][1] = (sc[2] + sc[3]) * n1;
            } else {
                s[0][rt][0] = (sc[0] + scl[0]) * n0;
                s[1][rt][0] = (sc[1] + scl[1]) * n0;
                s[0][rt][1] = (sc[2] + scl[2]) * n1;
                s[1][rt][1] = (sc[3] + scl[3]) * n1;
            }
        }

        // ---- one online-softmax update for the 32 tokens (log2 units).  The
        // running max only moves when a head's tile max exceeds it by more
        // than 8 (so p <= 2^8 otherwise), or when a value scale above 128
        // could take p * v_scale out of the fp16 range of P'.  Moving it
        // rescales the accumulators; keeping it changes no result, since
        // o and l share the same reference.
        float mt[NH];
        bool need = false;
#pragma unroll
        for (int j = 0; j < NH; ++j) {
            float m = -INFINITY;
#pragma unroll
            for (int rt = 0; rt < 2; ++rt)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (!ok[rt][r]) s[j][rt][r] = -INFINITY;
                    m = fmaxf(m, s[j][rt][r]);
                }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
            mt[j] = m;               // finite: the tile's first token is valid
            need |= m > m_run[j] + 8.f;
        }
        need |= fmaxf(fmaxf(vs[0][0], vs[0][1]), fmaxf(vs[1][0], vs[1][1])) > 128.f;
        if (__any_sync(0xffffffffu, need)) {
            float alpha[NH];
#pragma unroll
            for (int j = 0; j < NH; ++j) {
                const float mn = fmaxf(m_run[j], mt[j]);
                alpha[j] = fast_exp2(m_run[j] - mn);
                m_run[j] = mn;
                l_run[j] *= alpha[j];
                z_run[j] *= alpha[j];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if constexpr (G == 4) {
                    acc[i][0] *= alpha[0]; acc[i][1] *= alpha[0]; acc[i][2] *= alpha[0]; acc[i][3] *= alpha[0];
                } else {
                    acc[i][0] *= alpha[0]; acc[i][2] *= alpha[0]; acc[i][1] *= alpha[1]; acc[i][3] *= alpha[1];
                }
            }
        }
        // Sparse V: a row whose p (against the running reference max, never
        // above the final max) is at most vthr keeps its softmax weight in l
        // but adds nothing to the value sum; a 16-row tile with no such row
        // left skips its value MMAs (SPARSE instantiations only).
        float pp[2][NH][2];   // [row tile][head][row]: P' = p * v_scale
        bool vlive[2] = {!SPARSE, !SPARSE};    // 16-row tiles that keep a row
#pragma unroll
        for (int j = 0; j < NH; ++j) {
            float lsum = 0.f, zsum = 0.f;
#pragma unroll
            for (int rt = 0; rt < 2; ++rt)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float p = fast_exp2(s[j][rt][r] - m_run[j]);   // 0 for masked rows
                    lsum += p;
                    if constexpr (SPARSE) {
                        const bool keep = ok[rt][r] && p > a.vthr;
                        vlive[rt] |= keep;
                        zsum += keep ? p * vz[rt][r] : 0.f;
                        pp[rt][j][r] = keep ? p * vs[rt][r] : 0.f;
                    } else {
                        zsum += ok[rt][r] ? p * vz[rt][r] : 0.f;
                        pp[rt][j][r] = ok[rt][r] ? p * vs[rt][r] : 0.f;
                    }
                }
            l_run[j] += lsum;
            z_run[j] += zsum;
        }

        // ---- values
#pragma unroll
        for (int rt = 0; rt < 2; ++rt) {
            if (SPARSE && !__any_sync(0xffffffffu, vlive[rt])) continue;   // warp-uniform
            uint32_t pb[2][2];
            p_to_b<G>(pp[rt], gid, tig, pb);
            pv_tile<VBITS, G, VM>(st + 16 * rt * rs + a.g.v_off, rs, gid, tig, vmis, pb, acc);
        }
    };

    // The tile loop; returns the tile whose wait gave up, or -1.  2-bit keys
    // instantiate it with and without the lo part and pick once per CTA.
    auto run = [&](auto lo_tag, auto km_tag, auto vm_tag) {
        int stage = 0;               // it mod NST
        uint32_t parity = 0;         // (it / NST) mod 2
        for (int it = 0; it < ntiles; ++it) {
            // tile `it` has landed; a copy that never completes ends this warp's
            // heads with a NaN lse instead of hanging (bounded wait)
            const bool ok_wait = mbar_wait(&full[stage], parity, a.wait_polls);
            if (!__all_sync(0xffffffffu, ok_wait)) return it;
            const uint8_t* st = smem + stage * stage_bytes + hoff;
            const uint8_t* sm = smem + stage * stage_bytes + moff;
            const int t0 = t_begin + it * kTile;
            if (t0 + kTile <= t_end) tile(st, sm, t0, std::false_type{}, lo_tag, km_tag, vm_tag);
            else                     tile(st, sm, t0, std::true_type{}, lo_tag, km_tag, vm_tag);

            // ---- this warp is done with the stage; the last warp refills it
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                // release: this warp's reads of the stage come before the
                // count; acquire: the last warp's refill comes after all
                uint32_t prev;
                asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                             : "=r"(prev) : "r"(smem_u32(&done[stage])) : "memory");
                last = prev == uint32_t(nwarps - 1);
                if (last) done[stage] = 0;
            }
            if (__shfl_sync(0xffffffffu, last, 0)) issue(it + NST, stage);
            if (++stage == NST) { stage = 0; parity ^= 1u; }
        }
        return -1;
    };
    // Misalignment of the warp's key and value loads: FP8 keys are read as
    // aligned words and their values start aligned.  3-bit keys with 3-bit
    // values run an instantiation per (key, value) misalignment, picked per
    // warp (4.7% faster on 256K contexts); the other presets test it in the
    // loop (separate instantiations cost them instruction-cache misses).
    using M0 = std::integral_constant<int, 0>;
    using M2 = std::integral_constant<int, 2>;
    using MR = std::integral_constant<int, -1>;
    auto run_mis = [&](auto lo_tag) {
        if constexpr (KMODE == 8) return run(lo_tag, M0{}, M0{});
        else if constexpr (KMODE == 3 && VBITS == 3) {
            if (kmis == 0) return vmis == 0 ? run(lo_tag, M0{}, M0{}) : run(lo_tag, M0{}, M2{});
            else           return vmis == 0 ? run(lo_tag, M2{}, M0{}) : run(lo_tag, M2{}, M2{});
        } else return run(lo_tag, MR{}, MR{});
    };
    int failed_at;
    if constexpr (KMODE == 2) failed_at = key_lo ? run_mis(std::true_type{}) : run_mis(std::false_type{});
    else                      failed_at = run_mis(std::true_type{});
    // stage 2 (a programmatic dependent launch) may start its launch now; it
    // waits for this grid's completion before it reads the partials
    asm volatile("griddepcontrol.launch_dependents;");
    // Run by every warp once its partials are written.  If any warp's copies
    // replaced a page outside the cache, the last warp to get here (when
    // every epilogue of the CTA is done) gives all the CTA's heads a NaN lse.
    auto finish = [&]() {
        __syncwarp();                          // the warp's partial writes before lane 0's count
        const bool wbad = __any_sync(0xffffffffu, bad_seen);
        int last = 0;
        if (lane == 0) {
            if (wbad) atomicOr(bad_pages, 1);
            __threadfence_block();
            last = atomicAdd(finished, 1) == nwarps - 1;
            __threadfence_block();
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();
        if (last && *reinterpret_cast<volatile int*>(bad_pages))
            for (int i = lane; i < Hc * Greal; i += 32)
                a.mid[(((long long)b * Hq + (h0 + i / Greal) * Gall + qh0 + i % Greal) * S + split) *
                          (kHeadDim + 1) + kHeadDim] = __int_as_float(0x7fc00000);
    };
    if (failed_at >= 0) {
        // let the copies that may still be in flight (tiles failed_at ..
        // failed_at + NST - 1) land, with the same bounded wait, then mark
        // this warp's heads as failed
        for (int it = failed_at; it < min(ntiles, failed_at + NST); ++it)
            mbar_wait(&full[it % NST], uint32_t((it / NST) & 1), a.wait_polls);
        if (lane < Greal)
            a.mid[(((long long)b * Hq + h * Gall + qh0 + lane) * S + split) * (kHeadDim + 1) + kHeadDim] =
                __int_as_float(0x7fc00000);
        finish();
    } else {
        // ---------------- epilogue: finish the row sums, write o_s and lse_s.
        // The value accumulators hold 2^-9 of sum_t p_t v_scale_t code_t.
#pragma unroll
        for (int j = 0; j < NH; ++j) {
#pragma unroll
            for (int m = 4; m < 32; m <<= 1) {
                l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], m);
                z_run[j] += __shfl_xor_sync(0xffffffffu, z_run[j], m);
            }
        }
#pragma unroll
        for (int j = 0; j < NH; ++j) {
            const int g = G == 4 ? tig : 2 * tig + j;
            if (g >= Greal) continue;
            const int hq = h * Gall + qh0 + g;
            float* mp = a.mid + (((long long)b * Hq + hq) * S + split) * (kHeadDim + 1);
            const float inv = 1.f / l_run[j];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d = 16 * gid + 2 * i;
                float e, o;
                if constexpr (G == 4) { e = acc[i][0] + acc[i][1]; o = acc[i][2] + acc[i][3]; }
                else { e = j == 0 ? acc[i][0] : acc[i][1]; o = j == 0 ? acc[i][2] : acc[i][3]; }
                mp[d] = (e * 512.f + z_run[j]) * inv;
                mp[d + 1] = (o * 512.f + z_run[j]) * inv;
            }
            if (gid == 0) mp[kHeadDim] = (m_run[j] + log2f(l_run[j])) * 0.6931471805599453f;
        }
        finish();
    }
    // every warp of the CTA is done with its q columns: free them (the
    // allocating warp; all warps reach this point, the waits being bounded)
    if constexpr (kQt) {
        tmem_fence_before_sync();
        __syncthreads();
        if (warp == 0) {
            tmem_fence_after_sync();
            tmem_dealloc(*reinterpret_cast<volatile uint32_t*>(tmem_slot), q_cols);
        }
    }
}

template <typename TQ, int KMODE, int VBITS, int G, bool SPARSE>
cudaError_t launch_t(const MmaArgs& a, int B, size_t smem, cudaStream_t st)
{
    auto k = a.g.soa ? stage1_mma_kernel<TQ, KMODE, VBITS, G, true, SPARSE>
                     : stage1_mma_kernel<TQ, KMODE, VBITS, G, false, SPARSE>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_splits * a.nqg * (a.Hk / a.hpc), B, 1);   // see the kernel's blockIdx.x
    cfg.blockDim = dim3(32 * a.hpc);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a);
}

template <typename TQ, int KMODE, int VBITS, bool SPARSE>
cudaError_t launch_g(const MmaArgs& a, int B, size_t smem, cudaStream_t st)
{
    return a.G <= 4 ? launch_t<TQ, KMODE, VBITS, 4, SPARSE>(a, B, smem, st)
                    : launch_t<TQ, KMODE, VBITS, 8, SPARSE>(a, B, smem, st);
}

template <typename TQ, bool SPARSE>
cudaError_t launch_q(const MmaArgs& a, int B, size_t smem, cudaStream_t st)
{
    if (a.g.key_fp8) return launch_g<TQ, 8, 4, SPARSE>(a, B, smem, st);
    if (a.g.key_bits == 4) return launch_g<TQ, 4, 4, SPARSE>(a, B, smem, st);
    if (a.g.key_bits == 2) return launch_g<TQ, 2, 2, SPARSE>(a, B, smem, st);
    if (a.g.value_bits == 4) return launch_g<TQ, 3, 4, SPARSE>(a, B, smem, st);
    return launch_g<TQ, 3, 3, SPARSE>(a, B, smem, st);
}

}  // namespace
}  // namespace tq
