// Tensor-core decode stage 1: launch geometry, occupancy, dispatch, and the
// dense instantiations (the kernel itself is in tq_decode_mma.cuh).
#include "tq_decode_mma.cuh"

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdint>
#include <cstring>

namespace tq {

cudaError_t launch_mma_dense(const MmaArgs& a, int q_dtype, int B, size_t smem, cudaStream_t st)
{
    return q_dtype == TQ_F16 ? launch_q<__half, false>(a, B, smem, st)
                             : launch_q<__nv_bfloat16, false>(a, B, smem, st);
}

namespace {

// ---- 2-bit keys: a centroid scale alpha in [1, 2) with every alpha * c_k
// of the library's codebook (two magnitudes) an fp16 value to ~1e-7
// relative, so the score MMAs need no lo part.  Searched once per process
// on the host, rounding like the device (the fp32 product, then
// nearest-even fp16); candidates make one entry exact, plus a uniform grid.
// The kernel checks the result against the centroids it is given.
double round_f16(double x)
{
    if (x == 0.0) return 0.0;
    int e;
    const double m = std::frexp(x, &e);              // |m| in [0.5, 1)
    if (e - 1 < -14) return std::nearbyint(x * 16777216.0) / 16777216.0;   // subnormal: 2^-24 steps
    return std::ldexp(std::nearbyint(std::ldexp(m, 11)), e - 11);
}

double hi_error(const float* c, int n, float alpha)
{
    double err = 0.0;
    for (int k = 0; k < n; ++k) {
        const double x = double(alpha * c[k]);
        const double d = std::fabs(x - round_f16(x));
        err = std::fmax(err, x != 0.0 ? d / std::fabs(x) : d);
    }
    return err;
}

float two_bit_alpha()
{
    static const float alpha = [] {
        float c[4], mid[4];
        if (tq_build_codebook(kHeadDim, 2, c, mid) != TQ_OK) return 0.f;
        double best = INFINITY;
        float best_a = 0.f;
        auto consider = [&](double g) {
            const float a = float(g);
            if (!(a >= 1.f && a < 2.f)) return;
            const double e = hi_error(c, 4, a);
            if (e < best || (e == best && a < best_a)) { best = e; best_a = a; }
        };
        for (int k = 0; k < 4; ++k) {
            int e;
            const double f = 2.0 * std::frexp(std::fabs(double(c[k])), &e);   // in [1, 2)
            if (!(f >= 1.0)) continue;
            for (int m = 0; m < 1024; ++m) {
                double g = (1.0 + m / 1024.0) / f;
                consider(g < 1.0 ? 2.0 * g : g);
            }
        }
        for (int i = 0; i < 65536; ++i) consider(1.0 + i / 65536.0);
        return best <= 5e-7 ? best_a : 0.f;
    }();
    return alpha;
}

// cuTensorMapEncodeTiled, through the runtime's driver entry point (no link
// against the driver library); null when unavailable.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled()
{
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return EncodeTiledFn(nullptr);
        }
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// The cache as `rows` rows of row_bytes (32-bit words), boxes of box_bytes x
// box_rows.  False when the map cannot be encoded.
bool encode_rows_map(CUtensorMap* map, const void* base, long long rows, int row_bytes, int box_bytes,
                     int box_rows)
{
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(row_bytes / 4), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
    const cuuint32_t box[2] = {cuuint32_t(box_bytes / 4), cuuint32_t(box_rows)};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch geometry shared by the launcher and the occupancy query.
struct MmaGeom {
    int hpc, copy_bytes, smem_row, meta_bytes, nstages;
    size_t smem;          // dynamic shared memory
    size_t static_smem;   // the kernel's own: the 3- or 4-bit keys' pair table
};

MmaGeom mma_geom(const tq_layout& L, bool soa, int Hk, int G)
{
    MmaGeom m;
    const SlotGeom g = geom_of(L, soa);
    const int rec = soa ? g.data_bytes : L.slot_size_aligned;   // data bytes per (token, head)
    // FP8-key rows split into CTAs of 4 kv heads (4 records are a whole number
    // of 16-byte copy units): half-size CTAs, four per SM, each waiting on
    // only 4 warps before a stage is refilled; AoS rows arrive by one tensor
    // copy per page segment (the launcher's map)
    m.hpc = (L.key_fp8 && Hk % 4 == 0 && Hk > 4 && (4 * rec) % 16 == 0 &&
             (!soa || (4 * g.meta_bytes) % 16 == 0))
                ? 4 : Hk;
    m.copy_bytes = m.hpc * rec;
    m.meta_bytes = soa ? m.hpc * g.meta_bytes : 0;
    // a shared row stride of 16 mod 32 bytes (4 mod 8 words) puts the rows a
    // warp reads in the same instruction on distinct bank quads
    m.smem_row = (m.copy_bytes % 32 == 0) ? m.copy_bytes + 16 : m.copy_bytes;
    const int stage = kTile * (m.smem_row + m.meta_bytes);
    // ring budget: two CTAs of 8 kv-head warps, or four CTAs of 4 warps, per
    // SM (about 16 warps); fewer kv heads take a proportional share (at
    // least 28 KB), so that CTAs of 2 or 4 warps still fill an SM.  3- and
    // 4-bit keys hold their pair table (8 / 32 KB) in static shared memory;
    // MSE keys with G = 8 keep their q fragments in tensor memory
    m.static_smem = L.key_fp8 ? 0 : L.key_bits == 3 ? size_t(kLut3Entries) * 8
                                   : L.key_bits == 4 ? size_t(kLut4Entries) * 8 : 0;
    const int budget = m.hpc < Hk ? 56 * 1024 : (Hk >= 8 ? 100 * 1024 : std::max(28 * 1024, 100 * 1024 * Hk / 8));
    int nst = (budget - int(m.static_smem)) / stage;
    nst = nst < 2 ? 2 : (nst > 6 ? 6 : nst);
    // the q staging at kernel start borrows the ring: hpc * (4 or 8) heads * 512 B
    while (nst * stage < m.hpc * (G <= 4 ? 4 : 8) * kHeadDim * 4) ++nst;
    m.nstages = nst;
    // ring, mbarrier + counter per stage, the tensor-memory address
    m.smem = size_t(nst) * stage + 16 * size_t(nst) + 16;
    return m;
}

template <int KMODE, int VBITS, int G>
int slots_t(const MmaGeom& m, bool soa, int num_sms)
{
    auto k = soa ? stage1_mma_kernel<__nv_bfloat16, KMODE, VBITS, G, true, false>
                 : stage1_mma_kernel<__nv_bfloat16, KMODE, VBITS, G, false, false>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(m.smem)) != cudaSuccess)
        return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 32 * m.hpc, m.smem) != cudaSuccess)
        return 0;
    if constexpr (KMODE != 8 && G == 8) {
        // The instantiations that allocate tensor memory (32-128 of an SM's
        // 512 columns per CTA) are reported at one CTA per SM, but run as
        // many as registers and shared memory allow (two of 8 warps with 3-bit
        // keys: one wave of 296 CTAs at batch 8 takes one wave's time)
        cudaFuncAttributes at;
        int dev = 0, smem_sm = 0, reserved = 0;
        if (cudaFuncGetAttributes(&at, k) == cudaSuccess && at.numRegs > 0 && cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess) {
            const int regs = (at.numRegs + 7) / 8 * 8;
            const int by_regs = 65536 / (regs * 32 * m.hpc);
            const int by_smem = int(size_t(smem_sm) / (m.smem + at.sharedSizeBytes + size_t(reserved)));
            const int by_warps = 64 / m.hpc;
            per_sm = std::max(per_sm, std::min(std::min(by_regs, by_smem), by_warps));
        }
        cudaGetLastError();
    }
    return per_sm * num_sms;
}

}  // namespace

bool mma_stage1_supported(const tq_layout& L, bool soa, int num_kv_heads, int group)
{
    const bool keys_ok = (L.key_fp8 && L.value_bits == 4) ||
                         (!L.key_fp8 && (L.key_bits == 3 || (L.key_bits == 4 && L.value_bits == 4) ||
                                         (L.key_bits == 2 && L.value_bits == 2)));
    const bool vals_ok = L.value_bits >= 2 && L.value_bits <= 4;
    if (!keys_ok || !vals_ok || num_kv_heads < 1 || group < 1 || group > kMaxGroup) return false;
    const MmaGeom m = mma_geom(L, soa, num_kv_heads, group);
    const int row = m.copy_bytes;
    // Copies are 16-byte units: rows of a multiple of 16 bytes are copied
    // one by one (or per page segment); an AoS CTA that takes whole rows of
    // a multiple of 4 bytes copies whole page segments (16 or 32 rows: a
    // multiple of 16 bytes, from a 16-byte aligned page offset) into an
    // unpadded ring.  Rows must stay 4-byte aligned for the word loads.
    const bool rows_ok = row % 16 == 0 || (!soa && m.hpc == num_kv_heads && row % 4 == 0);
    return m.hpc <= 16 && rows_ok && m.meta_bytes % 16 == 0 &&
           2 * kTile * (row + 16 + m.meta_bytes) <= 110 * 1024;
}

void mma_stage1_shape(const tq_layout& L, bool soa, int num_kv_heads, int group, int num_sms,
                      int* ctas_per_split, int* slots)
{
    const MmaGeom m = mma_geom(L, soa, num_kv_heads, group);
    *ctas_per_split = num_kv_heads / m.hpc * (group > 4 ? (group + 7) / 8 : 1);
    int n = 0;
    if (num_sms > 0) {
        if (L.key_fp8) n = group <= 4 ? slots_t<8, 4, 4>(m, soa, num_sms) : slots_t<8, 4, 8>(m, soa, num_sms);
        else if (L.key_bits == 4) n = group <= 4 ? slots_t<4, 4, 4>(m, soa, num_sms) : slots_t<4, 4, 8>(m, soa, num_sms);
        else if (L.key_bits == 2) n = group <= 4 ? slots_t<2, 2, 4>(m, soa, num_sms) : slots_t<2, 2, 8>(m, soa, num_sms);
        else if (L.value_bits == 4) n = group <= 4 ? slots_t<3, 4, 4>(m, soa, num_sms) : slots_t<3, 4, 8>(m, soa, num_sms);
        else n = group <= 4 ? slots_t<3, 3, 4>(m, soa, num_sms) : slots_t<3, 3, 8>(m, soa, num_sms);
    }
    if (n <= 0) {
        // no device to ask: a GB300 SM's 228 KB of shared memory (1 KB kept
        // per CTA) and 64K registers at 128 per thread
        const int by_smem = int((228 * 1024) / (m.smem + m.static_smem + 1024));
        const int by_regs = 65536 / (128 * 32 * m.hpc);
        n = (by_smem < by_regs ? by_smem : by_regs) * kNumSMs;
    }
    *slots = n;
}

int launch_mma_stage1(const tq_layout& L, bool soa, int q_dtype, const void* query, const uint8_t* kv_cache,
                      long long num_blocks, const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                      float softmax_scale, int num_splits, const int8_t* signs,
                      const float* centroids, float* mid, int B, int Hq, int Hk, int bs,
                      float v_threshold, cudaStream_t st, int stuck_tile,
                      uint32_t wait_polls)
{
    MmaArgs a;
    a.vthr = v_threshold;
    a.stuck_tile = stuck_tile;
    a.wait_polls = wait_polls;
    a.key_alpha = (!L.key_fp8 && L.key_bits == 2) ? two_bit_alpha() : 0.f;
    a.query = query;
    a.cache = kv_cache;
    a.num_blocks = num_blocks;
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.seq_lens = seq_lens;
    a.qscale = softmax_scale * 1.4426950408889634f;
    a.num_splits = num_splits;
    a.signs = signs;
    a.centroids = centroids;
    a.mid = mid;
    a.Hq = Hq;
    a.Hk = Hk;
    a.G = Hq / Hk;
    a.bs = bs;
    a.bs_log2 = bs == 16 ? 4 : bs == 32 ? 5 : bs == 64 ? 6 : 7;
    a.row_bytes = Hk * L.slot_size_aligned;
    const MmaGeom m = mma_geom(L, soa, Hk, a.G);
    a.hpc = m.hpc;
    // groups above 8: CTAs of 8 query heads per kv head, each reading the
    // kv heads' rows (neighbouring CTAs: the second read mostly hits L2)
    a.nqg = a.G > 4 ? (a.G + 7) / 8 : 1;
    a.copy_bytes = m.copy_bytes;
    // CTAs of part of each AoS row (FP8 keys, 4 kv heads): a page segment's
    // parts by one tensor copy instead of one bulk copy per row, when the
    // rows land unpadded (784-byte parts: 16 mod 32) and the map's limits
    // hold (16-byte aligned cache and row stride, at most 256 words per box
    // row, rows addressable as int)
    a.use_tmap = 0;
    std::memset(&a.tmap, 0, sizeof(a.tmap));
    const int seg_rows = bs < kTile ? bs : kTile;
    if (!soa && m.hpc < Hk && m.smem_row == m.copy_bytes && m.copy_bytes % 16 == 0 && m.copy_bytes / 4 <= 256 &&
        a.row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(kv_cache) & 15) == 0 && num_blocks > 0 &&
        num_blocks * bs <= 0x7fffffffLL)
        a.use_tmap = encode_rows_map(&a.tmap, kv_cache, num_blocks * bs, a.row_bytes, m.copy_bytes, seg_rows) ? 1 : 0;
    a.smem_row = m.smem_row;
    a.meta_bytes = m.meta_bytes;
    a.nstages = m.nstages;
    a.g = geom_of(L, soa);
    a.lpt = (B <= 512 && m.smem >= size_t(4) * (B + 1)) ? 1 : 0;
    const cudaError_t e = v_threshold > 0.f ? launch_mma_sparse(a, q_dtype, B, m.smem, st)
                                            : launch_mma_dense(a, q_dtype, B, m.smem, st);
    return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace tq
