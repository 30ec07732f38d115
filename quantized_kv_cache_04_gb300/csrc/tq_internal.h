// Internal declarations shared by the host and CUDA translation units of the
// TurboQuant library.  Not part of the public ABI (include/tq.h is).
#pragma once

#include "tq.h"

#include <cstdint>
#include <cuda_runtime.h>

namespace tq {

constexpr int kHeadDim = 128;     // the served head dimension
constexpr int kMaxGroup = 16;     // query heads per kv head served by decode
constexpr int kNumSMs = 152;      // GB300

int fill_layout(int preset, int head_dim, tq_layout* L);
// Split count for num_splits = 0 (tq_decode.cu): the one that minimises the
// stage-1 critical path over the resident CTA slots of the kernel that runs.
int pick_splits(const tq_layout& L, bool soa, int batch, int num_q_heads, int num_kv_heads, int max_seq_len);

inline bool block_size_ok(int bs) { return bs == 16 || bs == 32 || bs == 64 || bs == 128; }
inline bool in_dtype_ok(int dt) { return dt == TQ_F16 || dt == TQ_BF16; }
inline bool out_dtype_ok(int dt) { return dt == TQ_F16 || dt == TQ_BF16 || dt == TQ_F32; }

// Plain-old-data copy of the slot layout handed to kernels by value, with
// the block byte convention.  Field addresses of record (token t of a block,
// kv head h) come from two pointers, `data` (key data at 0, value data at
// v_off) and `meta` (k_norm / v_scale / v_zero at m_norm / m_scale /
// m_zero): AoS: both are the slot, offsets as in tq_layout; SoA: data record
// and metadata record (TQ_LAYOUT_SOA in tq.h).
struct SlotGeom {
    int key_fp8, key_bits, value_bits, norm_correction;
    int key_data_bytes, off_k_norm, off_v_data, off_v_scale, off_v_zero;
    int slot;        // slot_size_aligned
    int soa;         // 1: TQ_LAYOUT_SOA
    int data_bytes;  // SoA data record: key_data_bytes + value_data_bytes
    int meta_bytes;  // SoA metadata record: 2 * fields
    int v_off;       // value data offset from `data`
    int m_norm, m_scale, m_zero;   // field offsets from `meta`
};

inline SlotGeom geom_of(const tq_layout& L, bool soa = false)
{
    SlotGeom g;
    g.key_fp8 = L.key_fp8;
    g.key_bits = L.key_bits;
    g.value_bits = L.value_bits;
    g.norm_correction = L.norm_correction;
    g.key_data_bytes = L.key_data_bytes;
    g.off_k_norm = L.off_k_norm;
    g.off_v_data = L.off_v_data;
    g.off_v_scale = L.off_v_scale;
    g.off_v_zero = L.off_v_zero;
    g.slot = L.slot_size_aligned;
    g.soa = soa ? 1 : 0;
    g.data_bytes = L.key_data_bytes + L.value_data_bytes;
    g.meta_bytes = L.key_fp8 ? 4 : 6;
    if (soa) {
        g.v_off = L.key_data_bytes;
        g.m_norm = L.key_fp8 ? -1 : 0;
        g.m_scale = L.key_fp8 ? 0 : 2;
        g.m_zero = L.key_fp8 ? 2 : 4;
    } else {
        g.v_off = L.off_v_data;
        g.m_norm = L.off_k_norm;
        g.m_scale = L.off_v_scale;
        g.m_zero = L.off_v_zero;
    }
    return g;
}

// Preset argument: low byte = preset, TQ_LAYOUT_SOA bit = block convention.
inline bool layout_flags_ok(int preset) { return (preset & ~(0xFF | TQ_LAYOUT_SOA)) == 0; }
inline bool is_soa(int preset) { return (preset & TQ_LAYOUT_SOA) != 0; }

#ifdef __CUDACC__
// Data and metadata pointers of record (block `page`, token `off`, head h).
__device__ __forceinline__ void slot_ptrs(const SlotGeom& g, const uint8_t* cache, long long page, int off,
                                          int h, int bs, int Hk, const uint8_t*& data, const uint8_t*& meta)
{
    if (g.soa) {
        const uint8_t* blk = cache + page * bs * (long long)Hk * g.slot;
        const long long rec = (long long)off * Hk + h;
        data = blk + rec * g.data_bytes;
        meta = blk + (long long)bs * Hk * g.data_bytes + rec * g.meta_bytes;
    } else {
        data = cache + ((page * bs + off) * (long long)Hk + h) * g.slot;
        meta = data;
    }
}
#endif

// Tensor-core stage 1 (tq_decode_mma.cu): which shapes it serves, and its launcher.
bool mma_stage1_supported(const tq_layout& L, bool soa, int num_kv_heads, int group);
// CTAs one split of one sequence launches, and resident CTA slots on num_sms
// SMs (0 when the occupancy query fails, e.g. without a device).
void mma_stage1_shape(const tq_layout& L, bool soa, int num_kv_heads, int group, int num_sms,
                      int* ctas_per_split, int* slots);
// Polls of a stage's mbarrier before stage 1 gives up on it (the split's
// lse becomes NaN); each poll sleeps at most 20 us waiting for the phase,
// so a stage that never completes is given up after about 1.3 s.  A test
// may pass a small count and a stuck tile.
constexpr uint32_t kWaitPolls = 1u << 16;
int launch_mma_stage1(const tq_layout& L, bool soa, int q_dtype, const void* query, const uint8_t* kv_cache,
                      long long num_blocks, const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                      float softmax_scale, int num_splits, const int8_t* signs,
                      const float* centroids, float* mid, int B, int Hq, int Hk, int bs,
                      float v_threshold, cudaStream_t st, int stuck_tile = -1,
                      uint32_t wait_polls = kWaitPolls);

}  // namespace tq
