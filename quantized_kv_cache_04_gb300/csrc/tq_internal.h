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
int pick_splits(const tq_layout& L, int batch, int num_q_heads, int num_kv_heads, int max_seq_len);

inline bool block_size_ok(int bs) { return bs == 16 || bs == 32 || bs == 64 || bs == 128; }
inline bool in_dtype_ok(int dt) { return dt == TQ_F16 || dt == TQ_BF16; }
inline bool out_dtype_ok(int dt) { return dt == TQ_F16 || dt == TQ_BF16 || dt == TQ_F32; }

// Plain-old-data copy of the slot layout handed to kernels by value.
struct SlotGeom {
    int key_fp8, key_bits, value_bits, norm_correction;
    int key_data_bytes, off_k_norm, off_v_data, off_v_scale, off_v_zero;
    int slot;   // slot_size_aligned
};

inline SlotGeom geom_of(const tq_layout& L)
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
    return g;
}

// Tensor-core stage 1 (tq_decode_mma.cu): which shapes it serves, and its launcher.
bool mma_stage1_supported(const tq_layout& L, int num_kv_heads, int group);
// CTAs one split of one sequence launches, and resident CTA slots on num_sms
// SMs (0 when the occupancy query fails, e.g. without a device).
void mma_stage1_shape(const tq_layout& L, int num_kv_heads, int group, int num_sms, int* ctas_per_split,
                      int* slots);
int launch_mma_stage1(const tq_layout& L, int q_dtype, const void* query, const uint8_t* kv_cache,
                      const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                      float softmax_scale, int num_splits, const int8_t* signs,
                      const float* centroids, float* mid, int B, int Hq, int Hk, int bs,
                      float v_threshold, cudaStream_t st);

}  // namespace tq
