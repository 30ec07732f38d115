/*
 * tq_oracle.h -- plain, slow CPU oracle for the TurboQuant KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes,
 * links or calls this code; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no header, helper or table
 * with the CUDA path.  It is written from the pages, step by step, in
 * double precision except where the method itself fixes a narrower
 * precision (fp16 norms/scales, fp32 codebook, fp32 decisions).
 *
 * Page titles used in citations:
 *   [vLLM-PR]   "vllm-project/vllm pull 38479" digest (TurboQuant backend):
 *               sections "turboquant_attn.py", "centroids.py", "attention.py".
 *   [vLLM-API]  "vllm.v1.attention.backends.turboquant_attn" API page:
 *               "_ensure_on_device", "_store_kv", "_continuation_prefill",
 *               "_decode_attention".
 *   [Atlas]     "turboquant-plus.md" (Atlas TQ+): "Background", feature table.
 *   [Issue]     "TurboQuant/HIGGS Attention follow-ups" tracking issue.
 */
#ifndef TQ_ORACLE_H
#define TQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Preset numbering (the four cache dtypes named in [vLLM-PR]
 * "turboquant_attn.py" supported_kv_cache_dtypes). */
#define ORC_K8V4    0
#define ORC_4BIT_NC 1
#define ORC_K3V4_NC 2
#define ORC_3BIT_NC 3
#define ORC_2BIT_NC 4   /* Turbo2: 2-bit Lloyd-Max keys + norm correction, 2-bit values */
/* OR-ed into a preset: the SoA byte convention inside each cache block (a
 * data region of [key data][value data] records, then a metadata region of
 * uint16 [k_norm][v_scale][v_zero] records, [v_scale][v_zero] for FP8 keys;
 * record (t, h) at index t * Hk + h of each region).  Slot bytes are the
 * same; only where they sit in the block changes. */
#define ORC_LAYOUT_SOA 0x100

/* Slot layout derived from [vLLM-API] "__init__" (mse bytes / value data
 * bytes formulas) and [vLLM-API] "_continuation_prefill" (field order
 * k_norm, v_scale, v_zero).  All offsets in bytes inside one slot. */
typedef struct {
    int key_fp8, key_bits, value_bits, norm_correction;
    int key_data_bytes;   /* D (fp8) or ceil(D*b_k/8)            */
    int off_k_norm;       /* -1 when the preset stores no norm    */
    int off_v_data, value_data_bytes;
    int off_v_scale, off_v_zero;
    int slot_size, slot_size_aligned;
} orc_layout;

int orc_get_layout(int preset, int head_dim, orc_layout* out);

/* ---- scalar formats -------------------------------------------------- */
double   orc_f16_to_double(uint16_t h);
uint16_t orc_double_to_f16(double x);       /* IEEE binary16, RNE       */
float    orc_bf16_to_float(uint16_t b);
uint8_t  orc_e4m3_encode(double x);         /* OCP E4M3FN, RNE, satfinite */
double   orc_e4m3_decode(uint8_t b);

/* ---- codebook ([vLLM-PR] "centroids.py": solve_lloyd_max) ------------- */
/* centroids64: the double iterate the algorithm returns (2^bits entries).
 * c32 / m32: fp32 centroids, and fp32 midpoints of the fp32 centroids as
 * [vLLM-API] "_ensure_on_device" forms them.  Any output may be NULL.
 * Returns the number of iterations run. */
int orc_lloyd_max(int d, int bits, int trapz_n, int max_iter, double tol,
                  double* centroids64, float* c32, float* m32);

/* ---- rotation ---------------------------------------------------------- */
/* Rademacher signs: s_i = +1 when the top bit of the i-th output of
 * SplitMix64 seeded with `seed` is 0, else -1. */
void orc_signs(int D, uint64_t seed, int8_t* s);
/* Normalised Sylvester Hadamard H[i][j] = (-1)^popcount(i&j) / sqrt(D). */
void orc_hadamard(int D, double* H);

/* ---- bit packing: every width LSB-first, code i at bits [b*i, b*i+b) of
 *      the little-endian byte stream (3 bits: 8 codes per 3 bytes) ---- */
void orc_pack(const int* codes, int n, int bits, uint8_t* out);
void orc_unpack(const uint8_t* in, int n, int bits, int* codes);

/* ---- store ------------------------------------------------------------- */
/* One (token, kv head): k, v are the exact fp32 values of the fp16/bf16
 * inputs.  Writes slot_size_aligned bytes to `slot`.  y32 (may be NULL)
 * receives the fp32 pre-quantisation coordinates (MSE presets) so a test
 * can find codes that sit on a decision boundary. */
int orc_store_one(int preset, int D, const float* k, const float* v,
                  const int8_t* signs, const float* c32, const float* m32,
                  uint8_t* slot, float* y32);

/* Whole batch: key/value (N, Hk, D) fp32; cache (num_blocks, bs, Hk, slot).
 * slot_mapping < 0 skips the token. */
int orc_store(int preset, int D, int N, int Hk, int bs,
              const float* key, const float* value, const int64_t* slot_mapping,
              uint8_t* cache, int64_t num_blocks,
              const int8_t* signs, const float* c32, const float* m32);

/* ---- dequantisation of one cached slot to the original space ---------- */
int orc_dequant_slot(int preset, int D, const uint8_t* slot,
                     const int8_t* signs, const float* c32,
                     double* k_hat, double* v_hat);

/* ---- decode attention --------------------------------------------------- */
/* Dense definition: dequantise every cached token, logits = scale*q.k_hat,
 * softmax in double.  q (B, Hq, D) fp32.  out (B, Hq, D), lse (B, Hq). */
int orc_decode_dense(int preset, int D, int B, int Hq, int Hk, int bs,
                     const float* q, const uint8_t* cache, int64_t num_blocks,
                     const int32_t* block_table, int64_t bt_stride,
                     const int32_t* seq_lens, double scale,
                     const int8_t* signs, const float* c32,
                     double* out, double* lse);

/* Split-K form: q rotated once, scores as norm * <q_rot, c[idx]>, per-split
 * softmax partials, then the log-sum-exp merge.  Same outputs. */
int orc_decode_split(int preset, int D, int B, int Hq, int Hk, int bs,
                     const float* q, const uint8_t* cache, int64_t num_blocks,
                     const int32_t* block_table, int64_t bt_stride,
                     const int32_t* seq_lens, double scale, int num_splits,
                     const int8_t* signs, const float* c32,
                     double* out, double* lse);

/* Sparse V ("turboquant-plus.md", feature table: attention-gated row skip
 * of the value dequantisation): a row t may drop out of the value sum when
 * its softmax factor exp(l_t - M) is at most tau (M = the sequence's largest
 * logit).  The output then moves from the dense one by at most
 *   bound[b, hq, d] = sum_{t: exp(l_t - M) <= tau} p_t |v_t,d| / sum_t p_t
 * and mass[b, hq] = sum_{t: exp(l_t - M) <= tau} p_t / sum_t p_t is the
 * weight of the rows that may drop.  Dense logits as orc_decode_dense. */
int orc_sparse_v_bound(int preset, int D, int B, int Hq, int Hk, int bs,
                       const float* q, const uint8_t* cache, int64_t num_blocks,
                       const int32_t* block_table, int64_t bt_stride,
                       const int32_t* seq_lens, double scale, double tau,
                       const int8_t* signs, const float* c32,
                       double* bound, double* mass);

#ifdef __cplusplus
}
#endif
#endif
