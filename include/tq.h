/*
 * tq.h -- C ABI of the TurboQuant KV-cache hot path on GB300 (sm_103a).
 *
 * The device operations and the host set-up they need:
 *   tq_store            fused quantising store of new K/V tokens into a paged cache
 *   tq_decode_attention split-K decode attention read straight from that cache
 *   tq_dequant          cached slots back to K/V in the original space
 *   tq_build_codebook, tq_make_signs, tq_get_layout   host set-up
 *
 * Cache layout (one combined K+V slot per (block, token, kv head), no leading
 * K/V dimension): uint8 [num_blocks][block_size][num_kv_heads][slot_size_aligned].
 * Source: "vllm-project/vllm pull 38479" digest, section "turboquant_attn.py"
 * (module docstring and get_kv_cache_shape).
 *
 * Slot interior (byte offsets in tq_layout):
 *   [key data][k_norm fp16, MSE presets only][value data][v_scale fp16][v_zero fp16][pad to even]
 * key data is either D bytes of FP8 E4M3 (k8v4) or a b_k-bit packed code
 * stream; value data is a b_v-bit packed code stream.  Every code stream is
 * LSB-first little-endian: code i occupies bits [b*i, b*i + b).  4-bit
 * codes: two per byte, low nibble first; 2-bit: four per byte; 3-bit: 8
 * codes per 3 bytes ("turboquant-plus.md", Background), e.g. codes 0..7 ->
 * bytes 0x88 0xC6 0xFA.  Sizes per
 * "vllm.v1.attention.backends.turboquant_attn" API page,
 * section "__init__" (mse bytes, value data bytes) and section
 * "_continuation_prefill" (field order k_norm, v_scale, v_zero).
 *
 * Conventions for every entry point:
 *   - Device pointers are raw CUDA device addresses on the current device;
 *     host pointers are ordinary host memory.  Each parameter says which.
 *   - The caller owns every buffer.  The library never allocates, frees or
 *     synchronises; device work is enqueued on `stream` (a cudaStream_t,
 *     NULL = legacy default stream) and runs asynchronously.
 *   - Arguments are validated on the host before any launch; on error nothing
 *     is enqueued and a negative TQ_ERR_* code is returned.  TQ_ERR_CUDA means
 *     a launch error reported by cudaGetLastError() right after the launch.
 *   - There is no CPU fallback: without a CUDA device the device entry points
 *     return TQ_ERR_CUDA.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Cache presets: the four cache dtypes of "vllm-project/vllm pull 38479"
 * digest, section "turboquant_attn.py" (supported_kv_cache_dtypes), and the
 * 2-bit Lloyd-Max codebook "Turbo2" of "turboquant-plus.md" (feature table),
 * here in the same slot form as the _nc presets.
 *   TQ_K8V4     FP8 E4M3 keys, 4-bit uniform values               slot 196 B @ D=128
 *   TQ_4BIT_NC  4-bit Lloyd-Max keys + norm correction, 4-bit V  slot 134 B
 *   TQ_K3V4_NC  3-bit Lloyd-Max keys + norm correction, 4-bit V  slot 118 B
 *   TQ_3BIT_NC  3-bit Lloyd-Max keys + norm correction, 3-bit V  slot 102 B
 *   TQ_2BIT_NC  2-bit Lloyd-Max keys + norm correction, 2-bit V  slot  70 B
 * 2-bit codes: four per byte, LSB first. */
typedef enum { TQ_K8V4 = 0, TQ_4BIT_NC = 1, TQ_K3V4_NC = 2, TQ_3BIT_NC = 3, TQ_2BIT_NC = 4 } tq_preset;

/* Byte convention inside a cache block, OR-ed into the preset argument of
 * tq_store, tq_decode_attention(_sparse_v / _noalloc), tq_dequant and
 * tq_decode_pick_splits (tq_get_layout accepts and ignores it).  The cache
 * shape and the slot sizes are the same either way.
 *   default (AoS): one combined slot per (token, kv head) as described above.
 *   TQ_LAYOUT_SOA: a data region of block_size * num_kv_heads records
 *     [key data][value data] (key_data_bytes + value_data_bytes each; record
 *     (t, h) at (t * num_kv_heads + h) * data_bytes from the block start),
 *     then a metadata region of the same number of records of little-endian
 *     uint16 fields, [k_norm][v_scale][v_zero] for the Lloyd-Max presets and
 *     [v_scale][v_zero] for k8v4 (record (t, h) at data region end +
 *     (t * num_kv_heads + h) * 2 * fields).  Source: "vllm.v1.attention.
 *     backends.turboquant_attn" API page, "do_kv_cache_update" (data region +
 *     metadata region separated per block) and "_continuation_prefill"
 *     (metadata field count and order); the record order inside each region
 *     is this library's reading. */
#define TQ_LAYOUT_SOA 0x100

/* Element types of K/V/Q inputs and of the attention output. */
typedef enum { TQ_F16 = 0, TQ_BF16 = 1, TQ_F32 = 2 } tq_dtype;

/* Status codes. */
#define TQ_OK               0
#define TQ_ERR_INVALID_ARG (-1)  /* null pointer, negative or inconsistent size */
#define TQ_ERR_UNSUPPORTED (-2)  /* preset, head_dim, block_size or dtype not served */
#define TQ_ERR_WORKSPACE   (-3)  /* workspace smaller than tq_decode_workspace_bytes() */
#define TQ_ERR_CUDA        (-4)  /* CUDA launch / device error */

/* Byte layout of one slot.  All offsets are from the slot start. */
typedef struct {
    int key_fp8;            /* 1: keys are FP8 E4M3, unrotated, no norm      */
    int key_bits;           /* 8 (fp8) or Lloyd-Max code width 2/3/4          */
    int value_bits;         /* uniform value code width 2/3/4                 */
    int norm_correction;    /* 1: stored norm is ||k|| / ||c[idx]||           */
    int n_centroids;        /* 2^key_bits for MSE keys, 0 for fp8             */
    int key_data_bytes;     /* D (fp8) or ceil(D*key_bits/8)                  */
    int key_packed_size;    /* key data + k_norm                              */
    int value_data_bytes;   /* ceil(D*value_bits/8)                           */
    int value_packed_size;  /* value data + v_scale + v_zero                  */
    int slot_size;          /* key_packed_size + value_packed_size            */
    int slot_size_aligned;  /* slot_size rounded up to an even byte count     */
    int off_k_norm;         /* -1 for fp8 keys                                */
    int off_v_data, off_v_scale, off_v_zero;
} tq_layout;

/* Fill *out with the slot layout of `preset` at `head_dim` (host only; the
 * TQ_LAYOUT_SOA bit is ignored).
 * head_dim must be a positive multiple of 8.  Returns TQ_OK or
 * TQ_ERR_INVALID_ARG / TQ_ERR_UNSUPPORTED. */
int tq_get_layout(int preset, int head_dim, tq_layout* out);

/* Lloyd-Max codebook for coordinates ~ N(0, 1/head_dim) (host only).
 * Source: "vllm-project/vllm pull 38479" digest, section "centroids.py"
 * (solve_lloyd_max: init on [-3.5 sigma, 3.5 sigma], outer edges at 3x that
 * range, 200-panel trapezoid integrals, at most 200 iterations, tolerance
 * 1e-10, previous iterate kept on convergence); midpoints per the API page,
 * section "_ensure_on_device" (fp32 mean of neighbouring fp32 centroids).
 * centroids: host float[2^bits], ascending.  midpoints: host float[2^bits-1]
 * (may be NULL).  bits in 1..8.  Deterministic; returns TQ_OK or
 * TQ_ERR_INVALID_ARG. */
int tq_build_codebook(int head_dim, int bits, float* centroids, float* midpoints);

/* Rademacher sign vector of the randomized Hadamard transform (host only).
 * Source: "turboquant-plus.md", section "Background" (random sign vector
 * before the Walsh-Hadamard transform); the pages name no generator, so
 * s_i = +1 when the top bit of the i-th output of SplitMix64 seeded with
 * `seed` is clear, else -1.  Per-layer seed = 42 + 1337 * layer ("attention.py"
 * section of the PR digest).  signs: host int8[head_dim].  Returns TQ_OK or
 * TQ_ERR_INVALID_ARG. */
int tq_make_signs(int head_dim, uint64_t seed, int8_t* signs);

/* Fused quantising store ("vllm.v1.attention.backends.turboquant_attn" API
 * page, sections "do_kv_cache_update" and "_store_kv"; method per
 * "turboquant-plus.md" section "Background").  For every token n < num_tokens
 * with slot_mapping[n] >= 0 and every kv head h, writes the slot at
 * block slot_mapping[n] / block_size, offset slot_mapping[n] % block_size:
 *   MSE keys: n_k = ||k||; y = H (s . k) / n_k with H the orthonormal
 *     Sylvester Hadamard matrix (fast transform); idx_j = #{midpoints < y_j};
 *     k_norm = fp16(n_k / ||c[idx]||) (norm correction) or fp16(n_k).
 *   FP8 keys: E4M3 of each coordinate, round to nearest even, saturating.
 *   Values: scale = fp16((max-min)/(2^b_v-1)), zero = fp16(min),
 *     code = clamp(rint((v - zero)/scale), 0, 2^b_v-1), 0 when scale == 0, with
 *     v - zero and the quotient each correctly rounded in fp32 and rint
 *     rounding half to even.
 * key, value: device, element type in_dtype, element (n, h, d) at
 *   [n*stride_tok + h*head_dim + d] (stride in elements, >= Hk*head_dim).
 * slot_mapping: device int64[num_tokens]; negative entries are skipped.
 * kv_cache: device uint8 [num_blocks][block_size][num_kv_heads][slot_size_aligned];
 *   must be 16-byte aligned.  Slots beyond num_blocks are a caller error (the
 *   kernel skips them rather than write out of bounds).
 * signs: device int8[head_dim]; centroids: device float[2^key_bits];
 *   midpoints: device float[2^key_bits - 1] (both ignored, may be NULL, for k8v4).
 * Supported: head_dim 128, block_size 16/32/64/128, in_dtype F16/BF16,
 *   1 <= num_kv_heads <= 32.  num_tokens == 0 is a no-op. */
int tq_store(int preset, int head_dim, int num_tokens, int num_kv_heads, int block_size,
             int in_dtype, const void* key, const void* value,
             long long key_stride_tok, long long value_stride_tok,
             const int64_t* slot_mapping, uint8_t* kv_cache, long long num_blocks,
             const int8_t* signs, const float* centroids, const float* midpoints,
             void* stream);

/* Dequantisation of cached slots back to K and V in the original space, the
 * inverse of tq_store for the slots slot_mapping names ("vllm.v1.attention.
 * backends.turboquant_attn" API page, "_continuation_prefill": the cached
 * prefix is dequantised in full and its MSE keys rotated back).  For every
 * token n < num_tokens and kv head h, from the slot at block
 * slot_mapping[n] / block_size, offset slot_mapping[n] % block_size:
 *   MSE keys: k = k_norm * (s . (H c[idx])) with H the orthonormal Sylvester
 *     Hadamard matrix (the store's rotation undone); FP8 keys: E4M3 decoded.
 *   Values: v = code * v_scale + v_zero.
 * Computed in fp32 (fast transform for H) and rounded once to out_dtype.
 * key_out, value_out: device, element type out_dtype (F16/BF16/F32), element
 *   (n, h, d) at [n*stride_tok + h*head_dim + d]; both 16-byte aligned, strides
 *   >= num_kv_heads*head_dim and multiples of 8 elements.
 * slot_mapping: device int64[num_tokens]; a negative slot or one at or beyond
 *   num_blocks*block_size gives zero rows and reads nothing.
 * kv_cache: device, 16-byte aligned, layout as for tq_store.  signs and
 *   centroids: as for tq_store (ignored, may be NULL, for k8v4).
 * Supported: head_dim 128, block_size 16/32/64/128.  num_tokens == 0 is a
 * no-op.  Returns TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED or
 * TQ_ERR_CUDA. */
int tq_dequant(int preset, int head_dim, int num_tokens, int num_kv_heads, int block_size,
               const uint8_t* kv_cache, long long num_blocks, const int64_t* slot_mapping,
               const int8_t* signs, const float* centroids, void* key_out, void* value_out,
               int out_dtype, long long key_stride_tok, long long value_stride_tok, void* stream);

/* Split count the library uses when tq_decode_attention gets num_splits = 0,
 * from host-known sizes (no device memory is read; the current device's SM
 * count and the stage-1 kernel's occupancy are queried, and cached).  It
 * minimises the stage-1 critical path: the waves of (split, sequence, head
 * group) CTAs over the resident CTA slots, times the 32-token tiles of one
 * split plus a fixed start-up cost; splits are at least 128 tokens long.
 * max_seq_len is an upper bound on seq_lens.  Returns a value in
 * [1, TQ_MAX_SPLITS] (1 for non-positive sizes), or TQ_ERR_UNSUPPORTED /
 * TQ_ERR_INVALID_ARG for an unknown preset or head_dim, or a head count that
 * is not a multiple of num_kv_heads.  Without a device it assumes two CTAs
 * per SM of a 152-SM GB300. */
#define TQ_MAX_SPLITS 256
int tq_decode_pick_splits(int preset, int head_dim, int batch, int num_q_heads, int num_kv_heads,
                          int max_seq_len);

/* Bytes of caller-owned workspace tq_decode_attention needs: the stage-1
 * partials mid_o fp32 [batch][num_q_heads][num_splits][head_dim + 1] (column
 * head_dim holds the split's log-sum-exp), per the "attention.py" section of
 * the PR digest.  One workspace may serve every layer in turn. */
size_t tq_decode_workspace_bytes(int batch, int num_q_heads, int num_splits, int head_dim);

/* Split-K decode attention over the compressed cache ("vllm-project/vllm
 * pull 38479" digest, implementation item 4: stage 1 scores and accumulates
 * values per split, stage 2 merges splits by log-sum-exp; API page section
 * "_decode_attention").  For query head hq of sequence b, kv head
 * h = hq / (num_q_heads / num_kv_heads):
 *   stage 1: q_rot = H (s . q) once; for tokens t of the split, page =
 *     block_table[b*block_table_stride + t/block_size]; score = softmax_scale *
 *     k_norm * <q_rot, c[idx]> (MSE) or softmax_scale * <q, k_fp8> (k8v4);
 *     online softmax; v_hat = code * v_scale + v_zero accumulated.
 *     Splits are consecutive token ranges (the tensor-core kernel rounds
 *     their length up to whole 32-token tiles); the result does not depend
 *     on the split count beyond rounding.
 *   stage 2: o = sum_s w_s o_s / sum_s w_s, w_s = exp(lse_s - max lse),
 *     lse = max + ln sum w_s (natural log, scale included).
 * seq_lens[b] == 0 gives o = 0 and lse = -inf.
 * query: device (B, Hq, D) contiguous, q_dtype F16/BF16.
 * kv_cache: device, layout above.  block_table: device int32; entries
 *   at or past ceil(seq_lens[b]/block_size) are never read.  An entry that is
 *   read and lies outside [0, num_blocks) is a caller error: both stage-1
 *   kernels check each page before reading it, read nothing outside the
 *   cache, and the query heads of that sequence come out NaN (output and
 *   lse); other sequences are unaffected (num_blocks = 0: every sequence
 *   with tokens).  The table must hold
 *   ceil(seq_lens[b]/block_size) entries per row (not checked).
 * seq_lens: device int32[B].  max_seq_len: host upper bound of seq_lens.
 * softmax_scale: usually 1/sqrt(head_dim).  num_splits: 0 = tq_decode_pick_splits.
 * signs / centroids: device, as for tq_store (centroids may be NULL for k8v4).
 * out: device (B, Hq, D) of out_dtype F16/BF16/F32.  lse: device float[B*Hq]
 *   or NULL.  workspace: device, >= tq_decode_workspace_bytes(B, Hq, S, D),
 *   16-byte aligned.  Supported: head_dim 128, block_size 16/32/64/128,
 *   num_q_heads % num_kv_heads == 0, group size <= 16. */
int tq_decode_attention(int preset, int head_dim, int batch, int num_q_heads,
                        int num_kv_heads, int block_size, int q_dtype, const void* query,
                        const uint8_t* kv_cache, long long num_blocks,
                        const int32_t* block_table, int block_table_stride,
                        const int32_t* seq_lens, int max_seq_len,
                        float softmax_scale, int num_splits,
                        const int8_t* signs, const float* centroids,
                        void* out, int out_dtype, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream);

/* tq_decode_attention with the sparse-V row skip ("turboquant-plus.md",
 * feature table: sparse V dequant, an attention-gated row skip).  Arguments
 * as tq_decode_attention plus v_threshold in [0, 1).  In stage 1 a token row
 * whose softmax factor p = exp(logit - m) is at most v_threshold, with m the
 * split's running reference max when the row is processed (never above the
 * split's final max), keeps its weight in the softmax denominator but adds
 * nothing to the value sum; the tensor-core kernel skips the value MMAs of a
 * 16-row tile that keeps no row, the CUDA-core kernel skips the value codes
 * of such a row.  v_threshold = 0 is tq_decode_attention exactly.  An
 * approximation: per output dimension the result moves from the dense one by
 * at most sum_{t: exp(logit_t - M) <= v_threshold} p_t |v_t| / sum_t p_t
 * (M the sequence's largest logit); the LSE is unchanged.  Returns as
 * tq_decode_attention, and TQ_ERR_INVALID_ARG for a threshold outside
 * [0, 1). */
int tq_decode_attention_sparse_v(int preset, int head_dim, int batch, int num_q_heads,
                                 int num_kv_heads, int block_size, int q_dtype, const void* query,
                                 const uint8_t* kv_cache, long long num_blocks,
                                 const int32_t* block_table, int block_table_stride,
                                 const int32_t* seq_lens, int max_seq_len, float softmax_scale,
                                 int num_splits, const int8_t* signs, const float* centroids,
                                 void* out, int out_dtype, float* lse, void* workspace,
                                 size_t workspace_bytes, float v_threshold, void* stream);

/* tq_decode_attention without a caller-supplied workspace.  The pages have
 * no counterpart to this entry point: it exists for callers that cannot
 * allocate device memory, for example a serving engine that gives nearly all
 * device memory to its own KV-cache pool at start-up and treats any later
 * cudaMalloc as a failure, or a host loop that must not take cudaMalloc's
 * implicit device-wide synchronisation.  The split partials go to an array of
 * TQ_NOALLOC_SCRATCH_BYTES that the library declares in device memory (every
 * GPU that loads the library holds it until the process exits); this call
 * allocates nothing.  Arguments and results are those of tq_decode_attention
 * minus workspace/workspace_bytes.  num_splits = 0 picks as
 * tq_decode_pick_splits does, lowered until B*Hq*S*(D+1)*4 bytes fit; an
 * explicit num_splits whose partials exceed the array returns
 * TQ_ERR_WORKSPACE, as does a shape for which even one split does not fit.
 * Every call looks up the array's device address in the current device's
 * context (cudaGetSymbolAddress); the first call on a device may load the
 * library's device code there, so make that first call before any stream
 * capture.  All calls share the one array and leave the
 * last call's partials in it (nothing in it has to start at zero): calls
 * whose kernels overlap on the GPU, e.g. on two streams at once, race. */
#define TQ_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int tq_decode_attention_noalloc(int preset, int head_dim, int batch, int num_q_heads,
                                int num_kv_heads, int block_size, int q_dtype, const void* query,
                                const uint8_t* kv_cache, long long num_blocks,
                                const int32_t* block_table, int block_table_stride,
                                const int32_t* seq_lens, int max_seq_len,
                                float softmax_scale, int num_splits,
                                const int8_t* signs, const float* centroids,
                                void* out, int out_dtype, float* lse, void* stream);

/* Test entry point for the bounded waits of the tensor-core stage 1; the
 * pages have no counterpart.  Runs tq_decode_attention (num_splits as there)
 * with every stage wait of stage 1 limited to `wait_polls` mbarrier polls,
 * and makes one wait run out without any fault: the tile `stuck_tile` (0 =
 * first) of split 0 of sequence 0, kv-head group 0, is announced to its
 * mbarrier as 16 bytes longer than the copies that fill it, so every copy
 * lands but that stage never completes.  The warps of that CTA give up after
 * `wait_polls` polls, wait (with the same limit) for the copies they had
 * requested, and give the query heads of that CTA a NaN lse for split 0, so
 * the merged output and lse of those heads of sequence 0 come out NaN; every
 * other output is what tq_decode_attention gives.  Nothing waits without a
 * limit, so the call returns and the context stays usable.
 * TQ_ERR_UNSUPPORTED for shapes the CUDA-core stage 1 serves
 * (tq_decode_kernel_kind != 1); TQ_ERR_INVALID_ARG for stuck_tile < 0 or
 * wait_polls == 0; other errors as tq_decode_attention. */
int tq_test_decode_wait_expiry(int preset, int head_dim, int batch, int num_q_heads,
                               int num_kv_heads, int block_size, int q_dtype, const void* query,
                               const uint8_t* kv_cache, long long num_blocks,
                               const int32_t* block_table, int block_table_stride,
                               const int32_t* seq_lens, int max_seq_len, float softmax_scale,
                               int num_splits, const int8_t* signs, const float* centroids,
                               void* out, int out_dtype, float* lse, void* workspace,
                               size_t workspace_bytes, int stuck_tile, unsigned int wait_polls,
                               void* stream);

/* Which stage-1 kernel tq_decode_attention runs for this shape (host only):
 * 1 = tensor-core stage 1: keys FP8 (k8v4), 3-bit (k3v4_nc, 3bit_nc),
 * 4-bit with 4-bit values (4bit_nc) or 2-bit with 2-bit values (2bit_nc);
 * group size (num_q_heads / num_kv_heads) <= 16 (a CTA takes up to 8 query
 * heads of each kv head); the bytes a CTA copies per token (all kv heads'
 * slots, or 4 heads' for FP8 keys with num_kv_heads a multiple of 4 above
 * 4) a multiple of 16, or a multiple of 4 when they are whole token rows,
 * and at most ~1.7 KB;
 * 0 = CUDA-core stage 1 (every other supported shape); -1 = unsupported. */
int tq_decode_kernel_kind(int preset, int head_dim, int num_q_heads, int num_kv_heads);

/* Human-readable text of a status code (static storage). */
const char* tq_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int tq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */
