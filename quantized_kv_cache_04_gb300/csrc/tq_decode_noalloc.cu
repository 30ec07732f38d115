// Decode attention for callers that cannot allocate device memory.
//
// tq_decode_attention needs a caller-owned workspace for the split partials.
// Some callers have no way to provide one: a serving engine that hands almost
// all device memory to its own KV-cache pool at start-up and treats any later
// cudaMalloc as a failure, or a host program whose latency-critical loop must
// not pay cudaMalloc's implicit device-wide synchronisation.  This entry point
// runs the same decode with the partials in a fixed-size array that the
// library itself declares in device memory, so the call allocates nothing.
#include "tq.h"
#include "tq_internal.h"

namespace {

// The split partials (fp32 [batch][q heads][splits][head_dim + 1]).  Every GPU
// that loads the library holds TQ_NOALLOC_SCRATCH_BYTES of it until the
// process exits.  Its name is only a host-side stand-in: host code must use
// the device address from cudaGetSymbolAddress.
static __device__ __align__(256) float tq_noalloc_scratch[TQ_NOALLOC_SCRATCH_BYTES / sizeof(float)];

}  // namespace

extern "C" int tq_decode_attention_noalloc(int preset, int head_dim, int batch, int num_q_heads,
                                           int num_kv_heads, int block_size, int q_dtype,
                                           const void* query, const uint8_t* kv_cache,
                                           long long num_blocks, const int32_t* block_table,
                                           int block_table_stride, const int32_t* seq_lens,
                                           int max_seq_len, float softmax_scale, int num_splits,
                                           const int8_t* signs, const float* centroids, void* out,
                                           int out_dtype, float* lse, void* stream)
{
    // The array's address in the current device's context, looked up on
    // every call: an address kept from an earlier call could belong to
    // another context (after cudaDeviceReset, or under a driver-API context
    // that is not the primary one).  Once the library's device code is
    // loaded in the context this is a host-side table lookup.
    void* scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, tq_noalloc_scratch) != cudaSuccess || !scratch) {
        cudaGetLastError();
        return TQ_ERR_CUDA;
    }

    // With num_splits = 0 the library's pick is lowered until the partials
    // fit; an explicit split count that does not fit is rejected.
    int splits = num_splits;
    if (batch > 0 && num_q_heads > 0 && head_dim > 0 && num_splits >= 0) {
        const size_t per_split = tq_decode_workspace_bytes(batch, num_q_heads, 1, head_dim);
        if (splits == 0) {
            splits = tq_decode_pick_splits(preset, head_dim, batch, num_q_heads, num_kv_heads,
                                           max_seq_len);
            if (splits < 0) return splits;
            const size_t fit = per_split ? TQ_NOALLOC_SCRATCH_BYTES / per_split : 0;
            if ((size_t)splits > fit) splits = (int)fit;
        }
        if (splits < 1 ||
            tq_decode_workspace_bytes(batch, num_q_heads, splits, head_dim) > TQ_NOALLOC_SCRATCH_BYTES)
            return TQ_ERR_WORKSPACE;
    }
    return tq_decode_attention(preset, head_dim, batch, num_q_heads, num_kv_heads, block_size, q_dtype,
                               query, kv_cache, num_blocks, block_table, block_table_stride, seq_lens,
                               max_seq_len, softmax_scale, splits, signs, centroids, out, out_dtype, lse,
                               scratch, TQ_NOALLOC_SCRATCH_BYTES, stream);
}
