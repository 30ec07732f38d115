// Tensor-core decode stage 1 with the sparse-V gate: its instantiations,
// compiled apart from the dense ones (the kernel is in tq_decode_mma.cuh).
#include "tq_decode_mma.cuh"

namespace tq {

cudaError_t launch_mma_sparse(const MmaArgs& a, int q_dtype, int B, size_t smem, cudaStream_t st)
{
    return q_dtype == TQ_F16 ? launch_q<__half, true>(a, B, smem, st)
                             : launch_q<__nv_bfloat16, true>(a, B, smem, st);
}

}  // namespace tq
