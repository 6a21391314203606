// Groupwise int4 weights with fp16 activations (and the int4 lm_head).
#include "gemv_core.cuh"

namespace dg {

cudaError_t gemv_w4a16(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ) {
    return run_family<PolicyW4A16>(L, p, s, occ);
}

size_t w4_mma_smem(int K) { return smem_bytes_for<PolicyW4A16>(1, K, kW4MmaRows); }

}  // namespace dg
