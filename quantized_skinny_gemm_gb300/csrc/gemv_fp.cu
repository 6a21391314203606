// fp16 / bf16 weight streaming (and the fp16 / bf16 lm_head with argmax).
#include "gemv_core.cuh"

namespace dg {

cudaError_t gemv_fp(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ) {
    if (L.fmt == F_BF16) return run_family<PolicyFP<true>>(L, p, s, occ);
    return run_family<PolicyFP<false>>(L, p, s, occ);
}

}  // namespace dg
