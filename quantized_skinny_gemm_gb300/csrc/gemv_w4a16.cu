// Groupwise int4 weights with fp16 activations (and the int4 lm_head).
#include "gemv_core.cuh"

namespace dg {

cudaError_t gemv_w4a16(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ) {
    return run_family<PolicyW4A16>(L, p, s, occ);
}

}  // namespace dg
