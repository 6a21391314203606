// W8A8: int8 weights x int8 activations, exact int32 accumulation.
#include "gemv_core.cuh"

namespace dg {

cudaError_t gemv_i8(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ) {
    return run_family<PolicyI8>(L, p, s, occ);
}

}  // namespace dg
