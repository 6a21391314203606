// Groupwise int4 weights with per-token int8 activations (and the int4 lm_head).
#include "gemv_core.cuh"

namespace dg {

cudaError_t gemv_w4a8(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ) {
    return run_family<PolicyW4A8>(L, p, s, occ);
}

size_t gemv_smem(Fmt f, int MT, int K, int group) {
    switch (f) {
        case F_F16:
        case F_BF16: return smem_bytes_for<PolicyFP<false>>(MT, K);
        case F_I8: return smem_bytes_for<PolicyI8>(MT, K);
        case F_W4A16: return smem_bytes_for<PolicyW4A16>(MT, K);
        case F_W4A8: return smem_bytes_for<PolicyW4A8>(MT, K);
    }
    return 0;
}

}  // namespace dg
