// lm_head + greedy argmax for callers that cannot allocate device memory.
//
// dg_lm_head_argmax needs a caller workspace for its per-CTA (value, index)
// partials.  Some callers have no way to provide one: a real-time decode loop
// that must not allocate once it is running, a plugin whose host runtime owns
// every byte of device memory through its own pool, or code whose memory plan
// was fixed ahead of time.  This entry point keeps those partials in a fixed
// array that lives inside the library instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kStaticArgParts * 8 bytes until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; later calls reuse it.  The cache is keyed by
// device ordinal only: a cudaDeviceReset invalidates it (documented in dg.h).
#include <mutex>

#include "dg_internal.cuh"

namespace dg {

// 16 KB: one (value, index) per CTA.  A head's grid is at most SMs x 8 CTAs
// (k_gemv runs 256 threads and configure() caps CTAs per SM at 8): 1216 on a
// 152-SM GB300, so the rejection below only triggers above 256 SMs.
constexpr int kStaticArgParts = 2048;

static __device__ __align__(256) ArgPart g_static_arg_parts[kStaticArgParts];

static constexpr int kMaxStaticDevices = 64;
static std::mutex g_static_mu;
static void* g_static_ptr[kMaxStaticDevices];

// Device address of g_static_arg_parts on the current device (set up once per
// device).
static dg_status static_parts(ArgPart** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DG_ERR_CUDA;
    if (dev < 0 || dev >= kMaxStaticDevices) return DG_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> g(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_arg_parts) != cudaSuccess || !p) return DG_ERR_CUDA;
        g_static_ptr[dev] = p;
    }
    *out = static_cast<ArgPart*>(g_static_ptr[dev]);
    return DG_OK;
}

}  // namespace dg

using namespace dg;

extern "C" dg_status dg_lm_head_argmax_noalloc(const dg_linear* head, dg_stream stream) {
    if (!head || !head->token) return DG_ERR_INVALID_ARG;
    dg_status st = validate(*head, false);
    if (st != DG_OK) return st;
    if ((st = check_smem(*head)) != DG_OK) return st;
    if (head_grid(*head) > kStaticArgParts) return DG_ERR_WORKSPACE;  // needs more partials than the array holds
    ArgPart* parts = nullptr;
    if ((st = static_parts(&parts)) != DG_OK) return st;
    return launch_head(*head, parts, stream);
}
