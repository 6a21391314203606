// C ABI of libdg.so: host-side validation, launch configuration and the
// decode-step sequencer.  Nothing here allocates device memory or
// synchronizes (except dg_check_device_status).
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "dg_internal.cuh"

namespace dg {

// ---- device facts ------------------------------------------------------------------

static constexpr int kMaxDevices = 64;

int sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

size_t smem_optin_limit() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v) return (size_t)v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return 0;
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
    return (size_t)n;
}

// The library's device error word (bounded waits record kErrTimeout here),
// located once per device.
static __device__ int g_dg_error = 0;

int* device_error_word() {
    static std::mutex mu;
    static int* cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> g(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dg_error) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<int*>(p);
    }
    return cache[dev];
}

// ---- tuning knobs ------------------------------------------------------------------
// DG_TUNE="R=2,KS=1,CPS=4,PF=32768,PDL=1,STEP=1,SPIN=20000000,SNW=16,MMA=1,TC=8"
// overrides the launch heuristic (for configuration sweeps); an unset key
// keeps the heuristic's choice.  STEP=0 runs decode steps as one launch per
// fused group instead of the persistent step kernel; STEP=2 puts a grid
// barrier between every pair of phases of the persistent kernel.
struct Tune {
    int R = 0, KS = 0, CPS = 0, PF = -1, PDL = -1, STEP = -1, SPIN = -1, SNW = 0, MMA = -1;
    int KP = 0;                                // split-K ranges of a per-op launch (1 = off)
    int TC = -1;                               // fewest tokens on the tcgen05 tile (0 = off)
    int TG = 0;                                // CTAs of the tcgen05 tile (0 = one per SM)
    int TS = 0;                                // TMA ring stages of the tcgen05 tile (6, 8, 12)
    int TP = -1;                               // weight boxes the tcgen05 tile prefetches early
    int TQ = -1;                               // fewest tokens on the int8 / int4 tcgen05 tile (0 = off)
    int TK = 0;                                // 64-k boxes per stage of the fp16 tcgen05 tile (1, 2; 0 = 2)
};

static Tune read_tune() {
    Tune t;
    const char* e = std::getenv("DG_TUNE");
    if (!e) return t;
    char buf[256];
    std::strncpy(buf, e, sizeof buf - 1);
    buf[sizeof buf - 1] = 0;
    for (char* tok = std::strtok(buf, ","); tok; tok = std::strtok(nullptr, ",")) {
        int v = 0;
        if (std::sscanf(tok, "R=%d", &v) == 1) t.R = v;
        else if (std::sscanf(tok, "KS=%d", &v) == 1) t.KS = v;
        else if (std::sscanf(tok, "CPS=%d", &v) == 1) t.CPS = v;
        else if (std::sscanf(tok, "PF=%d", &v) == 1) t.PF = v;
        else if (std::sscanf(tok, "PDL=%d", &v) == 1) t.PDL = v;
        else if (std::sscanf(tok, "STEP=%d", &v) == 1) t.STEP = v;
        else if (std::sscanf(tok, "SPIN=%d", &v) == 1) t.SPIN = v;
        else if (std::sscanf(tok, "SNW=%d", &v) == 1) t.SNW = v;
        else if (std::sscanf(tok, "MMA=%d", &v) == 1) t.MMA = v;
        else if (std::sscanf(tok, "KP=%d", &v) == 1) t.KP = v;
        else if (std::sscanf(tok, "TC=%d", &v) == 1) t.TC = v;
        else if (std::sscanf(tok, "TG=%d", &v) == 1) t.TG = v;
        else if (std::sscanf(tok, "TS=%d", &v) == 1) t.TS = v;
        else if (std::sscanf(tok, "TP=%d", &v) == 1) t.TP = v;
        else if (std::sscanf(tok, "TQ=%d", &v) == 1) t.TQ = v;
        else if (std::sscanf(tok, "TK=%d", &v) == 1) t.TK = v;
    }
    return t;
}

static const Tune& tune() {
    static Tune t = read_tune();
    return t;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = tune().PDL == 0 ? 0 : 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// ---- launch configuration ------------------------------------------------------------

static size_t elem_row_bytes(Fmt f, int K) {
    switch (f) {
        case F_F16:
        case F_BF16: return (size_t)K * 2;
        case F_I8: return (size_t)K;
        default: return (size_t)K / 2;
    }
}

static int pick_mt(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

// Warps per row: a function of the row length only, so that a row's summation
// order never depends on N (see the kernel's header comment).
static int pick_ks(Fmt f, int K) {
    const int t = tune().KS;
    if (t == 1 || t == 2 || t == 4 || t == 8) return t;
    const size_t rb = elem_row_bytes(f, K);
    if (rb >= 16384) return 4;
    if (rb >= 8192) return 2;
    return 1;
}

// Rows per slot.  At one token: W4A16 four (its MAC loads each activation
// piece once for all rows of the slot), W4A8 and int8 two, fp16 / bf16 one.
static int pick_r(Fmt f, int MT, int K) {
    (void)K;
    const int t = tune().R;
    if (t == 1 || t == 2 || t == 4) return t;
    // one token: W4A16 four rows per slot (activation pieces shared), W4A8 and
    // W8A8 two (W8A8 14336x4096: 11.8 -> 10.8 us with the 64 KB prefetch)
    if (MT == 1) return f == F_W4A16 ? 4 : (f == F_W4A8 || f == F_I8) ? 2 : 1;
    if (MT <= 4) return 2;
    if (f == F_I8) return MT >= 16 ? 4 : 2;
    return 1;
}

static cudaError_t family(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ) {
    switch (L.fmt) {
        case F_F16:
        case F_BF16: return gemv_fp(L, p, s, occ);
        case F_I8: return gemv_i8(L, p, s, occ);
        case F_W4A16: return gemv_w4a16(L, p, s, occ);
        case F_W4A8: return gemv_w4a8(L, p, s, occ);
    }
    return cudaErrorInvalidValue;
}

static int occupancy(const GemvLaunch& L) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, (int)L.fmt, L.MT, L.R, (int)L.argmax, L.K, L.group);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int occ = 0;
    if (family(L, nullptr, nullptr, &occ) != cudaSuccess) occ = 1;
    if (occ < 1) occ = 1;
    std::lock_guard<std::mutex> g(mu);
    cache[key] = occ;
    return occ;
}

// Fills L.grid and p.iters / ksplit / prefetch for a launch over p.N rows.
static void configure(GemvLaunch& L, GemvParams& p) {
    const int ks = pick_ks(L.fmt, p.a.K);
    const int slots = kWarps / ks;
    const int n_rg = (p.t.N + L.R - 1) / L.R;
    const int need = (n_rg + slots - 1) / slots;
    int cps = occupancy(L);
    const int tc = tune().CPS;
    cps = tc > 0 ? (tc < cps ? tc : cps) : (cps < 8 ? cps : 8);
    int maxg = sm_count() * cps;
    if (maxg < 1) maxg = 1;
    if (L.argmax && maxg > kMaxArgCtas) maxg = kMaxArgCtas;
    int grid = need < maxg ? need : maxg;
    const int iters = (n_rg + grid * slots - 1) / (grid * slots);
    grid = (n_rg + slots * iters - 1) / (slots * iters);  // even out the last pass
    L.grid = grid;
    p.ksplit = ks;
    p.iters = iters;
    // first rows warmed in L2 per CTA before the dependency wait (64 KB: W8A8
    // 14336x4096 at 1 / 4 tokens 11.2 -> 10.8 / 14.7 -> 14.5 us, fp16 2048^2 even)
    p.prefetch_bytes = tune().PF >= 0 ? tune().PF : 65536;
}

static dg_status to_status(cudaError_t e) { return e == cudaSuccess ? DG_OK : DG_ERR_CUDA; }

static bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
static bool al2(const void* p) { return ((uintptr_t)p & 1u) == 0; }
static bool al4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

// ---- op description shared by the entry points ------------------------------------------

static Fmt fmt_of(int kind) {
    switch (kind) {
        case DG_LINEAR_F16: return F_F16;
        case DG_LINEAR_BF16: return F_BF16;
        case DG_LINEAR_W8A8: return F_I8;
        case DG_LINEAR_W4A16: return F_W4A16;
        default: return F_W4A8;
    }
}

static bool quantized_act(int kind) { return kind == DG_LINEAR_W8A8 || kind == DG_LINEAR_W4A8; }

// Validates one op without touching the device.  `quantize_here` is set when
// the op carries fp16 activations that the caller wants quantized first.
dg_status validate(const dg_linear& op, bool allow_quant_input) {
    if (op.kind < DG_LINEAR_F16 || op.kind > DG_LINEAR_W4A8) return DG_ERR_INVALID_ARG;
    if (op.M < 1 || op.N < 1 || op.K < 1) return DG_ERR_INVALID_ARG;
    if (op.M > 16) return DG_ERR_UNSUPPORTED;
    if (!op.W) return DG_ERR_INVALID_ARG;
    const bool head = op.token != nullptr;
    if (head) {
        if (op.M != 1 || !op.logits) return DG_ERR_INVALID_ARG;
        if (op.kind == DG_LINEAR_W8A8) return DG_ERR_UNSUPPORTED;
        if (!al4(op.logits) || !al4(op.token)) return DG_ERR_MISALIGNED;
    } else if (op.kind == DG_LINEAR_W8A8) {
        if (!op.y && !op.acc_out) return DG_ERR_INVALID_ARG;
    } else if (!op.y) {
        return DG_ERR_INVALID_ARG;
    }
    if (op.y && !al2(op.y)) return DG_ERR_MISALIGNED;
    if (op.acc_out && !al4(op.acc_out)) return DG_ERR_MISALIGNED;
    if (!al16(op.W)) return DG_ERR_MISALIGNED;
    switch (op.kind) {
        case DG_LINEAR_F16:
        case DG_LINEAR_BF16:
            if (op.K % 8) return DG_ERR_MISALIGNED;
            break;
        case DG_LINEAR_W8A8:
            if (op.K % 16) return DG_ERR_MISALIGNED;
            if (op.K > 131072) return DG_ERR_UNSUPPORTED;  // int32 accumulator range
            if (!op.w_scale) return DG_ERR_INVALID_ARG;
            if (!al4(op.w_scale)) return DG_ERR_MISALIGNED;
            break;
        default:  // int4
            if (op.K % 32) return DG_ERR_MISALIGNED;
            if (op.group_size < 32 || op.group_size % 32 || op.K % op.group_size)
                return DG_ERR_UNSUPPORTED;
            if (!op.w_scale) return DG_ERR_INVALID_ARG;
            if (!al2(op.w_scale)) return DG_ERR_MISALIGNED;
            break;
    }
    if (op.reserved) return DG_ERR_INVALID_ARG;
    switch (op.epilogue) {
        case DG_EPI_NONE: break;
        case DG_EPI_RESIDUAL:
            if (head || op.acc_out || !op.y || !op.residual) return DG_ERR_INVALID_ARG;
            if (!al2(op.residual)) return DG_ERR_MISALIGNED;
            break;
        case DG_EPI_SWIGLU:
            if (head || op.acc_out || !op.y || !op.W2) return DG_ERR_INVALID_ARG;
            if (op.kind == DG_LINEAR_W8A8) return DG_ERR_UNSUPPORTED;
            if ((op.kind == DG_LINEAR_W4A16 || op.kind == DG_LINEAR_W4A8) && !op.w2_scale)
                return DG_ERR_INVALID_ARG;
            if (!al16(op.W2) || (op.w2_scale && !al2(op.w2_scale))) return DG_ERR_MISALIGNED;
            break;
        default: return DG_ERR_INVALID_ARG;
    }
    if (quantized_act(op.kind)) {
        if (!op.x_i8 || !op.x_scale) return DG_ERR_INVALID_ARG;
        if (!al16(op.x_i8) || !al4(op.x_scale)) return DG_ERR_MISALIGNED;
        if (op.x && !allow_quant_input) return DG_ERR_INVALID_ARG;
        if (op.x && (!al16(op.x) || op.K % 8)) return DG_ERR_MISALIGNED;
    } else {
        if (!op.x) return DG_ERR_INVALID_ARG;
        if (!al16(op.x)) return DG_ERR_MISALIGNED;
    }
    return DG_OK;
}

dg_status check_smem(const dg_linear& op) {
    // fp16 / bf16 at 8+ tokens runs on a tensor-core tile (tcgen05, or its
    // mma.sync fallback), neither of which stages the activations
    if ((op.kind == DG_LINEAR_F16 || op.kind == DG_LINEAR_BF16) && op.M >= 8 && !op.epilogue &&
        op.K % 32 == 0 && tune().MMA != 0)
        return DG_OK;
    const size_t need = gemv_smem(fmt_of(op.kind), pick_mt(op.M), op.K, op.group_size);
    const size_t lim = smem_optin_limit();
    if (lim == 0) return DG_ERR_CUDA;
    return need <= lim ? DG_OK : DG_ERR_UNSUPPORTED;
}

static void fill_common(GemvParams& p, const dg_linear& op) {
    std::memset(&p, 0, sizeof p);
    p.a.K = op.K;
    p.a.M = op.M;
    p.group = op.group_size >= 32 ? op.group_size : 32;
    p.a.x = op.x;
    p.a.xq = op.x_i8;
    p.a.x_scale = op.x_scale;
}

// Whether W8A8 with this many tokens runs on the tensor-core kernel.
static bool use_i8_mma(const dg_linear& op) {
    if (op.kind != DG_LINEAR_W8A8 || op.M < 8 || op.K % 64 || tune().MMA == 0 || op.epilogue)
        return false;
    return gemv_i8_mma_smem(op.K) <= smem_optin_limit();
}

// The tile runs on the fp16 tensor path (exact, see gemv_i8_mma.cu) unless
// DG_TUNE=MMA=1 selects the int8 one.
static dg_status launch_i8_mma(GemvParams& p, cudaStream_t s) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> cache;
    const bool f16 = tune().MMA != 1;
    int dev = 0;
    cudaGetDevice(&dev);
    int occ = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find({dev, p.a.K, (int)f16});
        if (it != cache.end()) occ = it->second;
    }
    if (!occ) {
        if (gemv_i8_mma(nullptr, p.a.K, 0, nullptr, &occ, f16) != cudaSuccess || occ < 1) occ = 1;
        std::lock_guard<std::mutex> g(mu);
        cache[{dev, p.a.K, (int)f16}] = occ;
    }
    // split K over ks warps per 16-row tile (ks | K / 64) until the GPU has
    // about four warps per SM sub-partition to stream with
    const int tiles = (p.t.N + 15) / 16;
    const int nblk = p.a.K / 64;
    int ks = 1;
    while (ks < 8 && nblk % (2 * ks) == 0 && nblk / (2 * ks) >= 4 &&
           tiles * ks < sm_count() * 16)
        ks *= 2;
    p.ksplit = ks;
    const int per_cta = kWarps / ks;
    const int need = (tiles + per_cta - 1) / per_cta;
    int maxg = sm_count() * occ;
    if (maxg < 1) maxg = 1;
    return to_status(gemv_i8_mma(&p, p.a.K, need < maxg ? need : maxg, s, nullptr, f16));
}

// Split-K across CTAs for a launch whose row groups would fill fewer than
// half of the SMs (k or v alone, a few hundred rows): K is cut into S ranges
// of each lane's chunk sequence (at most 8, at least two chunks per lane
// each), CTAs write fp32 / int32 partials to the workspace and a second kernel
// adds them in range order.  S follows the op's shape and the SM count.
static int pick_kparts(const GemvLaunch& L, int N, int K) {
    const int ks = pick_ks(L.fmt, K), slots = kWarps / ks;
    const int n_rg = (N + L.R - 1) / L.R, need = (n_rg + slots - 1) / slots;
    const int kelems = (L.fmt == F_F16 || L.fmt == F_BF16) ? 8 : L.fmt == F_I8 ? 16 : 32;
    // chunks per lane
    const int J = (K / kelems + ks * 32 - 1) / (ks * 32);
    int S = tune().KP;
    if (S <= 0) {
        const int sms = sm_count();
        if (need * 2 > sms) return 1;
        S = sms / need;
        if (S > 8) S = 8;
        if (S > J / 2) S = J / 2;
    }
    if (S > J) S = J;
    return S >= 2 ? S : 1;
}

// Workspace a per-op launch may use for split-K partials: 8 ranges of M x N
// 4-byte sums, for launches small enough to split (device-independent).
static size_t split_ws_bytes(const dg_linear& op) {
    if (op.token || op.epilogue) return 0;
    const size_t outs = (size_t)op.M * (size_t)op.N;
    if (outs > 65536) return 0;
    return (8 * outs * 4 + 255) & ~(size_t)255;
}

// Whether fp16 / bf16 with this many tokens runs on the tensor-core tile.
static bool use_fp_mma(const dg_linear& op) {
    if ((op.kind != DG_LINEAR_F16 && op.kind != DG_LINEAR_BF16) || op.M < 8 || op.K % 32 ||
        tune().MMA == 0 || op.epilogue)
        return false;
    return gemv_fp_mma_smem(op.K) <= smem_optin_limit();
}

// Whether fp16 / bf16 with this many tokens runs on the tcgen05 + TMA tile
// (the mma.sync tile and the CUDA-core tiles remain for epilogues and for
// what the TMA tile cannot address).
static constexpr int kTcMinTokens = 8;

static bool use_tc(const dg_linear& op) {
    const int min_m = tune().TC >= 0 ? tune().TC : kTcMinTokens;
    return (op.kind == DG_LINEAR_F16 || op.kind == DG_LINEAR_BF16) && min_m > 0 &&
           op.M >= min_m && !op.epilogue && op.K % 8 == 0;
}

static dg_status launch_tc(const GemvParams& p, bool bf16, cudaStream_t s, bool* launched) {
    *launched = false;
    if (!gemv_tc_supported(p)) return DG_OK;
    const unsigned spin = tune().SPIN > 0 ? (unsigned)tune().SPIN : 4000000u;
    // L2 prefetch of each CTA's first weight boxes pays off while the previous
    // launch's tail leaves DRAM idle (measured on a 117 MB launch at 16 tokens:
    // 25.2 us without, 24.9 with 6 boxes, 24.5 with 12, 26.1 with 24)
    size_t bytes = 0;
    for (int g = 0; g < p.t.nseg; ++g) bytes += (size_t)p.t.seg[g].rows * p.a.K * 2;
    const int prefetch = tune().TP >= 0 ? tune().TP : bytes <= ((size_t)64 << 20) ? 6 : 12;
    // two 64-k boxes per stage, four stages (measured best of 6x1, 8x1, 12x1, 3x2, 4x2, 6x2)
    const int nb = tune().TK == 1 ? 1 : 2;
    const int stages = tune().TS > 0 ? tune().TS : nb == 2 ? 4 : 6;
    return to_status(gemv_tc(p, bf16, spin, tune().TG, stages, nb, prefetch, s, launched));
}

// Whether int8 / int4 with this many tokens runs on the tcgen05 tile.  By
// default only where it measured faster than the mma.sync / CUDA-core tiles:
// int4 at 8+ tokens with rows longer than 8192 k (44 us against 57-69 us for
// 4096 x 14336 at 8 tokens); DG_TUNE TQ=m sends every int8 / int4 launch of
// m or more tokens to it.
static bool use_tcq(const dg_linear& op) {
    const bool int4 = op.kind == DG_LINEAR_W4A16 || op.kind == DG_LINEAR_W4A8;
    if (op.epilogue || (!int4 && op.kind != DG_LINEAR_W8A8)) return false;
    if (tune().TQ >= 0) return tune().TQ > 0 && op.M >= tune().TQ;
    // int4 rows longer than 8192 k, and W8A8 at 8+ tokens (14336x4096: 23.0 /
    // 23.4 us at 8 / 16 tokens against 23.7 / 24.3 on the mma.sync tile)
    return op.M >= 8 && (int4 ? op.K > 8192 : true);
}

static dg_status launch_tcq(const GemvParams& p, Fmt f, cudaStream_t s, bool* launched) {
    *launched = false;
    if (!gemv_tcq_supported(p, f)) return DG_OK;
    const unsigned spin = tune().SPIN > 0 ? (unsigned)tune().SPIN : 4000000u;
    return to_status(gemv_tcq(p, f, spin, tune().TG, s, launched));
}

// K split of the fp16 / bf16 tile, from K alone (so a row's result does not
// depend on N): the most warps (4, 2, 1) that divide the 32-wide k blocks and
// leave each at least 16 of them.
static int fp_mma_ks(int K) {
    const int nblk = K / 32;
    for (int ks = 4; ks > 1; ks /= 2)
        if (nblk % ks == 0 && nblk / ks >= 16) return ks;
    return 1;
}

static dg_status launch_fp_mma(GemvParams& p, bool bf16, cudaStream_t s) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    int occ = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find({dev, p.a.K, (int)bf16});
        if (it != cache.end()) occ = it->second;
    }
    if (!occ) {
        if (gemv_fp_mma(nullptr, bf16, p.a.K, 0, nullptr, &occ) != cudaSuccess || occ < 1) occ = 1;
        std::lock_guard<std::mutex> g(mu);
        cache[{dev, p.a.K, (int)bf16}] = occ;
    }
    p.ksplit = fp_mma_ks(p.a.K);
    const int tiles = (p.t.N + 15) / 16;
    const int per_cta = kWarps / p.ksplit;
    const int need = (tiles + per_cta - 1) / per_cta;
    int maxg = sm_count() * occ;
    if (maxg < 1) maxg = 1;
    return to_status(gemv_fp_mma(&p, bf16, p.a.K, need < maxg ? need : maxg, s, nullptr));
}

// Whether int4 with this many tokens runs on the tensor-core tile: 8..16
// tokens whose staged activations fit one CTA (K up to about 6900); longer
// rows stay on the CUDA-core tile.
static bool use_w4_mma(const dg_linear& op) {
    if ((op.kind != DG_LINEAR_W4A16 && op.kind != DG_LINEAR_W4A8) || op.M < 8 || op.K % 32 ||
        tune().MMA == 0 || op.epilogue)
        return false;
    return gemv_w4_mma_smem(op.K) <= smem_optin_limit();
}

static dg_status launch_w4_mma(GemvParams& p, bool a8, cudaStream_t s) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    int occ = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find({dev, p.a.K, (int)a8});
        if (it != cache.end()) occ = it->second;
    }
    if (!occ) {
        if (gemv_w4_mma(nullptr, a8, p.a.K, 0, nullptr, &occ) != cudaSuccess || occ < 1) occ = 1;
        std::lock_guard<std::mutex> g(mu);
        cache[{dev, p.a.K, (int)a8}] = occ;
    }
    p.ksplit = fp_mma_ks(p.a.K);  // the same rule on K alone: 32-wide blocks per warp
    const int tiles = (p.t.N + 15) / 16;
    const int per_cta = kW4MmaWarps / p.ksplit;
    const int need = (tiles + per_cta - 1) / per_cta;
    int maxg = sm_count() * occ;
    if (maxg < 1) maxg = 1;
    return to_status(gemv_w4_mma(&p, a8, p.a.K, need < maxg ? need : maxg, s, nullptr));
}

// Launches ops[0..n) (same kind, same activations) as one kernel (two with
// split-K, when ws holds the partials).
static dg_status launch_group(const dg_linear* ops, int n, cudaStream_t s, void* ws = nullptr,
                              size_t ws_bytes = 0) {
    GemvParams p;
    fill_common(p, ops[0]);
    const bool pair = ops[0].epilogue == DG_EPI_SWIGLU;  // (such an op is alone: n == 1)
    int rows = 0;
    for (int i = 0; i < n; ++i) {
        Segment& g = p.t.seg[i];
        g.W = ops[i].W;
        g.scale = ops[i].w_scale;
        g.y = ops[i].y;
        g.acc_out = ops[i].acc_out;
        g.row_begin = rows;
        g.rows = ops[i].N;
        rows += ops[i].N;
    }
    p.t.nseg = n;
    p.t.N = rows;
    if (pair) {  // gate and up rows interleaved: 2N rows, y = silu(gate) * up
        Segment& u = p.t.seg[1];
        u.W = ops[0].W2;
        u.scale = ops[0].w2_scale;
        u.y = nullptr;
        u.acc_out = nullptr;
        u.row_begin = 0;
        u.rows = ops[0].N;
        p.t.nseg = 2;
        p.t.N = 2 * ops[0].N;
        p.t.pair = 1;
    }
    if (ops[0].epilogue == DG_EPI_RESIDUAL) p.t.res = ops[0].residual;
    if (use_tcq(ops[0])) {
        bool launched = false;
        const dg_status st = launch_tcq(p, fmt_of(ops[0].kind), s, &launched);
        if (st != DG_OK || launched) return st;
    }
    if (use_i8_mma(ops[0])) return launch_i8_mma(p, s);
    if (use_tc(ops[0])) {
        bool launched = false;
        const dg_status st = launch_tc(p, ops[0].kind == DG_LINEAR_BF16, s, &launched);
        if (st != DG_OK || launched) return st;
    }
    if (use_fp_mma(ops[0])) return launch_fp_mma(p, ops[0].kind == DG_LINEAR_BF16, s);
    if (use_w4_mma(ops[0])) return launch_w4_mma(p, ops[0].kind == DG_LINEAR_W4A8, s);
    GemvLaunch L{fmt_of(ops[0].kind), pick_mt(ops[0].M), 0, false, ops[0].K, p.group, 0};
    L.R = pick_r(L.fmt, L.MT, L.K);
    if (pair && (L.R & 1)) L.R = 2;  // a row group holds whole pairs
    configure(L, p);
    if (ws && al16(ws) && !ops[0].epilogue) {
        const int S = pick_kparts(L, p.t.N, p.a.K);
        if (S > 1 && ws_bytes >= (size_t)S * p.a.M * p.t.N * 4) {
            p.kparts = S;
            p.kpart = ws;
            p.prefetch_bytes = 0;
            L.grid *= S;  // configure gave one pass (grid = row-group blocks)
        }
    }
    return to_status(family(L, &p, s, nullptr));
}

dg_status launch_head(const dg_linear& op, void* ws, cudaStream_t s) {
    GemvParams p;
    fill_common(p, op);
    p.t.seg[0].W = op.W;
    p.t.seg[0].scale = op.w_scale;
    p.t.seg[0].y = nullptr;
    p.t.seg[0].row_begin = 0;
    p.t.seg[0].rows = op.N;
    p.t.nseg = 1;
    p.t.N = op.N;
    p.logits = op.logits;
    p.part = static_cast<ArgPart*>(ws);
    GemvLaunch L{fmt_of(op.kind), 1, 0, true, op.K, p.group, 0};
    L.R = pick_r(L.fmt, 1, L.K);
    configure(L, p);
    cudaError_t e = family(L, &p, s, nullptr);
    if (e != cudaSuccess) return DG_ERR_CUDA;
    return to_status(launch_argmax_pass2(p.part, L.grid, op.token, s));
}

// CTAs (and so argmax partials) launch_head uses for this op.
int head_grid(const dg_linear& op) {
    GemvParams p;
    fill_common(p, op);
    p.t.nseg = 1;
    p.t.N = op.N;
    GemvLaunch L{fmt_of(op.kind), 1, 0, true, op.K, p.group, 0};
    L.R = pick_r(L.fmt, 1, L.K);
    configure(L, p);
    return L.grid;
}

static size_t head_ws_bytes() { return (size_t)kMaxArgCtas * sizeof(ArgPart); }

// Decode-step workspace: [0, 256) the persistent kernel's barrier words,
// then the argmax partials when the step has an lm_head.
constexpr size_t kStepHeader = 256;
// ---- the persistent decode-step path -----------------------------------------------

static bool same_group(const dg_linear& a, const dg_linear& b) {
    return !b.token && !a.epilogue && !b.epilogue && b.kind == a.kind && b.M == a.M && b.K == a.K && b.x == a.x &&
           b.x_i8 == a.x_i8 && b.x_scale == a.x_scale && b.group_size == a.group_size;
}

// Ops the persistent kernel runs: one token, no int32 accumulator output.
static bool step_eligible(const dg_linear& op) { return op.M == 1 && !op.acc_out; }

// CTAs of the step kernel per SM.
static int step_occupancy(Fmt f, int max_k, size_t smem, int nw, bool epi) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, size_t, int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, (int)f, max_k, smem, nw, (int)epi);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    StepParams* none = nullptr;
    int occ = 0;
    const cudaError_t e = step_launch(f, none, 0, smem, nullptr, &occ, nw, epi);
    if (e != cudaSuccess) occ = 0;
    std::lock_guard<std::mutex> g(mu);
    cache[key] = occ;
    return occ;
}

// Byte ranges an op reads (activations) and writes (outputs); weights and
// scales are read-only for the whole step and never conflict.
struct Range {
    uintptr_t lo, hi;
};
static bool overlaps(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi; }
static void add_range(std::vector<Range>& v, const void* p, size_t bytes) {
    if (p && bytes) v.push_back({(uintptr_t)p, (uintptr_t)p + bytes});
}
static size_t act_elem_bytes(int kind) {
    return (kind == DG_LINEAR_F16 || kind == DG_LINEAR_BF16 || kind == DG_LINEAR_W4A16) ? 2 : 1;
}
static void op_ranges(const dg_linear& op, std::vector<Range>& rd, std::vector<Range>& wr) {
    const size_t M = (size_t)op.M, N = (size_t)op.N, K = (size_t)op.K;
    if (quantized_act(op.kind)) {
        if (op.x) {  // quantized here: reads fp16 x, writes the codes and scale
            add_range(rd, op.x, M * K * 2);
            add_range(wr, op.x_i8, M * K);
            add_range(wr, op.x_scale, M * 4);
        } else {
            add_range(rd, op.x_i8, M * K);
            add_range(rd, op.x_scale, M * 4);
        }
    } else {
        add_range(rd, op.x, M * K * act_elem_bytes(op.kind));
    }
    if (op.epilogue == DG_EPI_RESIDUAL) add_range(rd, op.residual, M * N * 2);
    add_range(wr, op.y, M * N * 2);
    add_range(wr, op.logits, N * 4);
    add_range(wr, op.token, 4);
    add_range(wr, op.acc_out, M * N * 4);
}
static bool any_overlap(const std::vector<Range>& a, const std::vector<Range>& b) {
    for (const Range& x : a)
        for (const Range& y : b)
            if (overlaps(x, y)) return true;
    return false;
}

// Weight and scale bytes of an op.
static void weight_ranges(const dg_linear& op, std::vector<Range>& v) {
    const size_t N = (size_t)op.N, K = (size_t)op.K;
    switch (op.kind) {
        case DG_LINEAR_F16:
        case DG_LINEAR_BF16: add_range(v, op.W, N * K * 2); break;
        case DG_LINEAR_W8A8:
            add_range(v, op.W, N * K);
            add_range(v, op.w_scale, N * 4);
            break;
        default:  // int4
            add_range(v, op.W, N * K / 2);
            if (op.group_size > 0) add_range(v, op.w_scale, N * (K / (size_t)op.group_size) * 2);
            break;
    }
    if (op.epilogue == DG_EPI_SWIGLU) {  // the up projection, same format and shape
        dg_linear up = op;
        up.W = op.W2;
        up.w_scale = op.w2_scale;
        up.epilogue = DG_EPI_NONE;
        weight_ranges(up, v);
    }
}

// True when an op of ops[0..n) writes into the weights or scales of an op of
// the same run.  The persistent kernel reads weights without coherence, so
// such a run goes to the
// per-launch path, which keeps the ops' order.
static bool run_writes_weights(const dg_linear* ops, int n) {
    std::vector<Range> w, out, rd;
    for (int i = 0; i < n; ++i) {
        weight_ranges(ops[i], w);
        op_ranges(ops[i], rd, out);
    }
    return any_overlap(out, w);
}

// int4 step phases whose activations are ready before the launch get a copy
// in the kernel's interleaved layout, written by the launch's prologue into
// the workspace after the barrier words and argmax partials: W4A8 int8 codes
// (given, or quantized in the prologue) plus the chunk sums; W4A16 fp16 pairs.
static size_t int4_layout_bytes(int kind, int K) {
    const size_t nch = (size_t)(K / 32), padded = ((nch + 31) / 32) * 32;
    const size_t bytes = kind == DG_LINEAR_W4A8 ? padded * 32 + nch * 4 : padded * 64;
    return (bytes + 255) & ~(size_t)255;
}
static size_t step_scratch_offset(const dg_linear* ops, int n) {
    for (int i = 0; i < n; ++i)
        if (ops[i].token) return kStepHeader + head_ws_bytes();
    return kStepHeader;
}
static size_t step_scratch_bytes(const dg_linear* ops, int n) {
    size_t b = 0;
    for (int i = 0; i < n; ++i)
        if ((ops[i].kind == DG_LINEAR_W4A8 || ops[i].kind == DG_LINEAR_W4A16) && ops[i].M == 1)
            b += int4_layout_bytes(ops[i].kind, ops[i].K);
    return b;
}

// Runs ops[0..n) (all of one kind, all step-eligible) with the persistent
// kernel, in launches of at most kMaxStepPhases phases.  A phase gets a grid
// barrier when it conflicts with a phase since the previous barrier (RAW, WAR
// or WAW on the activation / output ranges), or follows an lm_head (whose
// token needs every CTA's partial).
static dg_status launch_step_run(const dg_linear* ops, int n, void* ws, cudaStream_t s) {
    static thread_local StepParams sp;
    const Fmt f = fmt_of(ops[0].kind);
    const bool always_sync = tune().STEP == 2;  // barrier between every pair of phases
    int i = 0;
    while (i < n) {
        std::memset(&sp, 0, sizeof sp);
        int max_k = 0;
        std::vector<Range> seen_rd, seen_wr;  // since the last barrier
        std::vector<Range> all_wr;            // the whole launch so far
        std::vector<std::vector<Range>> phase_rd, phase_wr;
        bool after_head = false;
        while (i < n && sp.nphase < kMaxStepPhases) {
            const dg_linear& a = ops[i];
            int j = i + 1;
            if (!a.token)
                while (j < n && j - i < kMaxSeg && same_group(a, ops[j])) ++j;
            std::vector<Range> rd, wr;
            for (int k = i; k < j; ++k) op_ranges(ops[k], rd, wr);
            const bool conflict = any_overlap(seen_wr, rd) || any_overlap(seen_wr, wr) ||
                                  any_overlap(seen_rd, wr);
            if (sp.nphase > 0 && (conflict || after_head || always_sync)) {
                seen_rd.clear();
                seen_wr.clear();
                sp.ph[sp.nphase].flags |= kPhaseBarrier;
            }
            if (any_overlap(all_wr, rd)) sp.ph[sp.nphase].flags |= kPhaseXWritten;
            seen_rd.insert(seen_rd.end(), rd.begin(), rd.end());
            seen_wr.insert(seen_wr.end(), wr.begin(), wr.end());
            all_wr.insert(all_wr.end(), wr.begin(), wr.end());
            after_head = a.token != nullptr;
            StepPhase& ph = sp.ph[sp.nphase++];
            int rows = 0;
            for (int k = i; k < j; ++k) {
                StepSeg& sg = ph.seg[k - i];
                sg.W = ops[k].W;
                sg.scale = ops[k].w_scale;
                sg.y = ops[k].y;
                sg.rows = ops[k].N;
                sg.row_begin = rows;
                rows += ops[k].N;
            }
            ph.nseg = j - i;
            ph.N = rows;
            if (a.epilogue == DG_EPI_SWIGLU) {  // gate and up rows interleaved (j == i + 1)
                StepSeg& u = ph.seg[1];
                u.W = a.W2;
                u.scale = a.w2_scale;
                u.y = nullptr;
                u.rows = a.N;
                u.row_begin = 0;
                ph.nseg = 2;
                ph.N = 2 * a.N;
                ph.pair = 1;
            }
            if (a.epilogue == DG_EPI_RESIDUAL) ph.res = a.residual;
            ph.K = a.K;
            ph.group = a.group_size >= 32 ? a.group_size : 32;
            ph.ks = pick_ks(f, a.K);
            ph.x = a.x;
            ph.xq = a.x_i8;
            ph.x_scale = const_cast<float*>(a.x_scale);
            if (quantized_act(a.kind) && a.x) {
                ph.xq_out = const_cast<int8_t*>(a.x_i8);
                ph.flags |= kPhaseQuantize;  // may become kPhasePreQuant below
            }
            phase_rd.push_back(rd);
            phase_wr.push_back(wr);
            if (a.token) {
                ph.flags |= kPhaseHead;
                ph.logits = a.logits;
                ph.token = a.token;
            }
            if (a.K > max_k) max_k = a.K;
            i = j;
        }
        // Quantize an input once in the launch's prologue instead of in every
        // CTA when nothing else in the launch touches its codes / scale and the
        // launch does not produce the input itself.
        for (int q = 0; q < sp.nphase; ++q) {
            StepPhase& ph = sp.ph[q];
            if (!(ph.flags & kPhaseQuantize) || (ph.flags & kPhaseXWritten)) continue;
            std::vector<Range> out;
            add_range(out, ph.xq_out, (size_t)ph.K);
            add_range(out, ph.x_scale, 4);
            bool private_out = true;
            for (int o = 0; o < sp.nphase && private_out; ++o)
                if (o != q && (any_overlap(out, phase_rd[o]) || any_overlap(out, phase_wr[o])))
                    private_out = false;
            if (private_out) {
                ph.flags = (ph.flags & ~kPhaseQuantize) | kPhasePreQuant;
                sp.prequant = 1;
            }
        }
        // int4: activations ready before the launch are laid out once by the
        // prologue and read from the workspace (no per-phase staging)
        if (f == F_W4A8 || f == F_W4A16) {
            unsigned char* scratch = static_cast<unsigned char*>(ws) + step_scratch_offset(ops, n);
            size_t off = 0;
            for (int q = 0; q < sp.nphase; ++q) {
                StepPhase& ph = sp.ph[q];
                const bool given = !(ph.flags & (kPhaseQuantize | kPhasePreQuant | kPhaseXWritten));
                if (!(ph.flags & kPhasePreQuant) && !given) continue;
                ph.flags |= kPhaseXLaid;
                ph.xlay = scratch + off;
                off += int4_layout_bytes(ops[0].kind, ph.K);
                sp.prequant = 1;
            }
        }
        sp.spin_limit = tune().SPIN > 0 ? (unsigned)tune().SPIN : 20000000u;
        sp.bar = static_cast<unsigned*>(ws);
        sp.part = reinterpret_cast<ArgPart*>(static_cast<unsigned char*>(ws) + kStepHeader);
        sp.err = device_error_word();
        if (!sp.err) return DG_ERR_CUDA;
        const size_t smem = step_smem(f, max_k);
        if (smem > smem_optin_limit()) return DG_ERR_UNSUPPORTED;
        // k_step runs 16 warps; W4A8 20 (one more row group in flight per SM
        // sub-partition: 883 -> 863 us for the 32-layer step) when no phase
        // splits K, since the split barriers' id ranges are disjoint only up
        // to 16 warps
        bool split = false, pairs = false, epi = false;
        for (int q = 0; q < sp.nphase; ++q) {
            split = split || sp.ph[q].ks > 1;
            pairs = pairs || sp.ph[q].pair;
            epi = epi || sp.ph[q].pair || sp.ph[q].res;
        }
        // (SwiGLU pair phases need an even number of rows per slot: the
        // formats' defaults give that; a tuned warp count might not)
        const int nw = split ? 16
                             : (tune().SNW > 0 && !pairs) ? tune().SNW
                                                          : f == F_W4A8 ? 20 : 16;
        const int occ = step_occupancy(f, max_k, smem, nw, epi);
        if (occ < 1) return DG_ERR_UNSUPPORTED;
        const int grid = sm_count() * occ;
        if (grid > kMaxArgCtas) return DG_ERR_UNSUPPORTED;
        if (cudaMemsetAsync(ws, 0, 2 * sizeof(unsigned), s) != cudaSuccess) return DG_ERR_CUDA;
        const cudaError_t e = step_launch(f, &sp, grid, smem, s, nullptr, nw, epi);
        if (e != cudaSuccess) return DG_ERR_CUDA;
    }
    return DG_OK;
}

}  // namespace dg

using namespace dg;

extern "C" {

const char* dg_status_string(dg_status s) {
    switch (s) {
        case DG_OK: return "DG_OK";
        case DG_ERR_INVALID_ARG: return "DG_ERR_INVALID_ARG";
        case DG_ERR_UNSUPPORTED: return "DG_ERR_UNSUPPORTED";
        case DG_ERR_MISALIGNED: return "DG_ERR_MISALIGNED";
        case DG_ERR_WORKSPACE: return "DG_ERR_WORKSPACE";
        case DG_ERR_CUDA: return "DG_ERR_CUDA";
        case DG_ERR_TIMEOUT: return "DG_ERR_TIMEOUT";
    }
    return "DG_ERR_UNKNOWN";
}

const char* dg_version(void) { return "dg 0.1 (sm_103a)"; }

size_t dg_workspace_bytes(const dg_linear* ops, int n_ops) {
    if (!ops || n_ops <= 0) return 0;
    size_t need = step_scratch_offset(ops, n_ops) + step_scratch_bytes(ops, n_ops);
    for (int i = 0; i < n_ops; ++i) need = std::max(need, split_ws_bytes(ops[i]));
    return need;
}

dg_status dg_gemv_f16(const void* W, const void* x, void* y, dg_ftype t, int M, int N, int K,
                      void* ws, size_t ws_bytes, dg_stream stream) {
    if (t != DG_F16 && t != DG_BF16) return DG_ERR_INVALID_ARG;
    dg_linear op;
    std::memset(&op, 0, sizeof op);
    op.kind = t == DG_F16 ? DG_LINEAR_F16 : DG_LINEAR_BF16;
    op.M = M;
    op.N = N;
    op.K = K;
    op.W = W;
    op.x = x;
    op.y = y;
    dg_status st = validate(op, false);
    if (st != DG_OK) return st;
    if ((st = check_smem(op)) != DG_OK) return st;
    return launch_group(&op, 1, stream, ws, ws_bytes);
}

dg_status dg_gemv_w8a8(const int8_t* W, const float* w_scale, const int8_t* x, const float* x_scale,
                       void* y, int32_t* acc_out, int M, int N, int K, void* ws, size_t ws_bytes,
                       dg_stream stream) {
    dg_linear op;
    std::memset(&op, 0, sizeof op);
    op.kind = DG_LINEAR_W8A8;
    op.M = M;
    op.N = N;
    op.K = K;
    op.W = W;
    op.w_scale = w_scale;
    op.x_i8 = x;
    op.x_scale = x_scale;
    op.y = y;
    op.acc_out = acc_out;
    dg_status st = validate(op, false);
    if (st != DG_OK) return st;
    if ((st = check_smem(op)) != DG_OK) return st;
    return launch_group(&op, 1, stream, ws, ws_bytes);
}

dg_status dg_gemv_w4(const uint8_t* Wq, const void* scales, int group_size, const void* x_f16,
                     const int8_t* x_i8, const float* x_scale, void* y, int M, int N, int K,
                     void* ws, size_t ws_bytes, dg_stream stream) {
    dg_linear op;
    std::memset(&op, 0, sizeof op);
    op.kind = x_i8 ? DG_LINEAR_W4A8 : DG_LINEAR_W4A16;
    op.M = M;
    op.N = N;
    op.K = K;
    op.group_size = group_size;
    op.W = Wq;
    op.w_scale = scales;
    op.x = x_i8 ? nullptr : x_f16;
    op.x_i8 = x_i8;
    op.x_scale = x_scale;
    op.y = y;
    dg_status st = validate(op, false);
    if (st != DG_OK) return st;
    if ((st = check_smem(op)) != DG_OK) return st;
    return launch_group(&op, 1, stream, ws, ws_bytes);
}

dg_status dg_linear_forward(const dg_linear* op, void* ws, size_t ws_bytes, dg_stream stream) {
    if (!op || op->token) return DG_ERR_INVALID_ARG;
    dg_status st = validate(*op, false);
    if (st != DG_OK) return st;
    if ((st = check_smem(*op)) != DG_OK) return st;
    return launch_group(op, 1, stream, ws, ws_bytes);
}

dg_status dg_quantize_act_i8(const void* x, int8_t* xq, float* x_scale, int M, int K,
                             dg_stream stream) {
    if (!x || !xq || !x_scale || M < 1 || K < 1) return DG_ERR_INVALID_ARG;
    if (K % 8 || !al16(x) || !al16(xq) || !al4(x_scale)) return DG_ERR_MISALIGNED;
    return to_status(launch_quant_act(static_cast<const __half*>(x), xq, x_scale, M, K, stream));
}

dg_status dg_lm_head_argmax(const dg_linear* head, void* ws, size_t ws_bytes, dg_stream stream) {
    if (!head || !head->token) return DG_ERR_INVALID_ARG;
    dg_status st = validate(*head, false);
    if (st != DG_OK) return st;
    if (!ws) return DG_ERR_WORKSPACE;
    if (ws_bytes < dg_workspace_bytes(head, 1)) return DG_ERR_WORKSPACE;
    if (!al16(ws)) return DG_ERR_MISALIGNED;
    if ((st = check_smem(*head)) != DG_OK) return st;
    return launch_head(*head, ws, stream);
}

dg_status dg_decode_step_weights(const dg_linear* ops, int n_ops, void* ws, size_t ws_bytes,
                                 dg_stream stream) {
    if (!ops || n_ops < 1) return DG_ERR_INVALID_ARG;
    for (int i = 0; i < n_ops; ++i) {
        dg_status st = validate(ops[i], true);
        if (st != DG_OK) return st;
    }
    const size_t need = dg_workspace_bytes(ops, n_ops);
    if (!ws || ws_bytes < need) return DG_ERR_WORKSPACE;
    if (!al16(ws)) return DG_ERR_MISALIGNED;
    for (int i = 0; i < n_ops; ++i) {
        dg_status st = check_smem(ops[i]);
        if (st != DG_OK) return st;
    }
    const bool persistent = tune().STEP != 0;
    int i = 0;
    while (i < n_ops) {
        // a maximal run of step-eligible ops of one kind goes to the persistent kernel
        int j = i;
        while (persistent && j < n_ops && ops[j].kind == ops[i].kind && step_eligible(ops[j])) ++j;
        if (j > i && !run_writes_weights(ops + i, j - i)) {
            dg_status st = launch_step_run(ops + i, j - i, ws, stream);
            if (st != DG_OK) return st;
            i = j;
            continue;
        }
        // otherwise one launch per fused group
        const dg_linear& a = ops[i];
        j = i + 1;
        if (!a.token)
            while (j < n_ops && j - i < kMaxSeg && same_group(a, ops[j])) ++j;
        if (quantized_act(a.kind) && a.x) {
            cudaError_t e = launch_quant_act(static_cast<const __half*>(a.x),
                                             const_cast<int8_t*>(a.x_i8),
                                             const_cast<float*>(a.x_scale), a.M, a.K, stream);
            if (e != cudaSuccess) return DG_ERR_CUDA;
        }
        void* parts = static_cast<unsigned char*>(ws) + kStepHeader;
        dg_status st = a.token ? launch_head(a, parts, stream) : launch_group(ops + i, j - i, stream);
        if (st != DG_OK) return st;
        i = j;
    }
    return DG_OK;
}

dg_status dg_check_device_status(dg_stream stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return DG_ERR_CUDA;
    if (cudaPeekAtLastError() != cudaSuccess) return DG_ERR_CUDA;
    int* w = device_error_word();
    if (!w) return DG_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return DG_ERR_CUDA;
    if (v == 0) return DG_OK;
    const int zero = 0;
    if (cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return DG_ERR_CUDA;
    return DG_ERR_TIMEOUT;
}

dg_status dg_selftest_wait_timeout(unsigned spin_limit, dg_stream stream) {
    if (spin_limit == 0 || spin_limit > 10000000u) return DG_ERR_INVALID_ARG;
    int* w = device_error_word();
    if (!w) return DG_ERR_CUDA;
    return to_status(launch_wait_selftest(spin_limit, w, stream));
}

static bool ranges_overlap(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + bn && y < x + an;
}

dg_status dg_swiglu(const void* g, const void* u, void* h, int n, dg_stream stream) {
    if (!g || !u || !h || n < 1) return DG_ERR_INVALID_ARG;
    if (n % 8 || !al16(g) || !al16(u) || !al16(h)) return DG_ERR_MISALIGNED;
    return to_status(launch_swiglu(g, u, h, n, stream));
}

dg_status dg_residual_add(const void* a, const void* b, void* out, int n, dg_stream stream) {
    if (!a || !b || !out || n < 1) return DG_ERR_INVALID_ARG;
    if (n % 8 || !al16(a) || !al16(b) || !al16(out)) return DG_ERR_MISALIGNED;
    return to_status(launch_residual_add(a, b, out, n, stream));
}

dg_status dg_causal_conv1d_update(const void* x, void* state, const void* w, const void* bias,
                                  void* y, int M, int C, int width, int act, dg_stream stream) {
    if (!x || !state || !w || !y || M < 1 || C < 1) return DG_ERR_INVALID_ARG;
    if (act != DG_ACT_NONE && act != DG_ACT_SILU) return DG_ERR_INVALID_ARG;
    if (width < 2 || width > 8) return DG_ERR_UNSUPPORTED;
    if (C % 8 || !al16(x) || !al16(state) || !al16(w) || !al16(y) || (bias && !al16(bias)))
        return DG_ERR_MISALIGNED;
    const size_t sb = (size_t)M * C * (width - 1) * 2;
    if (ranges_overlap(y, (size_t)M * C * 2, state, sb)) return DG_ERR_INVALID_ARG;
    return to_status(launch_conv1d_update(x, state, w, bias, y, M, C, width, act, stream));
}

dg_status dg_quantize_weights_i8(const void* W, int8_t* Wq, float* w_scale, int N, int K,
                                 dg_stream stream) {
    if (!W || !Wq || !w_scale || N < 1 || K < 1) return DG_ERR_INVALID_ARG;
    if (K % 16 || !al16(W) || !al16(Wq) || !al4(w_scale)) return DG_ERR_MISALIGNED;
    return to_status(launch_quant_w8(W, Wq, w_scale, N, K, stream));
}

dg_status dg_quantize_weights_w4(const void* W, uint8_t* Wq, void* scales, int N, int K,
                                 int group_size, dg_stream stream) {
    if (!W || !Wq || !scales || N < 1 || K < 1) return DG_ERR_INVALID_ARG;
    if (group_size < 32 || group_size % 32 || K % group_size) return DG_ERR_UNSUPPORTED;
    if (!al16(W) || !al16(Wq) || !al2(scales)) return DG_ERR_MISALIGNED;
    return to_status(launch_quant_w4(W, Wq, scales, N, K, group_size, stream));
}

dg_status dg_probe_copy(const void* src, void* dst, size_t bytes, dg_stream stream) {
    if (!src || !dst || bytes == 0) return DG_ERR_INVALID_ARG;
    if (bytes % 16 || !al16(src) || !al16(dst)) return DG_ERR_MISALIGNED;
    return to_status(launch_probe_copy(src, dst, bytes, stream));
}

dg_status dg_probe_read(const void* src, size_t bytes, uint32_t* sink, dg_stream stream) {
    if (!src || !sink || bytes == 0) return DG_ERR_INVALID_ARG;
    if (bytes % 16 || !al16(src) || !al4(sink)) return DG_ERR_MISALIGNED;
    return to_status(launch_probe_read(src, bytes, sink, stream));
}

}  // extern "C"
