// Internal definitions shared by the sm_103a kernels of libdg.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/dg.h"

namespace dg {

constexpr int kThreads = 256;          // one CTA = 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSeg = 4;             // matrices fused into one launch (q|k|v, gate|up)
constexpr int kMaxArgCtas = 4096;      // cap on lm_head CTAs (bounds the partials buffer)

// Element formats of the weight stream.
enum Fmt : int { F_F16 = 0, F_BF16 = 1, F_I8 = 2, F_W4A16 = 3, F_W4A8 = 4 };

// One matrix of a fused launch.  Global row r of the launch belongs to the
// segment with row_begin <= r < row_begin + rows.
struct Segment {
    const void* W;       // row 0 of this matrix
    const void* scale;   // W8A8: float [rows]; int4: half [rows][K/group]
    void* y;             // [M][rows] (fp16 / bf16); may be null for an lm_head
    int32_t* acc_out;    // W8A8 only, optional [M][rows]
    int32_t row_begin;
    int32_t rows;
};

// The matrices of one fused launch (same activations, K and format).
// Epilogues: `res` adds a residual [M][rows] to the op's result (a launch with
// a residual holds that one op); `pair` marks a SwiGLU op, whose two segments
// (gate, up) are walked row by row in pairs: global row 2i is gate row i,
// 2i + 1 up row i, and y[i] = silu(gate) * up lands in segment 0's y.
struct SegTable {
    Segment seg[kMaxSeg];
    int nseg;
    int N;               // rows over all segments
    int pair;
    const void* res;
};

// Activations of a launch or phase.
struct ActIn {
    const void* x;          // fp16 / bf16 [M][K]
    const int8_t* xq;       // int8 [M][K] (global or shared memory)
    const float* x_scale;   // [M] or null
    int K, M;
};

// (value, index) partial of the greedy argmax.
struct ArgPart {
    float v;
    int32_t i;
};

struct GemvParams {
    SegTable t;
    ActIn a;
    int group;               // int4 group size (multiple of 32)
    int ksplit;              // warps sharing one row group (splits K), 1/2/4/8
    int iters;               // row-group loop trip count, uniform over the grid
    int prefetch_bytes;      // per-CTA L2 prefetch issued before the dependency wait
    float* logits;           // lm_head: fp32 [N]
    ArgPart* part;           // lm_head: one partial per CTA
    int kparts;              // split-K across CTAs: K ranges (1 = none)
    void* kpart;             //   partial sums [kparts][M][N] (fp32 or int32 bits)
};

// ---- the persistent decode-step kernel's work list --------------------------------

constexpr int kMaxStepPhases = 144;   // phases per launch (kernel parameter space)

enum StepFlags : int {
    kPhaseHead = 1,       // lm_head: logits + greedy token
    kPhaseQuantize = 2,   // quantize the fp16 activations inside the phase
    kPhaseBarrier = 4,    // grid barrier before the phase
    kPhaseXWritten = 8,   // activations written earlier in this launch
    kPhasePreQuant = 16,  // activations quantized in the launch's prologue
    kPhaseXLaid = 64      // the prologue wrote x in the format's layout at xlay: the
                          // MACs read it from global memory (no staging, no meeting)
};

struct StepSeg {
    const void* W;
    const void* scale;
    void* y;
    int32_t rows;
    int32_t row_begin;
};

// One phase = one fused group of ops.  Phases run in order; a phase flagged
// kPhaseBarrier starts only after every CTA finished every earlier phase (it
// reads or overwrites memory an earlier phase wrote or read); other phases
// only follow their own CTA's earlier work.
struct StepPhase {
    StepSeg seg[kMaxSeg];
    const void* x;        // fp16 / bf16 activations (or the fp16 source to quantize)
    const int8_t* xq;     // given int8 codes
    float* x_scale;       // given per-token scale, or where the quantization writes it
    int8_t* xq_out;       // where the quantization writes its codes (may be null)
    float* logits;        // lm_head
    int32_t* token;       // lm_head
    unsigned char* xlay;  // kPhaseXLaid: the activations in the format's layout (workspace)
    const void* res;      // residual [1][N] added before rounding (a one-op phase)
    int32_t K, N, nseg, flags, ks;
    int32_t group;        // int4 scale group along K (the ops of a phase share it)
    int32_t pair;         // SwiGLU: segments 0 (gate) and 1 (up) interleaved by row
};

struct StepParams {
    StepPhase ph[kMaxStepPhases];
    int nphase;
    int prequant;         // the launch's prologue runs (kPhasePreQuant / kPhaseXLaid phases)
    unsigned spin_limit;  // bound on every barrier wait
    unsigned* bar;        // 2 zeroed words: arrivals, generation
    ArgPart* part;        // one partial per CTA (lm_head phases)
    int* err;             // device error word
};

// StepParams travels as a kernel parameter (at most 32,764 bytes).
static_assert(sizeof(StepParams) <= 32764, "step parameters exceed the kernel parameter space");

constexpr int kErrTimeout = 1;

// ---- PTX helpers ------------------------------------------------------------

// Streaming 16-byte load of weights: read-only path, not kept in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Hint L2 to fetch the 128-byte line holding p.
__device__ __forceinline__ void prefetch_line_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Activation loads: through the read-only path (L1-cached), or L2 only for
// data written earlier in the same kernel (L1 is not kept coherent).
__device__ __forceinline__ uint4 ld_nc16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_cg16(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const void* p) {
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Hint L2 to fetch [p, p + bytes); bytes a multiple of 16, p 16-byte aligned.
// A prefetch never changes what a later load returns (L2 is the point of
// coherence), so it is safe before the dependency wait.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch: let the next kernel on the stream be
// scheduled, and wait until the previous one completed (memory visible).
// Both are no-ops when the launch carried no programmatic dependency.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// acc + a * b with a, b fp16 (or bf16) and acc fp32: the product is exact in
// fp32 and one rounding happens, as in converting both and using fmaf.
__device__ __forceinline__ float fma_f16(uint16_t a, uint16_t b, float acc) {
    asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(b));
    return acc;
}
__device__ __forceinline__ float fma_bf16(uint16_t a, uint16_t b, float acc) {
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(b));
    return acc;
}

__device__ __forceinline__ uint16_t lo16(uint32_t v) { return (uint16_t)(v & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t v) { return (uint16_t)(v >> 16); }

// Two fp32 FMAs in one instruction: acc.{x,y} += a.{x,y} * b.{x,y}, each
// rounded once.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 acc) {
    unsigned long long ra, rb, rc;
    memcpy(&ra, &a, 8);
    memcpy(&rb, &b, 8);
    memcpy(&rc, &acc, 8);
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(rc) : "l"(ra), "l"(rb));
    float2 r;
    memcpy(&r, &rc, 8);
    return r;
}

// Dot products of four byte lanes.
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// d = (a & b) ^ c in one LOP3.
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) {
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) {
    return *reinterpret_cast<__half2*>(&u);
}

// silu(v) = v / (1 + e^-v) in fp32: the library exp and IEEE operations (a
// few fp32 roundings).  For v below about -88, e^-v overflows to infinity and
// the result is -0, next to the true value (whose magnitude is below 1e-36).
__device__ __forceinline__ float silu_f32(float v) { return v / (1.f + expf(-v)); }

// Total order of the greedy argmax: larger value first, then lower index; a
// NaN value is never better.
__device__ __forceinline__ bool arg_better(float v, int i, float bv, int bi) {
    if (v != v) return false;
    if (bv != bv) return true;
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Spins while *flag == old, at most `limit` polls (~100 ns apart).  On giving
// up it records kErrTimeout in *err and returns false; it never waits longer.
__device__ __forceinline__ bool bounded_wait_change(const unsigned* flag, unsigned old,
                                                    unsigned limit, int* err) {
    for (unsigned n = 0; ld_acquire_gpu(flag) == old; ++n) {
        if (n >= limit) {
            atomicExch(err, kErrTimeout);
            return false;
        }
        __nanosleep(100);
    }
    return true;
}

// ---- host-side launch helpers (defined in api.cu) ---------------------------

int sm_count();                      // SMs of the current device (cached per device)
int* device_error_word();            // the library's device error word (current device)
size_t smem_optin_limit();           // max dynamic shared memory per CTA
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       void** args);

// Which kernel instantiation a launch uses, and its grid.
struct GemvLaunch {
    Fmt fmt;
    int MT;        // token tile: 1, 2, 4, 8 or 16 (>= M)
    int R;         // rows per slot: 1, 2 or 4
    bool argmax;   // lm_head epilogue (MT == 1)
    int K, group;
    int grid;
};

// Kernel families, one translation unit each.  With occ != nullptr they
// report CTAs per SM instead of launching.
cudaError_t gemv_fp(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ);
cudaError_t gemv_i8(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ);
cudaError_t gemv_w4a16(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ);
cudaError_t gemv_w4a8(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ);
size_t gemv_smem(Fmt f, int MT, int K, int group);
// W8A8 for 8..16 tokens on the tensor cores (mma.sync s8, exact int32).
cudaError_t gemv_i8_mma(const GemvParams* p, int K, int grid, cudaStream_t s, int* occ, bool f16);
size_t gemv_i8_mma_smem(int K);
// Groupwise int4 for 8..16 tokens on the tensor cores (gemv_w4_mma.cu), CTAs
// of kW4MmaWarps warps.
constexpr int kW4MmaWarps = 16;
cudaError_t gemv_w4_mma(const GemvParams* p, bool a8, int K, int grid, cudaStream_t s, int* occ);
size_t gemv_w4_mma_smem(int K);
// fp16 / bf16 for 8..16 tokens on the tensor cores (gemv_fp_mma.cu).
cudaError_t gemv_fp_mma(const GemvParams* p, bool bf16, int K, int grid, cudaStream_t s, int* occ);
size_t gemv_fp_mma_smem(int K);
// fp16 / bf16, 1..16 tokens, on tcgen05 with TMA-fed operands (stream-K over
// all SMs).  gemv_tc leaves *launched false (and returns cudaSuccess) when it
// cannot take the launch: no tensor-map encoder, or no fixup scratch for this
// stream yet while the stream is being captured.
bool gemv_tc_supported(const GemvParams& p);
cudaError_t gemv_tc(const GemvParams& p, bool bf16, unsigned spin, int grid, int stages, int nb,
                    int prefetch, cudaStream_t s, bool* launched);
size_t gemv_tc_smem();
// int8 / int4 weights (W8A8, W4A16, W4A8), 1..16 tokens, on tcgen05: codes
// widened to fp16 into TMEM, group scales applied per accumulator run
// (gemv_tcq.cu).  Same launch contract as gemv_tc.
bool gemv_tcq_supported(const GemvParams& p, Fmt f);
cudaError_t gemv_tcq(const GemvParams& p, Fmt f, unsigned spin, int grid, cudaStream_t s,
                     bool* launched);

// Host helpers of api.cu shared with the static-scratch lm_head entry point.
dg_status validate(const dg_linear& op, bool allow_quant_input);
dg_status check_smem(const dg_linear& op);
dg_status launch_head(const dg_linear& op, void* parts, cudaStream_t s);
int head_grid(const dg_linear& op);

// Persistent decode-step kernel (step_kernel.cu): one cooperative launch over
// sp.nphase phases of format f, with nw warps per CTA (16, or 0 for the
// format's default); epi: some phase carries an epilogue (residual, SwiGLU).
// occ != nullptr: report CTAs per SM instead.
cudaError_t step_launch(Fmt f, const StepParams* sp, int grid, size_t smem, cudaStream_t s,
                        int* occ, int nw, bool epi);
size_t step_smem(Fmt f, int max_k);
cudaError_t launch_wait_selftest(unsigned limit, int* err, cudaStream_t s);

cudaError_t launch_argmax_pass2(const ArgPart* part, int nparts, int32_t* token, cudaStream_t s);
cudaError_t launch_quant_act(const __half* x, int8_t* xq, float* s, int M, int K,
                             cudaStream_t st);
cudaError_t launch_probe_copy(const void* src, void* dst, size_t bytes, cudaStream_t s);
// aux_kernels.cu
cudaError_t launch_swiglu(const void* g, const void* u, void* h, int n, cudaStream_t s);
cudaError_t launch_residual_add(const void* a, const void* b, void* out, int n, cudaStream_t s);
cudaError_t launch_conv1d_update(const void* x, void* state, const void* w, const void* bias,
                                 void* y, int M, int C, int width, int silu, cudaStream_t s);
cudaError_t launch_quant_w8(const void* W, int8_t* Wq, float* s, int N, int K, cudaStream_t st);
cudaError_t launch_quant_w4(const void* W, uint8_t* Wq, void* scales, int N, int K, int G,
                            cudaStream_t st);
cudaError_t launch_probe_read(const void* src, size_t bytes, uint32_t* sink, cudaStream_t s);

}  // namespace dg
