/*
 * dg.h -- C ABI of the GB300 (sm_103a) decode-step skinny GEMV library (libdg.so).
 *
 * What it computes: the weight-streaming matrix-vector product of single-request
 * LLM decoding, y = x * W^T with x holding M = 1 token (or a few draft/verify
 * tokens), in three forms:
 *   - FP16 / BF16 weights                 (dg_gemv_f16)
 *   - a very wide lm_head + greedy argmax (dg_lm_head_argmax)
 *   - weight-quantized: W8A8 per-channel int8 (dg_gemv_w8a8) and groupwise
 *     int4 with fp16 or int8 activations (dg_gemv_w4), dequantized in registers.
 * Sources: the M=1 custom cube matmul, the 16-slice lm_head with a host reduce
 * and the weight-bandwidth floor of "MiniCPM-V on Orange Pi AIPro (Ascend 310B)";
 * single-request decode and graph-replayed decode steps of "EdgeFM: Efficient
 * Edge Inference for Vision-Language Models" (sections 2.B and 2.C); W8A8 and
 * W4A8 of "vLLM Arm CPU optimizations" (sections "INT8 W8A8", "INT8 W4A8").
 * The pages give no formulas: the definitions below are the plain readings.
 *
 * Conventions (every entry point):
 *  - Layout.  W is [N][K] row-major (output features x input features, K
 *    contiguous).  x is [M][K] and y is [M][N], row-major.
 *    y[m][n] = sum_k W[n][k] * x[m][k].
 *  - Pointers.  All tensor pointers are DEVICE pointers owned by the caller.
 *    The library allocates and frees nothing; scratch comes from the caller's
 *    workspace (ws, ws_bytes), sized by dg_workspace_bytes.
 *  - Streams.  Work is enqueued on `stream` (NULL = legacy default stream);
 *    calls never synchronize and can be captured into a CUDA graph.  Kernels
 *    are launched with programmatic dependent launch: a kernel may prefetch its
 *    weights into L2 while the previous kernel on the stream finishes, and
 *    touches activations, outputs and workspace only after it completed.
 *  - Errors.  Arguments are validated on the host before anything is launched;
 *    on failure nothing is enqueued and a dg_status other than DG_OK returns.
 *    A failed launch returns DG_ERR_CUDA.  No C++ exception crosses the ABI.
 *  - Determinism.  Each output is summed in a fixed order that depends only on
 *    K and the element format (never on N, M, the row offset or the launch
 *    grid), so repeated calls are bitwise identical and a row slice of W gives
 *    bitwise the same rows as the whole matrix.  One exception, opt-in: a
 *    per-op call (dg_gemv_*) with few rows (its row groups would fill fewer
 *    than half the SMs) that is given workspace splits K across CTAs (split-K:
 *    S fixed K ranges, partial sums in ws, a second kernel adding them in range
 *    order); its order then also depends on N, M and the SM count, and is still
 *    the same on every call.  Integer (W8A8) sums are exact either way.  The
 *    second exception: fp16 / bf16 calls with 8 <= M <= 16 and no epilogue run
 *    on the tcgen05 tensor cores with the work split stream-K over all SMs (the
 *    launch's 128-row x 64-k weight blocks cut into one equal range per SM; a
 *    row tile cut between CTAs is summed in fp32 piece by piece in CTA order),
 *    so their order depends on K, on the rows of the whole launch and on the
 *    SM count, and is still the same on every call.  The same holds for int4
 *    calls on the int8 / int4 tcgen05 tile (by default 8+ tokens with K >
 *    8192; one fp32 accumulator per group, scaled as in the scalar
 *    definition); W8A8 calls with 8+ tokens also run there by default and
 *    keep exact int32 sums.  Such a call keeps a small
 *    fixup scratch per (device, stream) (about 4.3 MB, allocated on the
 *    stream's first such call); a stream first used inside graph capture runs
 *    the mma.sync tile instead (K split by a rule on K alone).
 *  - Alignment.  W, x, xq and y must be 16-byte aligned; K must be a multiple
 *    of 8 (fp16/bf16), 16 (int8) or 32 (int4).
 *  - Tuning.  The environment variable DG_TUNE (comma-separated KEY=value,
 *    read once per process) overrides launch choices for configuration
 *    sweeps; unset, the defaults above hold.  Every setting stays within the
 *    parity bound; KS (warps per row), KP (split-K ranges), MMA (tensor-core
 *    tiles off / int8 tile), TC (fewest tokens on the fp16 / bf16 tcgen05
 *    tile, 0 = off), TQ (fewest tokens on the int8 / int4 tcgen05 tile, 0 =
 *    off; by default W8A8 with 8+ tokens and int4 with 8+ tokens and K > 8192
 *    go there) and TG
 *    (the tcgen05 tiles' CTA count) change a row's summation order, the others
 *    (TK: 64-k boxes per stage of the fp16 tile, 1 or 2; TS: its ring stages,
 *    6 / 8 / 12 with one box, 3 / 4 / 6 with two; TP: stages it prefetches to
 *    L2 before the dependency wait) only the schedule.
 */
#ifndef DG_H_
#define DG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* dg_stream; /* same type as cudaStream_t */

typedef enum {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad enum */
    DG_ERR_UNSUPPORTED = 2, /* shape or option outside what the kernels handle */
    DG_ERR_MISALIGNED = 3,  /* a pointer or K breaks the alignment rules */
    DG_ERR_WORKSPACE = 4,   /* ws smaller than dg_workspace_bytes asks for */
    DG_ERR_CUDA = 5,        /* a CUDA call or launch failed */
    DG_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up */
} dg_status;

typedef enum { DG_F16 = 0, DG_BF16 = 1 } dg_ftype;

/* Kind of one linear op in a decode step (dg_linear.kind). */
typedef enum {
    DG_LINEAR_F16 = 0,   /* W fp16 [N][K], x fp16 [M][K], y fp16 */
    DG_LINEAR_BF16 = 1,  /* W bf16, x bf16, y bf16 */
    DG_LINEAR_W8A8 = 2,  /* W int8 [N][K] + float w_scale[N]; x_i8 + x_scale; y fp16 */
    DG_LINEAR_W4A16 = 3, /* W packed int4 [N][K/2] + half w_scale[N][K/group]; x fp16; y fp16 */
    DG_LINEAR_W4A8 = 4   /* as W4A16 but x_i8 + x_scale; y fp16 */
} dg_kind;

/* Epilogue applied to an op's fp32 result before it is rounded to y
 * (dg_linear.epilogue); the pages motivate only removing the launches around
 * the weight stream (EdgeFM, section 2.C, graph-accelerated decode), so these
 * are the plain decoder definitions:
 *   DG_EPI_RESIDUAL: y = x * W^T + residual     (residual [M][N], y's type)
 *   DG_EPI_SWIGLU:   y = silu(x * W^T) * (x * W2^T),  silu(v) = v / (1 + e^-v)
 *                    (W the gate projection, W2 the up projection: same kind,
 *                    shape and group; w2_scale their scales for int4 kinds).
 * Both are evaluated in fp32 on the sums and rounded once into y; y may be
 * the residual itself (an in-place add: each element is read, then written,
 * by the same thread).  Not for
 * lm_heads (token != NULL), nor with acc_out; SwiGLU is not offered for
 * DG_LINEAR_W8A8 (DG_ERR_UNSUPPORTED). */
typedef enum { DG_EPI_NONE = 0, DG_EPI_RESIDUAL = 1, DG_EPI_SWIGLU = 2 } dg_epilogue;

/* One linear op: y = x * W^T in the format `kind`.
 * For the quantized-activation kinds (W8A8, W4A8), x_i8 [M][K] and x_scale[M]
 * are read; if `x` (fp16 [M][K]) is also given, dg_decode_step_weights first
 * quantizes x into x_i8 / x_scale (see dg_quantize_act_i8).
 * An op with token != NULL is an lm_head: M must be 1, logits (fp32 [N]) and
 * the greedy token are written and y may be NULL. */
typedef struct {
    int32_t kind;
    int32_t M, N, K;
    int32_t group_size;    /* int4 kinds: multiple of 32 dividing K (32 in the workloads) */
    const void* W;
    const void* w_scale;
    const void* x;
    const int8_t* x_i8;
    const float* x_scale;
    void* y;
    float* logits;
    int32_t* token;
    int32_t* acc_out;      /* W8A8 only, optional: exact int32 accumulators [M][N] */
    int32_t epilogue;      /* dg_epilogue (0 = none) */
    int32_t reserved;      /* must be 0 */
    const void* residual;  /* DG_EPI_RESIDUAL */
    const void* W2;        /* DG_EPI_SWIGLU: up-projection weights */
    const void* w2_scale;  /* DG_EPI_SWIGLU: their scales (int4 kinds) */
} dg_linear;

/* FP16 / BF16 weights (paragraph on the custom M=1 cube matmul of the Orange
 * Pi AIPro post; the vector-matrix product at M=1).
 * W [N][K], x [M][K], y [M][N], all of type t; 1 <= M <= 16 and M * K * 4
 * bytes within the shared memory of one CTA (DG_ERR_UNSUPPORTED otherwise).
 * Products are exact in fp32 and summed in fp32; y = round-to-nearest-even of
 * the fp32 sum.  ws may be NULL.  With ws (16-byte aligned) of at least
 * dg_workspace_bytes(&op, 1) bytes for the equivalent dg_linear, a call with
 * few rows may split K across CTAs (see Determinism above); with less, or
 * NULL, it does not.  The same holds for dg_gemv_w8a8 and dg_gemv_w4. */
dg_status dg_gemv_f16(const void* W, const void* x, void* y, dg_ftype t, int M, int N, int K,
                      void* ws, size_t ws_bytes, dg_stream stream);

/* W8A8 ("vLLM Arm CPU optimizations", section "INT8 W8A8").
 * W int8 [N][K], w_scale float [N] (per output channel), x int8 [M][K],
 * x_scale float [M] (per token), 1 <= M <= 16.
 * acc[m][n] = sum_k W[n][k] x[m][k] exactly in int32 (|acc| <= K*128*128
 * must fit: K <= 131072); y[m][n] = fp16(float(acc) * w_scale[n] * x_scale[m]).
 * acc_out (int32 [M][N]) receives acc when non-NULL. */
dg_status dg_gemv_w8a8(const int8_t* W, const float* w_scale, const int8_t* x,
                       const float* x_scale, void* y, int32_t* acc_out, int M, int N, int K,
                       void* ws, size_t ws_bytes, dg_stream stream);

/* Groupwise int4 weights ("vLLM Arm CPU optimizations", section "INT8 W4A8";
 * fused INT4 dequantization of the Orange Pi AIPro post's closing paragraph).
 * Wq uint8 [N][K/2]: byte j of a row holds k = 2j in bits 0-3 and k = 2j+1 in
 * bits 4-7 as 4-bit two's complement (codes -8..7).  scales fp16
 * [N][K/group_size]; group_size a multiple of 32 that divides K.
 * W4A16 when x_i8 == NULL:  y = fp16( sum_g s[n][g] * P_g ),
 *                           P_g = sum_{k in g} q[n][k] * x[m][k]   (fp32)
 * W4A8 when x_i8 != NULL:   acc_g = sum_{k in g} q * x_i8 (exact int32),
 *                           y = fp16( x_scale[m] * sum_g s[n][g] * acc_g ).
 * x_f16 [M][K] is read for W4A16 and ignored for W4A8.  1 <= M <= 16, and the
 * staged activations (2 bytes per element for W4A16, about 1 for W4A8) must
 * fit one CTA's shared memory (DG_ERR_UNSUPPORTED otherwise). */
dg_status dg_gemv_w4(const uint8_t* Wq, const void* scales, int group_size, const void* x_f16,
                     const int8_t* x_i8, const float* x_scale, void* y, int M, int N, int K,
                     void* ws, size_t ws_bytes, dg_stream stream);

/* One op described by a dg_linear (any kind except an lm_head; any epilogue),
 * M <= 16, as one launch (two with split-K).  Same arithmetic as the
 * dg_gemv_* entry points of its kind; ws as for them (may be NULL; an op
 * with an epilogue never splits K).  W8A8 / W4A8 ops read x_i8 / x_scale
 * and must not carry fp16 x here (quantize first with dg_quantize_act_i8). */
dg_status dg_linear_forward(const dg_linear* op, void* ws, size_t ws_bytes, dg_stream stream);

/* Elementwise fp16 epilogues as separate launches (what a decoder runs when
 * they are not fused into the weight stream; same fp32 arithmetic):
 *   dg_swiglu:       h[i] = fp16( silu(g[i]) * u[i] )
 *   dg_residual_add: out[i] = fp16( a[i] + b[i] )
 * n elements; pointers 16-byte aligned, n a multiple of 8; out may alias a
 * or b (elementwise), h may alias g or u. */
dg_status dg_swiglu(const void* g, const void* u, void* h, int n, dg_stream stream);
dg_status dg_residual_add(const void* a, const void* b, void* out, int n, dg_stream stream);

/* One decode step of a depthwise causal 1-D convolution (the causal-conv1d
 * step kernel of "MiniCPM-V on Orange Pi AIPro (Ascend 310B)"; the page gives
 * no formula, this is the plain definition).  For token m and channel c, with
 * u = state[m][c][0 .. width-2] (oldest first) followed by x[m][c]:
 *   v = bias[c] + sum_{j < width} w[c][j] * u[j]     (fp32: exact products,
 *       one rounding per term, j ascending after the bias)
 *   y[m][c] = fp16(act == DG_ACT_SILU ? silu(v) : v)
 * then state[m][c] becomes u[1 .. width-1] (the oldest input drops out).
 * x, y fp16 [M][C]; state fp16 [M][C][width-1] (read and rewritten in place);
 * w fp16 [C][width]; bias fp16 [C] or NULL.  2 <= width <= 8, C a multiple
 * of 8, pointers 16-byte aligned; y must not overlap state. */
typedef enum { DG_ACT_NONE = 0, DG_ACT_SILU = 1 } dg_act;
dg_status dg_causal_conv1d_update(const void* x, void* state, const void* w, const void* bias,
                                  void* y, int M, int C, int width, int act, dg_stream stream);

/* Load-time weight quantizers and packers ("vLLM Arm CPU optimizations",
 * section "Dense layer weight prepacking": weights are put in the kernels'
 * format once, at warm-up).  Decided in IEEE fp32, as the library's kernels
 * expect them; W fp16 [N][K] (16-byte aligned, K a multiple of 16 / of
 * group_size).
 *   dg_quantize_weights_i8: s[n] = max_k |W[n][k]| / 127 (1 for an all-zero
 *     row), Wq[n][k] = clamp(rne(W / s), -127, 127)  -> DG_LINEAR_W8A8 input.
 *   dg_quantize_weights_w4: per group of group_size k, s = fp16(amax / 7)
 *     raised to the smallest fp16 subnormal if it rounds to 0 (1 for an
 *     all-zero group), code = clamp(rne(W / s), -7, 7), packed two per byte
 *     (k = 2j in bits 0-3 of byte j, k = 2j+1 in bits 4-7); scales fp16
 *     [N][K/group_size]  -> DG_LINEAR_W4A16 / W4A8 input. */
dg_status dg_quantize_weights_i8(const void* W, int8_t* Wq, float* w_scale, int N, int K,
                                 dg_stream stream);
dg_status dg_quantize_weights_w4(const void* W, uint8_t* Wq, void* scales, int N, int K,
                                 int group_size, dg_stream stream);

/* Per-token symmetric int8 activations for W8A8 / W4A8 (same page, same
 * sections).  x fp16 [M][K] -> xq int8 [M][K], x_scale float [M]:
 *   amax = max_k |x[m][k]|,  s = amax / 127 (IEEE fp32 division),
 *   q = clamp(round-half-even(x / s), -127, 127);  s = 1, q = 0 if amax = 0. */
dg_status dg_quantize_act_i8(const void* x, int8_t* xq, float* x_scale, int M, int K,
                             dg_stream stream);

/* Wide lm_head with fused greedy argmax (paragraph on the ~248k-vocabulary
 * lm_head of the Orange Pi AIPro post, which splits it into 16 slices and
 * reduces on the host; here one launch plus a tiny second pass).
 * head->kind is DG_LINEAR_F16, DG_LINEAR_BF16, DG_LINEAR_W4A16 or
 * DG_LINEAR_W4A8; head->M must be 1.  Writes fp32 logits[N] and
 * token = the index of the largest logit, the lowest index on exact ties
 * (+0 equals -0); a NaN logit never wins.  Needs dg_workspace_bytes(head, 1)
 * bytes of workspace (per-CTA (value, index) partials). */
dg_status dg_lm_head_argmax(const dg_linear* head, void* ws, size_t ws_bytes, dg_stream stream);

/* dg_lm_head_argmax without a workspace argument, for callers that cannot
 * allocate device memory: a decode loop that must not allocate once running,
 * a plugin whose host runtime owns all device memory through its own pool, or
 * code whose memory plan was fixed ahead of time.  (The pages have no
 * counterpart to this entry point.)  Same inputs, outputs and results as
 * dg_lm_head_argmax (the same kernels and launch configuration, so the same
 * bits); the per-CTA partials live in a fixed 16 KB array inside the library
 * (2048 partials; every GPU that loads the library keeps it until the
 * process exits).  A head launches at most SMs x 8 CTAs (1216 on a 152-SM
 * GB300), so every head fits there.
 *  - The first call on a device looks up that array's address (with the
 *    device current) and caches it: make that first call before any stream
 *    capture.  The cached address belongs to the device's primary context:
 *    do not keep using the library across a cudaDeviceReset of that device.
 *    No call allocates or frees memory.
 *  - A head that would need more than 2048 partials (a GPU with more than 256
 *    SMs) returns DG_ERR_WORKSPACE and launches nothing.
 *  - Every call shares the array; nothing in it needs to start at zero (each
 *    call writes every partial it reads).  Calls that can overlap on the GPU
 *    (different streams, or different host threads on one device) race on the
 *    array: serialize them. */
dg_status dg_lm_head_argmax_noalloc(const dg_linear* head, dg_stream stream);

/* One decode step's weight stream (graph-accelerated decode of EdgeFM,
 * section 2.C): runs ops[0..n_ops) in order.  Consecutive ops of the same
 * kind that read the same activations (same x / x_i8 / x_scale pointers,
 * same M, K and group) and are not lm_heads are fused (q|k|v, gate|up); every
 * other boundary is a dependency: an op reads its activations only after
 * every earlier op finished.
 * Runs of single-token ops (M = 1, no acc_out) of one kind execute as ONE
 * persistent cooperative launch: one CTA per SM takes a contiguous row slice
 * of every fused group, groups meet at a grid-wide barrier, and each CTA
 * prefetches its upcoming weight rows into L2 ahead of use, across group
 * boundaries.  Other ops run as one launch per fused group.  Both give the
 * same bits as calling dg_gemv_* / dg_lm_head_argmax op by op.
 * For W8A8 / W4A8 ops that carry fp16 `x`, the step quantizes x exactly as
 * dg_quantize_act_i8 does and also writes the codes / scale to x_i8 / x_scale.
 * Ops may carry epilogues (dg_epilogue): a SwiGLU op streams W and W2 row by
 * row in pairs, and an op reading another op's output (the down projection
 * reading the SwiGLU result) waits for it like any other dependency.
 * Weights and scales must stay unchanged during the step (they are read
 * early).  ws: dg_workspace_bytes(ops, n_ops) bytes, 16-byte aligned, owned
 * by the caller; the step overwrites it (nothing needs to be zeroed first).
 * A barrier wait that exceeds its bound (about a second) makes the launch
 * end early; dg_check_device_status then reports DG_ERR_TIMEOUT. */
dg_status dg_decode_step_weights(const dg_linear* ops, int n_ops, void* ws, size_t ws_bytes,
                                 dg_stream stream);

/* Workspace bytes that dg_decode_step_weights needs for these ops (256 for
 * the persistent kernel's barrier, plus 32 KB of argmax partials when an op is
 * an lm_head, plus, per int4 op at M = 1, its activations in the kernel's
 * layout: DG_LINEAR_W4A8 ceil(K/1024)*1024 + K/8 bytes, DG_LINEAR_W4A16
 * ceil(K/1024)*2048 bytes, each rounded up to 256); for a
 * single lm_head this also covers dg_lm_head_argmax; for a single op of at
 * most 65536 outputs (M * N) it also covers split-K partials of a dg_gemv_*
 * call (8 ranges x M x N x 4 bytes).
 * 0 for n_ops <= 0.  Host-only; touches no device. */
size_t dg_workspace_bytes(const dg_linear* ops, int n_ops);

/* Synchronizes `stream`, then reports DG_ERR_CUDA for a sticky CUDA error or
 * DG_ERR_TIMEOUT if a bounded device-side wait gave up on the current device
 * since the last call (clearing that flag).  DG_OK otherwise. */
dg_status dg_check_device_status(dg_stream stream);

/* Diagnostic (not part of the method): launches one tiny kernel that waits on
 * a device word nothing ever sets, with the same bounded wait the step
 * kernel's barriers use, giving up after `spin_limit` polls (1..10^7, ~100 ns
 * each).  The following dg_check_device_status reports DG_ERR_TIMEOUT: the
 * failure path can be exercised without hanging or faulting anything. */
dg_status dg_selftest_wait_timeout(unsigned spin_limit, dg_stream stream);

/* Static, human-readable name of a status. */
const char* dg_status_string(dg_status s);

/* Measurement probes (not part of the method): stream `bytes` through HBM.
 * dg_probe_copy copies src to dst (bytes read + bytes written);
 * dg_probe_read reads src and writes one word per CTA to sink[0..1023].
 * bytes must be a multiple of 16; pointers 16-byte aligned. */
dg_status dg_probe_copy(const void* src, void* dst, size_t bytes, dg_stream stream);
dg_status dg_probe_read(const void* src, size_t bytes, uint32_t* sink, dg_stream stream);

/* Library version string. */
const char* dg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DG_H_ */
