// Persistent decode-step kernel: one cooperative launch streams a whole
// decode step's weights (graph-accelerated decode of EdgeFM, section 2.C,
// taken one step further: one launch per step instead of one per op).
//
// One CTA per SM.  Each phase (a fused group of ops sharing their
// activations) is split into contiguous row slices, one per CTA, and every CTA
// walks the phases in the ops' order.  Where a phase depends on earlier ones
// (it reads or overwrites memory they wrote, or overwrites what they read; the
// host finds these from the ops' address ranges) the grid meets at a barrier
// first; independent phases flow through without one, so the weight stream
// never stops; each CTA copies the next phase's activations into shared
// memory while it streams the current one.  The per-row arithmetic is the same
// device code as the per-launch kernel (gemv_core.cuh), so every output is
// bitwise what the per-op entry points return.
//
// Every wait is bounded: a barrier that does not complete within the spin
// limit records an error (reported by dg_check_device_status) and the CTA
// leaves; the other CTAs then time out at their next barrier as well.
#include "step_common.cuh"

namespace dg {

// Rows per slot (M = 1): int4 rows are short, so several per warp keep enough
// loads in flight; W4A16 takes four (each activation piece is loaded once for
// the four rows; two chunks of each row are in flight per batch).
template <class P>
struct StepRows { static constexpr int v = P::kMacRows ? 4 : P::kElems == 32 ? 2 : 1; };
// fp16 / bf16 (16 warps): two rows per slot, six chunks of each per batch (a
// 1536-wide row in one round trip); measured against one row per slot at 24
// warps: 475 -> 459 us for the 28-layer 1536-wide step, fewer warps per small
// phase and the same bytes in flight.
template <class P, int NW>
struct StepRowsNW { static constexpr int v = (!P::kIntAct && P::kElems == 8 && NW == 16) ? 2 : StepRows<P>::v; };
template <class P, int NW>
struct StepUnroll { static constexpr int v = (!P::kIntAct && P::kElems == 8 && NW == 16) ? 6 : 0; };
constexpr int kStepRMax = 4;

// Warps per CTA (one CTA per SM): the default for each format, or 16.
template <class P>
struct StepCfg;
template <bool B>
struct StepCfg<PolicyFP<B>> { static constexpr int kWarps = 16; };
template <>
struct StepCfg<PolicyI8> { static constexpr int kWarps = 16; };
template <>
struct StepCfg<PolicyW4A16> { static constexpr int kWarps = 16; };
template <>
struct StepCfg<PolicyW4A8> { static constexpr int kWarps = 16; };

// Grid barrier for a co-resident (cooperative) grid.  bar[0] counts arrivals
// over the whole launch (zeroed before it); barrier number e (1, 2, ...)
// completes when it reaches e * nblocks.  One release add per CTA, then
// acquire polls: a single round trip after the last arrival.
__device__ __forceinline__ bool grid_barrier(unsigned* bar, unsigned target, unsigned limit,
                                             int* err) {
    __syncthreads();
    int ok = 1;
    if (threadIdx.x == 0) {
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
        for (unsigned n = 0; ld_acquire_gpu(bar) < target; ++n) {
            if (n >= limit) {
                atomicExch(err, kErrTimeout);
                ok = 0;
                break;
            }
            __nanosleep(32);
        }
        __threadfence();
    }
    return __syncthreads_and(ok) != 0;
}

// Per-token int8 quantization of the fp16 activations of one token into
// shared memory, with the arithmetic of k_quant_act: amax = max |x|,
// s = amax / 127 (IEEE), q = clamp(rne(x / s), -127, 127); s = 1, q = 0 if
// amax = 0.  Returns s (in every thread).
__device__ float quantize_token_smem(const __half* x, int K, int8_t* q, float* red) {
    float amax = 0.f;
    for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(x + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(u32_as_h2(w[i]));
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, red[w]);
    __syncthreads();
    const float s = amax > 0.f ? __fdiv_rn(amax, 127.f) : 1.f;
    for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(x + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(u32_as_h2(w[i]));
            int q0 = 0, q1 = 0;
            if (amax > 0.f) {
                q0 = max(-127, min(127, __float2int_rn(__fdiv_rn(f.x, s))));
                q1 = max(-127, min(127, __float2int_rn(__fdiv_rn(f.y, s))));
            }
            out[i >> 1] |= ((uint32_t)(q0 & 0xFF) | ((uint32_t)(q1 & 0xFF) << 8)) << ((i & 1) * 16);
        }
        *reinterpret_cast<uint2*>(q + k) = make_uint2(out[0], out[1]);
    }
    return s;
}

// The launch's prologue.  CTA b takes the b-th, (b+G)-th, ... phase flagged
// kPhasePreQuant or kPhaseXLaid (each distinct input once, not once per CTA):
// a kPhasePreQuant input is quantized with the arithmetic of k_quant_act into
// the phase's x_i8 / x_scale; a kPhaseXLaid phase's activations (W4A8: the
// codes just quantized, or given; W4A16: the fp16 input) are then written in
// the format's layout to its xlay, from where every CTA's MACs read them.
template <class P>
__device__ void prologue(const StepParams& sp, int8_t* qbuf, float* red) {
    int j = 0;
    for (int p = 0; p < sp.nphase; ++p) {
        const StepPhase& ph = sp.ph[p];
        if (!(ph.flags & (kPhasePreQuant | kPhaseXLaid))) continue;
        if (j++ % (int)gridDim.x != (int)blockIdx.x) continue;
        const int8_t* codes = ph.xq;
        if (ph.flags & kPhasePreQuant) {
            const float s = quantize_token_smem(static_cast<const __half*>(ph.x), ph.K, qbuf, red);
            __syncthreads();
            for (int k = threadIdx.x * 16; k < ph.K; k += blockDim.x * 16)
                *reinterpret_cast<uint4*>(ph.xq_out + k) = *reinterpret_cast<const uint4*>(qbuf + k);
            if (threadIdx.x == 0) ph.x_scale[0] = s;
            codes = qbuf;
        }
        if (ph.flags & kPhaseXLaid) {
            ActIn a{ph.x, codes, ph.x_scale, ph.K, 1};  // W4A16 reads x, W4A8 the codes
            P::stage_x(a, ph.xlay, 1);
        }
        __syncthreads();
    }
}

// Staged activations (formats that read x from shared memory).
template <class P>
__host__ __device__ constexpr size_t step_smem_layout_x(int max_k) {
    return P::kDirectX ? 0 : (P::x_bytes(1, max_k) + 15) & ~(size_t)15;
}
// Each of the two raw activation buffers (none when x is read from global).
template <class P>
__host__ __device__ constexpr size_t step_raw_bytes(int max_k) {
    return P::kDirectX ? 0 : ((size_t)max_k * 2 + 15) & ~(size_t)15;
}

// Raw activation bytes of a phase as they sit in global memory: fp16 / bf16 x,
// or the given int8 codes.
template <class P>
__device__ __forceinline__ int raw_act_bytes(const StepPhase& ph) {
    return (P::kIntAct && !(ph.flags & kPhaseQuantize)) ? ph.K : ph.K * 2;
}
template <class P>
__device__ __forceinline__ const void* raw_act_src(const StepPhase& ph) {
    if (P::kIntAct && (ph.flags & kPhasePreQuant)) return ph.xq_out;
    return (P::kIntAct && !(ph.flags & kPhaseQuantize)) ? static_cast<const void*>(ph.xq) : ph.x;
}

// Copies `bytes` (a multiple of 16, 16-byte aligned ends) from global to
// shared memory with cp.async, all threads of the CTA, one commit group.
__device__ __forceinline__ void async_copy_block(void* dst, const void* src, int bytes) {
    for (int off = threadIdx.x * 16; off < bytes; off += blockDim.x * 16) {
        const unsigned s = (unsigned)__cvta_generic_to_shared(static_cast<char*>(dst) + off);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s),
                     "l"(static_cast<const char*>(src) + off)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Shared memory of k_step: phase table | staged activations | two raw
// activation buffers | scratch (sized for the largest CTA).
template <class P>
__host__ __device__ size_t step_smem_for(int max_k) {
    constexpr int NW = 32;  // the largest CTA any format uses
    return kPhaseTableBytes + step_smem_layout_x<P>(max_k) + 2 * step_raw_bytes<P>(max_k) +
           (size_t)NW * kStepRMax * 4 + (size_t)NW * sizeof(ArgPart) + (size_t)NW * 4 + 16 +
           (P::kDirectX ? 0 : (size_t)max_k + 16);
}

// EPI: the launch has epilogue phases (residual adds, SwiGLU pairs); the
// variant without them carries none of that code.
template <class P, int NW, bool EPI>
__global__ void __launch_bounds__(NW * 32, 1)
    k_step(const __grid_constant__ StepParams sp, int max_k) {
    extern __shared__ __align__(16) unsigned char smem[];
    using Acc = typename P::Acc;
    constexpr int R = StepRowsNW<P, NW>::v;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x, b = blockIdx.x;

    // shared memory: phase table | staged activations | two raw activation
    // buffers | scratch
    PhaseSlice* table = reinterpret_cast<PhaseSlice*>(smem);
    const size_t raw_bytes = step_raw_bytes<P>(max_k);
    unsigned char* xs_fmt = smem + kPhaseTableBytes;
    unsigned char* rawx[2] = {xs_fmt + step_smem_layout_x<P>(max_k),
                              xs_fmt + step_smem_layout_x<P>(max_k) + raw_bytes};
    int* red = reinterpret_cast<int*>(rawx[1] + raw_bytes);
    ArgPart* cta_best = reinterpret_cast<ArgPart*>(red + NW * kStepRMax);
    float* fred = reinterpret_cast<float*>(cta_best + NW);
    float* sx_smem = fred + NW;
    int8_t* qraw = reinterpret_cast<int8_t*>(sx_smem + 4);
    bool staged_ahead = false;  // this phase's raw activations are already in flight

    unsigned nbar = 0;  // grid barriers passed
    // work units: row groups of R rows
    plan_phases(sp, table, b, G, [](const StepPhase&, int n) { return (n + R - 1) / R; });

    if constexpr (!P::kDirectX) {
        if (sp.prequant) {
            prologue<P>(sp, qraw, fred);
            ++nbar;
            if (!grid_barrier(sp.bar, nbar * G, sp.spin_limit, sp.err)) return;
        }
    }

    // The first read of a phase's parameters on an SM misses the constant
    // cache; thread 0 touches the lines of phase p + 2 while phase p runs (the
    // values only feed a comparison at the end, so the loads never stall it).
    int touch = 0;
    for (int p = 0; p < sp.nphase; ++p) {
        const StepPhase& ph = sp.ph[p];
        if (threadIdx.x == 0 && p + 2 < sp.nphase) {
            const int* w = reinterpret_cast<const int*>(&sp.ph[p + 2]);
            touch ^= w[0] ^ w[16] ^ w[32] ^ w[48];
        }
        if (p > 0 && (ph.flags & kPhaseBarrier)) {
            ++nbar;
            if (!grid_barrier(sp.bar, nbar * G, sp.spin_limit, sp.err)) return;
            if ((sp.ph[p - 1].flags & kPhaseHead) && b == 0 && threadIdx.x < 32)
                reduce_token(sp.part, G, sp.ph[p - 1].token);
        }
        float sx = 1.f;
        unsigned char* xs = xs_fmt;
        bool laid = false;
        if constexpr (!P::kDirectX) laid = (ph.flags & kPhaseXLaid) != 0;
        if (laid) {
            // laid out by the prologue: read from global memory in the MACs (the
            // prologue's writes are not in this SM's L1), no staging and no
            // CTA-wide meeting between phases
            xs = ph.xlay;
            if constexpr (P::kIntAct) sx = __ldcg(ph.x_scale);
        } else if constexpr (!P::kDirectX) {
            // activations of this phase: raw bytes in rawx[p & 1] (copied ahead
            // during the previous phase when no barrier separates them), then
            // restaged in the format's layout
            unsigned char* raw = rawx[p & 1];
            if (!staged_ahead) async_copy_block(raw, raw_act_src<P>(ph), raw_act_bytes<P>(ph));
            async_wait_all();
            __syncthreads();
            staged_ahead = false;
            if (p + 1 < sp.nphase && !(sp.ph[p + 1].flags & (kPhaseBarrier | kPhaseXLaid))) {
                const StepPhase& nx = sp.ph[p + 1];
                async_copy_block(rawx[(p + 1) & 1], raw_act_src<P>(nx), raw_act_bytes<P>(nx));
                staged_ahead = true;
            }
            ActIn a{raw, reinterpret_cast<const int8_t*>(raw), ph.x_scale, ph.K, 1};
            if constexpr (P::kIntAct) {
                if (ph.flags & kPhaseQuantize) {
                    const float s = quantize_token_smem(reinterpret_cast<const __half*>(raw), ph.K,
                                                        qraw, fred);
                    __syncthreads();
                    if (b == 0) {  // the documented side outputs of the fused quantization
                        if (ph.xq_out)
                            for (int k = threadIdx.x * 16; k < ph.K; k += blockDim.x * 16)
                                *reinterpret_cast<uint4*>(ph.xq_out + k) =
                                    *reinterpret_cast<const uint4*>(qraw + k);
                        if (threadIdx.x == 0 && ph.x_scale) ph.x_scale[0] = s;
                    }
                    a.xq = qraw;
                    sx = s;
                } else {
                    // given codes, or codes the prologue wrote in this launch
                    // (read through L2: the prologue's writes are not in L1)
                    sx = (ph.flags & kPhasePreQuant) ? __ldcg(ph.x_scale) : __ldg(ph.x_scale);
                }
            }
            P::stage_x(a, xs, 1);
            __syncthreads();
        } else {
            // one token read from global memory in the MACs: no staging and no
            // CTA-wide meeting between phases
            xs = static_cast<unsigned char*>(const_cast<void*>(ph.x));
        }
        const bool coherent = (ph.flags & kPhaseXWritten) != 0;
        const int ks = ph.ks;                  // 1, 2, 4 or 8 warps per row
        const int lks = __ffs(ks) - 1;
        const int slots = NW >> lks;
        const int slot = warp >> lks, kw = warp & (ks - 1);
        const PhaseSlice sl = table[p];
        const RowGeom g = row_geom_gk<P>(ph.K, ph.group, ks, sl.gk);
        const int r0 = sl.r0, r1 = sl.r0 + sl.n;
        const int n_rg = (sl.n + R - 1) / R;
        // row groups are dealt round-robin over the whole step (continuing
        // where the previous phase stopped) so every warp streams a fair share
        const int lead = mod_slots<NW>(sl.deal0, ks);
        const int mine = slot >= lead ? slot - lead : slot - lead + slots;  // first row group
        // the same in all of the slot's warps
        const int iters = n_rg > mine ? div_slots<NW>(n_rg - mine + slots - 1, ks) : 0;
        const bool head = (ph.flags & kPhaseHead) != 0;
        float best_v = NAN;
        int best_i = INT_MAX;

        for (int it = 0; it < iters; ++it) {
            const int rg = mine + it * slots;
            const bool active = true;
            RowRef rows[R];
            {
                const int first = r0 + rg * R;
                const RowRef f = active ? locate_step<EPI>(ph, first, g.rb) : RowRef{};
                // the group's rows in the first row's matrix (segments are
                // contiguous; SwiGLU pairs interleave two): the next rows of it
                const bool one_seg = !(EPI && ph.pair) && f.local + R <= f.seg_rows;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int gr = first + r;
                    if (active && gr < r1) {
                        if (one_seg) {
                            rows[r] = f;
                            rows[r].w = f.w + (size_t)r * g.rb;
                            rows[r].local = f.local + r;
                            rows[r].global = gr;
                        } else {
                            rows[r] = locate_step<EPI>(ph, gr, g.rb);
                        }
                    } else {
                        rows[r] = f;
                        rows[r].valid = false;
                    }
                }
            }
            Acc acc[R][1];
            row_group<P, 1, R, P::kDirectX, StepUnroll<P, NW>::v>(rows, active, g, xs, red, acc,
                                                                  coherent);
            if (kw == 0 && active) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (!rows[r].valid) continue;
                    if (head) {
                        const float v = P::finish(rows[r], acc[r][0], sx);
                        if (lane == 0) {
                            ph.logits[rows[r].global] = v;
                            if (arg_better(v, rows[r].global, best_v, best_i)) {
                                best_v = v;
                                best_i = rows[r].global;
                            }
                        }
                    } else if constexpr (EPI) {
                        if (lane == r && !(ph.pair && (r & 1))) {
                            const int ru = r + 1 < R ? r + 1 : r;  // (pairs: R is even)
                            store_row<P>(rows[r], 0, acc[r][0], sx, ph.res, ph.pair != 0,
                                         rows[ru], acc[ru][0]);
                        }
                    } else if (lane == r) {
                        P::store(rows[r], 0, acc[r][0], sx);
                    }
                }
            }
        }
        if (head) {
            if (lane == 0) {
                cta_best[warp].v = best_v;
                cta_best[warp].i = best_i;
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                float bv = NAN;
                int bi = INT_MAX;
                for (int w = 0; w < NW; ++w)
                    if (arg_better(cta_best[w].v, cta_best[w].i, bv, bi)) {
                        bv = cta_best[w].v;
                        bi = cta_best[w].i;
                    }
                sp.part[b].v = bv;
                sp.part[b].i = bi;
            }
        }
        // (the next phase's first barrier orders its restaging after this phase)
    }

    if (touch == 0x5eed && b == G) sp.err[1] = touch;  // never true (b < G): keeps the loads

    if (sp.ph[sp.nphase - 1].flags & kPhaseHead) {
        ++nbar;
        if (!grid_barrier(sp.bar, nbar * G, sp.spin_limit, sp.err)) return;
        if (b == 0 && threadIdx.x < 32) reduce_token(sp.part, G, sp.ph[sp.nphase - 1].token);
    }
}


template <class P, int NW, bool EPI>
cudaError_t step_run_nw(const StepParams* sp, int grid, size_t smem, cudaStream_t s, int* occ,
                        int max_k) {
    auto fn = k_step<P, NW, EPI>;
    constexpr int threads = NW * 32;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, threads, smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<StepParams*>(sp), &max_k};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(fn), args);
}

template <class P, int NW>
cudaError_t step_run_epi(const StepParams* sp, int grid, size_t smem, cudaStream_t s, int* occ,
                         int max_k, bool epi) {
    return epi ? step_run_nw<P, NW, true>(sp, grid, smem, s, occ, max_k)
               : step_run_nw<P, NW, false>(sp, grid, smem, s, occ, max_k);
}

template <class P>
cudaError_t step_run(const StepParams* sp, int grid, size_t smem, cudaStream_t s, int* occ,
                     int max_k, int nw, bool epi) {
    // W4A8 may run 20 warps (the host picks it only when no phase splits K:
    // the split barriers' id ranges are disjoint up to 16 warps)
    if constexpr (std::is_same<P, PolicyW4A8>::value)
        if (nw == 20) return step_run_epi<P, 20>(sp, grid, smem, s, occ, max_k, epi);
    return step_run_epi<P, StepCfg<P>::kWarps>(sp, grid, smem, s, occ, max_k, epi);
}

size_t step_smem(Fmt f, int max_k) {
    switch (f) {
        case F_F16:
        case F_BF16: return step_smem_for<PolicyFP<false>>(max_k);
        case F_I8: return step_smem_for<PolicyI8>(max_k);
        case F_W4A16: return step_smem_for<PolicyW4A16>(max_k);
        case F_W4A8: return step_smem_for<PolicyW4A8>(max_k);
    }
    return 0;
}

cudaError_t step_launch(Fmt f, const StepParams* sp, int grid, size_t smem, cudaStream_t s,
                        int* occ, int nw, bool epi) {
    int max_k = 0;
    if (sp)
        for (int p = 0; p < sp->nphase; ++p)
            if (sp->ph[p].K > max_k) max_k = sp->ph[p].K;
    switch (f) {
        case F_F16: return step_run<PolicyFP<false>>(sp, grid, smem, s, occ, max_k, nw, epi);
        case F_BF16: return step_run<PolicyFP<true>>(sp, grid, smem, s, occ, max_k, nw, epi);
        case F_I8: return step_run<PolicyI8>(sp, grid, smem, s, occ, max_k, nw, epi);
        case F_W4A16: return step_run<PolicyW4A16>(sp, grid, smem, s, occ, max_k, nw, epi);
        case F_W4A8: return step_run<PolicyW4A8>(sp, grid, smem, s, occ, max_k, nw, epi);
    }
    return cudaErrorInvalidValue;
}

// ---- bounded-wait self test ---------------------------------------------------------
// Waits on a word that nothing ever changes, with the same bounded wait the
// barriers use, so that a test can see the timeout reach the host as a status
// without hanging or faulting anything.
static __device__ unsigned g_never_set = 0;

__global__ void k_wait_selftest(unsigned limit, int* err) {
    if (threadIdx.x == 0) bounded_wait_change(&g_never_set, 0u, limit, err);
}

cudaError_t launch_wait_selftest(unsigned limit, int* err, cudaStream_t s) {
    k_wait_selftest<<<1, 32, 0, s>>>(limit, err);
    return cudaGetLastError();
}

}  // namespace dg
