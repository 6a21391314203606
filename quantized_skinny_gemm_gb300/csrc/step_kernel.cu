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
// never stops.  Optionally each CTA keeps an L2 prefetch cursor running ahead
// of its own consumption across phases.  The per-row arithmetic is the same
// device code as the per-launch kernel (gemv_core.cuh), so every output is
// bitwise what the per-op entry points return.
//
// Every wait is bounded: a barrier that does not complete within the spin
// limit records an error (reported by dg_check_device_status) and the CTA
// leaves; the other CTAs then time out at their next barrier as well.
#include "gemv_core.cuh"

namespace dg {

constexpr int kStepR = 1;  // rows per slot (M = 1)

// Warps per CTA (one CTA per SM): the default for each format, or 16.
template <class P>
struct StepCfg;
template <bool B>
struct StepCfg<PolicyFP<B>> { static constexpr int kWarps = 32; };
template <>
struct StepCfg<PolicyI8> { static constexpr int kWarps = 24; };
template <>
struct StepCfg<PolicyW4A16> { static constexpr int kWarps = 24; };
template <>
struct StepCfg<PolicyW4A8> { static constexpr int kWarps = 24; };

// Row r (global over the phase's segments) of phase ph.
__device__ __forceinline__ RowRef locate_step(const StepPhase& ph, int r, size_t rb) {
    RowRef rr{};
    int s = 0;
#pragma unroll
    for (int i = 1; i < kMaxSeg; ++i)
        if (i < ph.nseg && r >= ph.seg[i].row_begin) s = i;
    const StepSeg& sg = ph.seg[s];
    rr.local = r - sg.row_begin;
    rr.w = static_cast<const unsigned char*>(sg.W) + (size_t)rr.local * rb;
    rr.scale = sg.scale;
    rr.y = sg.y;
    rr.acc_out = nullptr;
    rr.seg_rows = sg.rows;
    rr.global = r;
    rr.valid = true;
    return rr;
}

__device__ __forceinline__ int slice_begin(int N, int b, int G) {
    return (int)(((long long)N * b) / G);
}

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

// L2 prefetch cursor of one CTA: the next row (of its own slices, in phase
// order) whose weights have not been prefetched yet, and the bytes of its
// stream before that row.  Kept identically by every lane of warp 0.
struct Cursor {
    int phase;
    int row;         // global row within `phase`
    long long done;  // bytes of this CTA's stream before (phase, row)
};

template <class P>
__device__ __forceinline__ size_t scale_row_bytes(int K, int group) {
    return P::kElems == 32 ? (size_t)(K / group) * 2 : 0;
}

__device__ __forceinline__ void prefetch_range(const unsigned char* p, size_t bytes, int mode) {
    const int lane = threadIdx.x & 31;
    if (mode == 1) {
        if (lane == 0)
            for (size_t off = 0; off < bytes; off += 32768) {
                const size_t left = bytes - off;
                prefetch_l2(p + off, (uint32_t)(left < 32768 ? left : 32768));
            }
    } else {
        for (size_t off = (size_t)lane * 128; off < bytes; off += 32 * 128) prefetch_line_l2(p + off);
    }
}

// Advances the cursor (all lanes of warp 0) until `target` bytes of this CTA's
// stream have been requested, at most 32 KB of consecutive rows of one matrix
// at a time.
template <class P>
__device__ void prefetch_until(const StepParams& sp, Cursor& cu, long long target) {
    const int G = gridDim.x, b = blockIdx.x;
    while (cu.done < target && cu.phase < sp.nphase) {
        const StepPhase& ph = sp.ph[cu.phase];
        const int r1 = slice_begin(ph.N, b + 1, G);
        if (cu.row >= r1) {
            ++cu.phase;
            if (cu.phase < sp.nphase) cu.row = slice_begin(sp.ph[cu.phase].N, b, G);
            continue;
        }
        const size_t rb = P::row_bytes(ph.K);
        const size_t sb = scale_row_bytes<P>(ph.K, sp.group);
        int s = 0;
#pragma unroll
        for (int i = 1; i < kMaxSeg; ++i)
            if (i < ph.nseg && cu.row >= ph.seg[i].row_begin) s = i;
        const StepSeg& sg = ph.seg[s];
        const int seg_end = sg.row_begin + sg.rows;
        int n = (seg_end < r1 ? seg_end : r1) - cu.row;
        int cap = (int)(32768 / rb);
        if (cap < 1) cap = 1;
        if (n > cap) n = cap;
        const size_t local = (size_t)(cu.row - sg.row_begin);
        prefetch_range(static_cast<const unsigned char*>(sg.W) + local * rb, (size_t)n * rb,
                       sp.pf_mode);
        if (sb) {
            const unsigned char* sc = static_cast<const unsigned char*>(sg.scale) + local * sb;
            const size_t bytes = ((size_t)n * sb) & ~(size_t)15;
            // scale rows are 16-byte multiples when K / group is a multiple of 8
            if (bytes && ((uintptr_t)sc & 15) == 0) prefetch_range(sc, bytes, sp.pf_mode);
        }
        cu.row += n;
        cu.done += (long long)n * (long long)(rb + sb);
    }
}

// Bytes of phase p's slice for CTA b.
template <class P>
__device__ __forceinline__ long long slice_bytes(const StepParams& sp, int p, int b, int G) {
    const StepPhase& ph = sp.ph[p];
    const long long rows = slice_begin(ph.N, b + 1, G) - slice_begin(ph.N, b, G);
    return rows * (long long)(P::row_bytes(ph.K) + scale_row_bytes<P>(ph.K, sp.group));
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

template <class P>
__host__ __device__ constexpr size_t step_smem_layout_x(int max_k) {
    return (P::x_bytes(1, max_k) + 15) & ~(size_t)15;
}

template <class P, int NW>
__global__ void __launch_bounds__(NW * 32, 1)
    k_step(const __grid_constant__ StepParams sp, int max_k) {
    extern __shared__ __align__(16) unsigned char smem[];
    using Acc = typename P::Acc;
    constexpr int R = kStepR;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x, b = blockIdx.x;

    unsigned char* xs = smem;
    int* red = reinterpret_cast<int*>(smem + step_smem_layout_x<P>(max_k));
    ArgPart* cta_best = reinterpret_cast<ArgPart*>(red + NW * R);
    float* fred = reinterpret_cast<float*>(cta_best + NW);
    float* sx_smem = fred + NW;
    int8_t* qraw = reinterpret_cast<int8_t*>(sx_smem + 4);

    Cursor cu{0, slice_begin(sp.ph[0].N, b, G), 0};
    unsigned nbar = 0;  // grid barriers passed
    long long consumed = 0;  // bytes of this CTA's slices before the current phase

    for (int p = 0; p < sp.nphase; ++p) {
        const StepPhase& ph = sp.ph[p];
        if (p > 0 && (ph.flags & kPhaseBarrier)) {
            ++nbar;
            if (!grid_barrier(sp.bar, nbar * G, sp.spin_limit, sp.err)) return;
            if ((sp.ph[p - 1].flags & kPhaseHead) && b == 0 && threadIdx.x < 32) {
                // greedy token of the previous (lm_head) phase from the CTAs' partials
                float bv = NAN;
                int bi = INT_MAX;
                for (int i = lane; i < G; i += 32)
                    if (arg_better(sp.part[i].v, sp.part[i].i, bv, bi)) {
                        bv = sp.part[i].v;
                        bi = sp.part[i].i;
                    }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    if (arg_better(ov, oi, bv, bi)) {
                        bv = ov;
                        bi = oi;
                    }
                }
                if (lane == 0) *sp.ph[p - 1].token = bi == INT_MAX ? -1 : bi;
            }
        }
        const long long here = slice_bytes<P>(sp, p, b, G);
        if (warp == 0 && sp.pf_mode != 0 && sp.window > 0) {
            // the current phase is left to the demand loads: start at the next one
            if (cu.phase <= p) {
                cu.phase = p + 1;
                cu.row = p + 1 < sp.nphase ? slice_begin(sp.ph[p + 1].N, b, G) : 0;
                cu.done = consumed + here;
            }
            prefetch_until<P>(sp, cu, consumed + here + sp.window);
        }

        // activations of this phase
        float sx = 1.f;
        ActIn a{ph.x, ph.xq, ph.x_scale, ph.K, 1};
        if constexpr (P::kIntAct) {
            if (ph.flags & kPhaseQuantize) {
                const float s = quantize_token_smem(static_cast<const __half*>(ph.x), ph.K, qraw, fred);
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
                sx = __ldg(ph.x_scale);
            }
        }
        P::stage_x(a, xs, 1);
        __syncthreads();

        const int ks = ph.ks;
        const int slots = NW / ks;
        const int slot = warp / ks, kw = warp - slot * ks;
        const RowGeom g = row_geom<P>(ph.K, sp.group, ks);
        const int r0 = slice_begin(ph.N, b, G), r1 = slice_begin(ph.N, b + 1, G);
        const int n_rg = (r1 - r0 + R - 1) / R;
        const int iters = (n_rg + slots - 1) / slots;
        const bool head = (ph.flags & kPhaseHead) != 0;
        float best_v = NAN;
        int best_i = INT_MAX;

        for (int it = 0; it < iters; ++it) {
            const int rg = it * slots + slot;
            const bool active = rg < n_rg;
            RowRef rows[R];
            {
                const int first = r0 + rg * R;
                const RowRef f = active ? locate_step(ph, first, g.rb) : RowRef{};
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int gr = first + r;
                    if (active && gr < r1) {
                        rows[r] = locate_step(ph, gr, g.rb);
                    } else {
                        rows[r] = f;
                        rows[r].valid = false;
                    }
                }
            }
            Acc acc[R][1];
            row_group<P, 1, R>(rows, active, g, xs, red, acc);
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
        consumed += here;
        __syncthreads();  // shared activations are restaged by the next phase
    }

    if (sp.ph[sp.nphase - 1].flags & kPhaseHead) {
        ++nbar;
        if (!grid_barrier(sp.bar, nbar * G, sp.spin_limit, sp.err)) return;
        if (b == 0 && threadIdx.x < 32) {
            float bv = NAN;
            int bi = INT_MAX;
            for (int i = lane; i < G; i += 32)
                if (arg_better(sp.part[i].v, sp.part[i].i, bv, bi)) {
                    bv = sp.part[i].v;
                    bi = sp.part[i].i;
                }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (arg_better(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (lane == 0) *sp.ph[sp.nphase - 1].token = bi == INT_MAX ? -1 : bi;
        }
    }
}

template <class P>
size_t step_smem_for(int max_k) {
    constexpr int NW = 32;  // the largest CTA any format uses
    return step_smem_layout_x<P>(max_k) + (size_t)NW * kStepR * 4 + (size_t)NW * sizeof(ArgPart) +
           (size_t)NW * 4 + 16 + (size_t)max_k + 16;
}

template <class P, int NW>
cudaError_t step_run_nw(const StepParams* sp, int grid, size_t smem, cudaStream_t s, int* occ,
                        int max_k) {
    auto fn = k_step<P, NW>;
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

template <class P>
cudaError_t step_run(const StepParams* sp, int grid, size_t smem, cudaStream_t s, int* occ,
                     int max_k, int nw) {
    if (nw == 16) return step_run_nw<P, 16>(sp, grid, smem, s, occ, max_k);
    return step_run_nw<P, StepCfg<P>::kWarps>(sp, grid, smem, s, occ, max_k);
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
                        int* occ, int nw) {
    int max_k = 0;
    if (sp)
        for (int p = 0; p < sp->nphase; ++p)
            if (sp->ph[p].K > max_k) max_k = sp->ph[p].K;
    switch (f) {
        case F_F16: return step_run<PolicyFP<false>>(sp, grid, smem, s, occ, max_k, nw);
        case F_BF16: return step_run<PolicyFP<true>>(sp, grid, smem, s, occ, max_k, nw);
        case F_I8: return step_run<PolicyI8>(sp, grid, smem, s, occ, max_k, nw);
        case F_W4A16: return step_run<PolicyW4A16>(sp, grid, smem, s, occ, max_k, nw);
        case F_W4A8: return step_run<PolicyW4A8>(sp, grid, smem, s, occ, max_k, nw);
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
