// Helpers of the persistent decode-step kernel: row addressing within a phase,
// the CTA row slices, and the greedy-token reduction of an lm_head phase.
#pragma once

#include "gemv_core.cuh"

namespace dg {

// Row r (global over the phase's segments) of phase ph; a SwiGLU phase
// (ph.pair) interleaves its gate and up rows: row 2i is gate row i, 2i + 1 up
// row i (PAIRS = false: the launch has no such phase).
template <bool PAIRS = true>
__device__ __forceinline__ RowRef locate_step(const StepPhase& ph, int r, size_t rb) {
    RowRef rr{};
    int s = 0;
    if (PAIRS && ph.pair) {
        s = r & 1;
        rr.local = r >> 1;
    } else {
#pragma unroll
        for (int i = 1; i < kMaxSeg; ++i)
            if (i < ph.nseg && r >= ph.seg[i].row_begin) s = i;
        rr.local = r - ph.seg[s].row_begin;
    }
    const StepSeg& sg = ph.seg[s];
    rr.w = static_cast<const unsigned char*>(sg.W) + (size_t)rr.local * rb;
    rr.scale = sg.scale;
    rr.y = sg.y;
    rr.acc_out = nullptr;
    rr.seg_rows = sg.rows;
    rr.global = r;
    rr.valid = true;
    return rr;
}

// First row of CTA b's contiguous slice of an N-row phase (G CTAs):
// floor(N b / G), from a float estimate corrected exactly (no 64-bit
// division: this runs once per phase in every warp).
__device__ __forceinline__ int slice_begin(int N, int b, int G) {
    const long long nb = (long long)N * b;
    int q = __float2int_rz((float)N * __fdividef((float)b, (float)G));
    while ((long long)q * G > nb) --q;
    while ((long long)(q + 1) * G <= nb) ++q;
    return q;
}

// floor(a / d) for 0 <= a, 1 <= d, both below 2^22: the float estimate is
// within one of the quotient and is corrected exactly.
__device__ __forceinline__ int div_floor_small(int a, int d) {
    int q = __float2int_rz(__fdividef((float)a, (float)d));
    if (q * d > a)
        --q;
    else if ((q + 1) * d <= a)
        ++q;
    return q;
}

// v mod (NW / ks), the slot count, for ks in {1, 2, 4, 8} with compile-time
// divisors (NW / ks rounded down, as the kernels count slots).
template <int NW>
__device__ __forceinline__ int mod_slots(unsigned v, int ks) {
    return ks == 1   ? (int)(v % (unsigned)NW)
           : ks == 2 ? (int)(v % (unsigned)(NW / 2))
           : ks == 4 ? (int)(v % (unsigned)(NW / 4))
                     : (int)(v % (unsigned)(NW / 8));
}

// Per-phase values of one CTA, computed once per launch (plan_phases) so
// that a phase's set-up in the main loop is a few shared-memory loads: the
// slice [r0, r0 + n) of the phase's rows, the phase's scale groups per row
// (K / group; int4), and where the round-robin dealing of the CTA's work
// units (row groups) stands when the phase begins.
struct PhaseSlice {
    int r0, n, gk;
    unsigned deal0;
};
constexpr size_t kPhaseTableBytes = (size_t)kMaxStepPhases * sizeof(PhaseSlice);

// Fills table[0, nphase) for CTA b of G; all threads of the CTA call it.
// Warp w takes phases w, w + nw, ... (parameter reads stay warp-uniform);
// warp 0 then scans the work units.  units(ph, n) = units of n rows.
template <class Units>
__device__ void plan_phases(const StepParams& sp, PhaseSlice* table, int b, int G, Units units) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int p = warp; p < sp.nphase; p += nw) {
        const StepPhase& ph = sp.ph[p];
        // a SwiGLU phase is sliced by pairs, so a pair never straddles CTAs
        const int f = ph.pair ? 2 : 1, Nu = ph.N / f;
        const int r0 = f * slice_begin(Nu, b, G), r1 = f * slice_begin(Nu, b + 1, G);
        if (lane == 0) {
            table[p].r0 = r0;
            table[p].n = r1 - r0;
            table[p].gk = ph.group > 0 ? ph.K / ph.group : 0;
            table[p].deal0 = (unsigned)units(ph, r1 - r0);  // scanned below
        }
    }
    __syncthreads();
    if (warp == 0) {
        unsigned carry = 0;
        for (int base = 0; base < sp.nphase; base += 32) {
            const int p = base + lane;
            const unsigned v = p < sp.nphase ? table[p].deal0 : 0u;
            unsigned inc = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned t = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += t;
            }
            if (p < sp.nphase) table[p].deal0 = carry + inc - v;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
    }
    __syncthreads();
}

// v / (NW / ks) for ks in {1, 2, 4, 8} with compile-time divisors.
template <int NW>
__device__ __forceinline__ int div_slots(int v, int ks) {
    return ks == 1 ? v / NW : ks == 2 ? v / (NW / 2) : ks == 4 ? v / (NW / 4) : v / (NW / 8);
}

// Greedy token of an lm_head phase from the G per-CTA partials, by one full
// warp: the largest logit, lowest index among equals, NaN never wins; -1 if
// every logit is NaN.  The partials were written by other CTAs before a grid
// barrier, so they are read through L2.
__device__ __forceinline__ void reduce_token(const ArgPart* part, int G, int32_t* token) {
    const int lane = threadIdx.x & 31;
    float bv = NAN;
    int bi = INT_MAX;
    for (int i = lane; i < G; i += 32) {
        const float v = __ldcg(&part[i].v);
        const int ix = __ldcg(&part[i].i);
        if (arg_better(v, ix, bv, bi)) {
            bv = v;
            bi = ix;
        }
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
    if (lane == 0) *token = bi == INT_MAX ? -1 : bi;
}

}  // namespace dg
