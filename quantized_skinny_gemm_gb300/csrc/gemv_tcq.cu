// int8 and int4 weights for 8..16 tokens on the 5th-generation tensor cores:
// W8A8 (int8 x int8, exact int32 sums), W4A16 (int4 x fp16) and W4A8 (int4 x
// int8), with the paragraphs the CUDA-core kernels follow for their
// arithmetic ("vLLM Arm CPU optimizations", sections "INT8 W8A8" and "INT8
// W4A8"; fused INT4 dequantization of the Orange Pi AIPro post).
//
// tcgen05 has no int8 kind on this part, so the codes are widened to fp16,
// which holds every int8 and int4 value exactly; a product of two such values
// is exact in the fp32 accumulator.  TMA moves each 128-row x 128-byte weight
// box (128 int8 or 256 int4 codes per row) into a shared-memory ring;
// converter warps widen a box row by row (thread <-> row) into a second ring,
// in the K-major 128-byte swizzled layout the MMA reads (measured: an A operand
// kept in tensor memory and rewritten while the MMAs run issues four times
// slower); the tokens (B) come from shared memory too: fp16 activations by TMA
// in that layout, int8 codes widened into it by the converter warps.
//
// Sums follow the scalar definitions group by group.  Each group of the int4
// formats (or each 1024-k run of W8A8, whose fp32 partial sums stay below
// 2^24 and so are exact integers) accumulates in a TMEM accumulator of its
// own, from a ring of them; the MMA issuer hands the int4 groups over four
// at a time (one commit), and the epilogue warps read them back and apply
// them in ascending k, with the group scales that the TMA producer brought
// into a shared-memory ring of 8-group windows (128 rows x 16 bytes each):
//   W4A16:  a = fmaf(P_g, s_g, a),  P_g the fp32 group sum;  y = fp16(a)
//   W4A8:   a = fmaf(acc_g, s_g, a), acc_g exact;           y = fp16(x_scale * a)
//   W8A8:   acc += run sum (exact int32);  y = fp16(float(acc) * w_scale * x_scale)
// Work is split stream-K over all SMs exactly as in the fp16 tile (gemv_tc.cu),
// at the granularity of one weight box, and a row tile cut between CTAs is
// finished by the last of its CTAs to arrive, in CTA order (int32 pieces for
// W8A8, so the W8A8 sums stay exact whatever the split).
//
// Measured: the epilogue used to load its scales from global memory in
// register windows, whose moves waited on the loads and whose registers
// spilled; with the shared-memory windows and the batched hand-off a
// 14336 x 4096 int4 launch at 16 tokens went from 44 to 26 us.  What paces
// it now is the chain each 256-k box goes through (TMA -> converters -> MMAs
// -> epilogue, two widened slots), about 2200 cycles per box per SM; no unit
// is saturated (ncu: issue 39 %, shared-memory wavefronts 16 %, DRAM 14 %).
//
// CTA roles (warp w runs on scheduler w % 4): warp 0 lane 0 TMA producer;
// warp 1 TMEM owner and (lane 0) MMA issuer; warps 2-5 epilogue (thread <->
// weight row, reading TMEM lane quarter warp % 4); eight converter warps (two
// per row, each widening half of the row's box).  int4: 14 warps, converters
// 6-13, two on every scheduler.  W8A8: 16 warps, converters 6, 7 and 10-15, so
// that the schedulers of the producer and the MMA issuer carry one each and
// the other two three (warps 8 and 9 idle): measured 24.4 -> 23.3 us at 16
// tokens, while the same layout made int4 slower (25.9 -> 26.4 us).
// Every wait is bounded; a timeout records the library's timeout error.
#include "tc_common.cuh"

namespace dg {

using namespace tc;

namespace {

enum QFmt : int { Q_W8A8 = 0, Q_W4A16 = 1, Q_W4A8 = 2 };

constexpr int kQConv = 8 * 32;          // converter threads
constexpr int kQEpiWarp0 = 2;

// Converter index 0..7 of warp w, or -1 (the layouts above).
template <bool INT4>
__device__ __forceinline__ int q_conv_of_warp(int w) {
    if (INT4) return w >= 6 && w < 14 ? w - 6 : -1;
    return w == 6 ? 0 : w == 7 ? 1 : (w >= 10 && w <= 15) ? w - 8 : -1;
}
constexpr int kQRawA = kRows * 128;     // 16 KB weight box
constexpr int kQAccSlots = 16;          // TMEM accumulators (16 columns each)
constexpr int kQRun8 = 1024;            // W8A8: k per exact fp32 run
constexpr int kQBatch = 4;              // int4: groups per accumulator hand-off, at most
constexpr int kQScWin = 8;              // int4: groups per scale window (16 bytes of a scale row)
constexpr int kQScSlots = 8;            // int4: scale windows in the shared-memory ring
constexpr int kQScBytes = kRows * 2 * kQScWin;  // one window for the 128 rows of a tile: 2 KB

template <int F>
struct QTraits {
    static constexpr bool kInt4 = F != Q_W8A8;
    static constexpr bool kActF16 = F == Q_W4A16;
    static constexpr int KS = kInt4 ? 256 : 128;           // k per weight box
    static constexpr int kAtoms = KS / 64;                 // 64-k swizzle atoms per box
    static constexpr int kWideA = kAtoms * kRows * 128;    // widened box: 32 or 64 KB
    static constexpr int kRawB = kActF16 ? kAtoms * 2048 : kTok * KS;  // B bytes per box as loaded
    static constexpr int kConvB = kActF16 ? 0 : kAtoms * 2048;         // widened B per slot
    static constexpr int kStage = kQRawA + kRawB;
    static constexpr int kStages = kInt4 ? 3 : 4;          // raw ring
    static constexpr int kTmemCols = kQAccSlots * kTok;    // accumulators only
    static constexpr int kThreads = (kInt4 ? 14 : 16) * 32;
    static constexpr int kScRing = kInt4 ? kQScSlots * kQScBytes : 0;
    static size_t smem() {
        return (size_t)kStages * kStage + 2 * (size_t)(kWideA + kConvB) + kScRing + 1024 + 1024;
    }
};

struct TcqParams {
    CUtensorMap wmap[kMaxSeg];   // per matrix: bytes {K bytes, rows}, box {128, 128}, 128B swizzle
    CUtensorMap xmap;            // W4A16: fp16 {K, M} box {64, 16} swizzled; else int8 {K, M} box {KS, 16}
    CUtensorMap smap[kMaxSeg];   // int4: fp16 scales {K / group, rows}, box {8 groups, 128 rows}
    void* y[kMaxSeg];            // fp16 [M][rows]
    int32_t* acc_out[kMaxSeg];   // W8A8, optional [M][rows]
    const void* scale[kMaxSeg];  // int4: fp16 [rows][K / group]; W8A8: float [rows]
    int rows[kMaxSeg];
    int tile_begin[kMaxSeg + 1];
    int nseg, nkb, M, K;
    int seg_k;                   // k per accumulator run: the int4 group, or 1024 for W8A8
    int ngroups;                 // int4: K / group (scale row length)
    const float* x_scale;        // W8A8 / W4A8: [M]
    long long total;             // tiles * nkb
    float* part;                 // fixup pieces (fp32, or int32 bits for W8A8)
    unsigned* count;
    int* err;
    unsigned spin;
};

__device__ __forceinline__ int q_seg_of_tile(const TcqParams& p, int tile) {
    int g = 0;
    while (g + 1 < p.nseg && tile >= p.tile_begin[g + 1]) ++g;
    return g;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Byte j of w holds codes k = 2j (bits 0-3) and 2j+1 (bits 4-7), 4-bit two's
// complement.  Returns the fp16 pair (k = 2j low half, 2j+1 high half): byte j
// copied to bytes 0 and 2; 0x64 exponent bits put over the low nibble of the
// low half (1024 + (c ^ 8)) and over the high nibble of the high half
// (1024 + 16 (c ^ 8)); one fp16x2 FMA with (1, 1/16) and (-1032, -72) leaves
// c exactly in both halves.
template <int J>
__device__ __forceinline__ uint32_t widen_int4_pair(uint32_t w) {
    const uint32_t t = prmt(w, 0u, (uint32_t)(J | (4 << 4) | (J << 8) | (4 << 12)));
    const uint32_t u = and_xor(t, 0x00F0000Fu, 0x64806408u);
    const __half2 scl = __halves2half2(__float2half_rn(1.f), __float2half_rn(0.0625f));
    const __half2 off = __halves2half2(__float2half_rn(-1032.f), __float2half_rn(-72.f));
    return h2_as_u32(__hfma2(u32_as_h2(u), scl, off));
}

// Bytes 2j, 2j+1 of w (int8) as the fp16 pair (low, high): the byte with its
// sign bit flipped under exponent bits 0x64 is 1024 + 128 + v, minus 1152.
template <int J>
__device__ __forceinline__ uint32_t widen_int8_pair(uint32_t wf /* w ^ 0x80808080 */) {
    const uint32_t t = prmt(wf, 0x64646464u, J == 0 ? 0x5140u : 0x7362u);
    return h2_as_u32(__hsub2(u32_as_h2(t), __float2half2_rn(1152.f)));
}

}  // namespace

// RS: MMAs (16-k steps) per int4 group (2, 4, 8, 16); unused for W8A8.
template <int F, int RS>
__global__ void __launch_bounds__(QTraits<F>::kThreads, 1) k_gemv_tcq(const __grid_constant__ TcqParams p) {
    using T = QTraits<F>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    constexpr int kQStages = T::kStages;
    constexpr int kSteps = T::KS / 16;  // MMAs per weight box
    // Accumulator batches: the int4 formats hand kB groups (kB adjacent
    // 16-column accumulators, one commit, one TMEM load) to the epilogue at a
    // time; W8A8 one 1024-k run.  kNB batches fill the accumulator ring.
    constexpr int kB = T::kInt4 ? (kSteps / RS < kQBatch ? kSteps / RS : kQBatch) : 1;
    constexpr int kNB = kQAccSlots / kB;
    unsigned char* wideA = smem;                                 // [2][kAtoms][128 rows][128 B]
    unsigned char* convB = wideA + 2 * T::kWideA;                // [2][kAtoms][16][128 B]
    unsigned char* ring = convB + 2 * T::kConvB;                 // [stage]{A box, B box}
    unsigned char* scring = ring + kQStages * T::kStage;         // int4: [kQScSlots][128 rows][8 groups] fp16
    uint64_t* full = reinterpret_cast<uint64_t*>(scring + T::kScRing);
    uint64_t* empty = full + kQStages;
    uint64_t* a_full = empty + kQStages;       // [2]
    uint64_t* a_empty = a_full + 2;            // [2]
    uint64_t* acc_full = a_empty + 2;          // [kQAccSlots]
    uint64_t* acc_empty = acc_full + kQAccSlots;
    uint64_t* mma_done = acc_empty + kQAccSlots;
    uint64_t* sc_full = mma_done + 1;          // [kQScSlots]
    uint64_t* sc_empty = sc_full + kQScSlots;  // [kQScSlots]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sc_empty + kQScSlots);
    int* last_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long G = gridDim.x, c = blockIdx.x;
    const long long b0 = range_begin(c, p.total, G), b1 = range_begin(c + 1, p.total, G);
    const int nkb = p.nkb;
    const int nblk = (int)(b1 - b0);
    const int t0 = (int)(b0 / nkb), kb_first = (int)(b0 % nkb);

    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int g = 0; g < p.nseg; ++g) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.wmap[g]))
                         : "memory");
            if (T::kInt4)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.smap[g]))
                             : "memory");
        }
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.xmap))
                     : "memory");
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            mbar_init(smem_addr(&empty[i]), kQConv + 1);  // converters + the MMA's commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&a_full[i]), kQConv);
            mbar_init(smem_addr(&a_empty[i]), 1);
        }
        for (int i = 0; i < kQAccSlots; ++i) {
            mbar_init(smem_addr(&acc_full[i]), 1);
            mbar_init(smem_addr(&acc_empty[i]), 128);
        }
        mbar_init(smem_addr(mma_done), 1);
        for (int i = 0; i < kQScSlots; ++i) {
            mbar_init(smem_addr(&sc_full[i]), 1);
            mbar_init(smem_addr(&sc_empty[i]), 128);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_addr(tmem_slot)),
            "r"(T::kTmemCols)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_wait();

    if (warp == 0 && lane == 0) {
        // ---- TMA producer ----
        int tile = t0, kb = kb_first, g = q_seg_of_tile(p, t0), s = 0, issued = 0;
        int sc_u = 0;  // int4: scale windows issued
        uint32_t ph = 0;
        for (int n = 0; n < nblk; ++n) {
            if (T::kInt4 && (n == 0 || ((kb * (kSteps / RS)) % kQScWin) == 0)) {
                // the 8-group scale window holding this box's groups, for the epilogue
                const int sl = sc_u % kQScSlots;
                if (sc_u >= kQScSlots &&
                    !mbar_wait(smem_addr(&sc_empty[sl]), (uint32_t)(((sc_u / kQScSlots) & 1) ^ 1), p.spin, p.err))
                    break;
                mbar_expect_tx(smem_addr(&sc_full[sl]), kQScBytes);
                tma_load_2d(smem_addr(scring + sl * kQScBytes), &p.smap[g], (kb * (kSteps / RS)) & ~(kQScWin - 1),
                            (tile - p.tile_begin[g]) * kRows, smem_addr(&sc_full[sl]));
                ++sc_u;
            }
            if (n >= kQStages && !mbar_wait(smem_addr(&empty[s]), ph ^ 1u, p.spin, p.err)) break;
            unsigned char* st = ring + s * T::kStage;
            mbar_expect_tx(smem_addr(&full[s]), kQRawA + T::kRawB);
            tma_load_2d(smem_addr(st), &p.wmap[g], kb * 128, (tile - p.tile_begin[g]) * kRows,
                        smem_addr(&full[s]));
            if (T::kActF16) {
#pragma unroll
                for (int a = 0; a < T::kAtoms; ++a)
                    tma_load_2d(smem_addr(st + kQRawA + a * 2048), &p.xmap, kb * T::KS + 64 * a, 0,
                                smem_addr(&full[s]));
            } else {
                tma_load_2d(smem_addr(st + kQRawA), &p.xmap, kb * T::KS, 0, smem_addr(&full[s]));
            }
            issued = n + 1;
            if (++kb == nkb) {
                kb = 0;
                ++tile;
                if (g + 1 < p.nseg && tile >= p.tile_begin[g + 1]) ++g;
            }
            if (++s == kQStages) {
                s = 0;
                ph ^= 1u;
            }
        }
        for (int j = issued > kQStages ? issued - kQStages : 0; j < issued; ++j)
            mbar_wait(smem_addr(&full[j % kQStages]), (uint32_t)((j / kQStages) & 1), p.spin, p.err);
        for (int j = sc_u > kQScSlots ? sc_u - kQScSlots : 0; j < sc_u; ++j)
            mbar_wait(smem_addr(&sc_full[j % kQScSlots]), (uint32_t)((j / kQScSlots) & 1), p.spin, p.err);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer: A and B from shared memory ----
        constexpr uint32_t idesc = idesc_f16<false>();
        int kb = kb_first, s = 0, acc_i = 0;  // acc_i: accumulator batches issued
        int run_left = 0;  // W8A8: k left in the current run (0: start a new one)
        uint32_t ph = 0;
        bool ok = true;
        for (int n = 0; n < nblk && ok; ++n) {
            const int r = n & 1;
            if (!mbar_wait(smem_addr(&a_full[r]), (uint32_t)((n >> 1) & 1), p.spin, p.err)) break;
            tc_fence_after();
            const bool piece_first = n == 0 || kb == 0;
            const bool piece_last = n == nblk - 1 || kb == nkb - 1;
            const uint64_t da = sw128_desc(smem_addr(wideA + r * T::kWideA));
            const uint64_t db = sw128_desc(T::kActF16 ? smem_addr(ring + s * T::kStage + kQRawA)
                                                       : smem_addr(convB + r * T::kConvB));
            // k step j: A at atom j / 4 (16 KB apart), B at atom j / 4 (2 KB apart),
            // 32 bytes per step inside an atom (descriptor addresses count 16 bytes)
            if (T::kInt4) {  // RS steps per group, kB groups per batch: boxes hold whole batches
#pragma unroll
                for (int bb = 0; bb < kSteps / (RS * kB); ++bb) {
                    if (acc_i >= kNB &&
                        !mbar_wait(smem_addr(&acc_empty[acc_i % kNB]), (uint32_t)((acc_i / kNB - 1) & 1),
                                   p.spin, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d0 = tmem + (uint32_t)((acc_i % kNB) * kB * kTok);
#pragma unroll
                    for (int gg = 0; gg < kB; ++gg) {
#pragma unroll
                        for (int jj = 0; jj < RS; ++jj) {
                            const int j = (bb * kB + gg) * RS + jj;
                            tc_mma(d0 + (uint32_t)(gg * kTok),
                                   da + (uint64_t)(((j >> 2) * (kRows * 128) + (j & 3) * 32) >> 4),
                                   db + (uint64_t)(((j >> 2) * 2048 + (j & 3) * 32) >> 4), idesc,
                                   jj ? 1u : 0u);
                        }
                    }
                    tc_commit(smem_addr(&acc_full[acc_i % kNB]));
                    ++acc_i;
                }
                if (!ok) break;
            } else {  // W8A8: a run spans whole boxes (1024 k), cut at piece edges
                if (piece_first) run_left = 0;
                uint32_t fresh = 0;
                if (run_left == 0) {
                    if (acc_i >= kNB &&
                        !mbar_wait(smem_addr(&acc_empty[acc_i % kNB]), (uint32_t)((acc_i / kNB - 1) & 1),
                                   p.spin, p.err))
                        break;
                    tc_fence_after();
                    run_left = p.seg_k - ((kb * T::KS) & (p.seg_k - 1));
                    fresh = 1;
                }
                const uint32_t d = tmem + (uint32_t)((acc_i % kNB) * kTok);
#pragma unroll
                for (int j = 0; j < kSteps; ++j)
                    tc_mma(d, da + (uint64_t)(((j >> 2) * (kRows * 128) + (j & 3) * 32) >> 4),
                           db + (uint64_t)(((j >> 2) * 2048 + (j & 3) * 32) >> 4), idesc,
                           (fresh && j == 0) ? 0u : 1u);
                run_left -= T::KS;
                if (run_left == 0 || piece_last) {
                    tc_commit(smem_addr(&acc_full[acc_i % kNB]));
                    ++acc_i;
                    run_left = 0;
                }
            }
            tc_commit(smem_addr(&a_empty[r]));
            tc_commit(smem_addr(&empty[s]));
            if (++kb == nkb) kb = 0;
            if (++s == kQStages) {
                s = 0;
                ph ^= 1u;
            }
        }
        tc_commit(smem_addr(mma_done));
        mbar_wait(smem_addr(mma_done), 0, p.spin, p.err);
    } else if (q_conv_of_warp<T::kInt4>(warp) >= 0) {
        // ---- converters: widen the weight box (and int8 tokens) into the MMA's layout ----
        const int cw = q_conv_of_warp<T::kInt4>(warp);  // 0..7
        const int half = cw >> 2;                   // which half of the row's 8 raw chunks
        const int row = 32 * (cw & 3) + lane;
        const int ct = cw * 32 + lane;              // 0..255
        int s = 0;
        uint32_t ph = 0;
        for (int n = 0; n < nblk; ++n) {
            const int r = n & 1;
            if (!mbar_wait_sleep(smem_addr(&full[s]), ph, p.spin, p.err)) break;
            if (n >= 2 && !mbar_wait_sleep(smem_addr(&a_empty[r]), (uint32_t)(((n >> 1) - 1) & 1), p.spin, p.err))
                break;
            const unsigned char* st = ring + s * T::kStage;
            unsigned char* arow = wideA + r * T::kWideA + row * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int ch = 4 * half + i;   // raw chunk: 32 int4 codes or 16 int8 codes
                const uint4 w = *reinterpret_cast<const uint4*>(st + row * 128 + ((ch ^ (row & 7)) << 4));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                if (T::kInt4) {
                    // k 32 ch .. 32 ch + 31: atom ch / 2, 16-byte chunks 4 (ch % 2) .. + 3
                    unsigned char* atom = arow + (ch >> 1) * (kRows * 128);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int kc = 4 * (ch & 1) + e;
                        *reinterpret_cast<uint4*>(atom + ((kc ^ (row & 7)) << 4)) =
                            make_uint4(widen_int4_pair<0>(ws[e]), widen_int4_pair<1>(ws[e]),
                                       widen_int4_pair<2>(ws[e]), widen_int4_pair<3>(ws[e]));
                    }
                } else {
                    // k 16 ch .. 16 ch + 15: atom ch / 4, 16-byte chunks 2 (ch % 4), + 1
                    unsigned char* atom = arow + (ch >> 2) * (kRows * 128);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint32_t a = ws[2 * e] ^ 0x80808080u, b = ws[2 * e + 1] ^ 0x80808080u;
                        const int kc = 2 * (ch & 3) + e;
                        *reinterpret_cast<uint4*>(atom + ((kc ^ (row & 7)) << 4)) =
                            make_uint4(widen_int8_pair<0>(a), widen_int8_pair<1>(a), widen_int8_pair<0>(b),
                                       widen_int8_pair<1>(b));
                    }
                }
            }
            if (!T::kActF16) {
                // int8 tokens [16][KS] -> fp16 K-major 128-byte swizzle atoms of 64 k
                constexpr int per = kTok * T::KS / kQConv;   // codes per thread: 8 (W8A8) or 16
                const int m = ct / (kQConv / kTok), k0 = (ct % (kQConv / kTok)) * per;
                const unsigned char* src = st + kQRawA + m * T::KS + k0;
                unsigned char* dst = convB + r * T::kConvB + (k0 >> 6) * 2048 + m * 128;
#pragma unroll
                for (int e = 0; e < per / 8; ++e) {
                    const uint2 w = *reinterpret_cast<const uint2*>(src + 8 * e);
                    const uint32_t a = w.x ^ 0x80808080u, b = w.y ^ 0x80808080u;
                    const int chunk = ((k0 + 8 * e) & 63) >> 3;
                    *reinterpret_cast<uint4*>(dst + ((chunk ^ (m & 7)) << 4)) =
                        make_uint4(widen_int8_pair<0>(a), widen_int8_pair<1>(a), widen_int8_pair<0>(b),
                                   widen_int8_pair<1>(b));
                }
            }
            // generic-proxy stores -> the tensor core's async-proxy reads
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(smem_addr(&a_full[r]));
            mbar_arrive(smem_addr(&empty[s]));
            if (++s == kQStages) {
                s = 0;
                ph ^= 1u;
            }
        }
    } else if (warp >= kQEpiWarp0 && warp < kQEpiWarp0 + 4) {
        // ---- epilogue: 128 threads, thread <-> weight row ----
        const int q = warp & 3;
        const int rl = 32 * q + lane;
        const int t1 = (int)((b1 - 1) / nkb);
        int acc_i = 0;
        // int4 scales: the producer's 8-group windows, in the order it issued them
        int sc_u = 0;
        uint4 swin = make_uint4(0, 0, 0, 0);
        for (int tile = t0; tile <= t1; ++tile) {
            const long long tb = (long long)tile * nkb, te = tb + nkb;
            const long long pb = tb > b0 ? tb : b0, pe = te < b1 ? te : b1;  // this CTA's piece
            const int g = q_seg_of_tile(p, tile);
            const int row = (tile - p.tile_begin[g]) * kRows + rl;
            const bool live = row < p.rows[g];
            float a[kTok];
            int ai[kTok];
#pragma unroll
            for (int m = 0; m < kTok; ++m) {
                a[m] = 0.f;
                ai[m] = 0;
            }
            // the piece's runs, in the MMA issuer's order
            const int k_lo = (int)(pb - tb) * T::KS, k_hi = (int)(pe - tb) * T::KS;
            // one batch per pass: kB groups (int4; k stays a multiple of kB groups,
            // as every piece is whole boxes) or one W8A8 run
            for (int k = k_lo; k < k_hi;) {
                const int k_end = min(k_hi, (k / p.seg_k + kB) * p.seg_k);
                const int slot = acc_i % kNB;
                int gi0 = 0;
                if (T::kInt4) {
                    gi0 = k / p.seg_k;
                    if (sc_u == 0 || (gi0 & (kQScWin - 1)) == 0) {  // the batch opens a window
                        if (sc_u > 0) mbar_arrive(smem_addr(&sc_empty[(sc_u - 1) % kQScSlots]));
                        const int sl = sc_u % kQScSlots;
                        if (mbar_wait_sleep(smem_addr(&sc_full[sl]), (uint32_t)((sc_u / kQScSlots) & 1), p.spin,
                                            p.err))
                            swin = *reinterpret_cast<const uint4*>(scring + sl * kQScBytes + rl * 16);
                        else
                            swin = make_uint4(0, 0, 0, 0);
                        ++sc_u;
                    }
                }
                const bool got =
                    mbar_wait_sleep(smem_addr(&acc_full[slot]), (uint32_t)((acc_i / kNB) & 1), p.spin, p.err);
                if (got) tc_fence_after();
                // kH groups per TMEM read (32 registers at most), the slot released
                // after the last read
                constexpr int kH = kB > 2 ? 2 : kB;
#pragma unroll
                for (int h = 0; h < kB; h += kH) {
                    uint32_t v[kH][16];
                    if (got) {
#pragma unroll
                        for (int gg = 0; gg < kH; ++gg)
                            tmem_ld16_async(tmem + ((uint32_t)(32 * q) << 16) +
                                                (uint32_t)((slot * kB + h + gg) * kTok),
                                            v[gg]);
#pragma unroll
                        for (int gg = 0; gg < kH; ++gg) tmem_ld_wait(v[gg]);
                    } else {
#pragma unroll
                        for (int gg = 0; gg < kH; ++gg)
#pragma unroll
                            for (int j = 0; j < 16; ++j) v[gg][j] = 0u;
                    }
                    if (h + kH == kB) {
                        tc_fence_before();
                        mbar_arrive(smem_addr(&acc_empty[slot]));
                    }
                    if (T::kInt4) {
#pragma unroll
                        for (int gg = 0; gg < kH; ++gg) {  // groups in ascending k
                            const int e = (gi0 + h + gg) & (kQScWin - 1);
                            const uint32_t wd = (e >> 1) == 0 ? swin.x : (e >> 1) == 1 ? swin.y : (e >> 1) == 2 ? swin.z : swin.w;
                            const float sg = __half2float(__ushort_as_half((uint16_t)((e & 1) ? wd >> 16 : wd)));
#pragma unroll
                            for (int m = 0; m < kTok; ++m) a[m] = fmaf(__uint_as_float(v[gg][m]), sg, a[m]);
                        }
                    } else {
#pragma unroll
                        for (int m = 0; m < kTok; ++m) ai[m] += __float2int_rn(__uint_as_float(v[0][m]));
                    }
                }
                ++acc_i;
                k = k_end;
            }
            const bool whole = b0 <= tb && b1 >= te;
            if (!whole) {
                float4* dst = reinterpret_cast<float4*>(
                    p.part + ((size_t)(2 * c + (tile == t0 ? 0 : 1)) * kPiece + (size_t)rl * kTok));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float4 w;
                    if (T::kInt4)
                        w = make_float4(a[4 * j], a[4 * j + 1], a[4 * j + 2], a[4 * j + 3]);
                    else
                        w = make_float4(__int_as_float(ai[4 * j]), __int_as_float(ai[4 * j + 1]),
                                        __int_as_float(ai[4 * j + 2]), __int_as_float(ai[4 * j + 3]));
                    __stcg(dst + j, w);
                }
                named_sync(1, 128);
                const int fc = cta_of_block(tb, p.total, G), lc = cta_of_block(te - 1, p.total, G);
                if (threadIdx.x == 32 * kQEpiWarp0) {
                    unsigned old;
                    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                                 : "=r"(old)
                                 : "l"(p.count + tile)
                                 : "memory");
                    *last_flag = old == (unsigned)(lc - fc) ? 1 : 0;
                }
                named_sync(1, 128);
                if (!*last_flag) continue;
#pragma unroll
                for (int m = 0; m < kTok; ++m) {
                    a[m] = 0.f;
                    ai[m] = 0;
                }
                for (int c0 = fc; c0 <= lc; c0 += 2) {  // two pieces in flight at a time
                    float4 w[2][4];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int cc = c0 + u;
                        if (cc > lc) break;
                        const int first_tile = (int)(range_begin(cc, p.total, G) / nkb);
                        const float4* src = reinterpret_cast<const float4*>(
                            p.part + ((size_t)(2 * cc + (tile == first_tile ? 0 : 1)) * kPiece +
                                      (size_t)rl * kTok));
#pragma unroll
                        for (int j = 0; j < 4; ++j) w[u][j] = __ldcg(src + j);
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        if (c0 + u > lc) break;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (T::kInt4) {
                                a[4 * j] += w[u][j].x;
                                a[4 * j + 1] += w[u][j].y;
                                a[4 * j + 2] += w[u][j].z;
                                a[4 * j + 3] += w[u][j].w;
                            } else {
                                ai[4 * j] += __float_as_int(w[u][j].x);
                                ai[4 * j + 1] += __float_as_int(w[u][j].y);
                                ai[4 * j + 2] += __float_as_int(w[u][j].z);
                                ai[4 * j + 3] += __float_as_int(w[u][j].w);
                            }
                        }
                    }
                }
                if (threadIdx.x == 32 * kQEpiWarp0) p.count[tile] = 0u;
            }
            if (!live) continue;
            const size_t rows = (size_t)p.rows[g];
            __half* y = static_cast<__half*>(p.y[g]);
            if (F == Q_W8A8) {
                const float sw = __ldg(static_cast<const float*>(p.scale[g]) + row);
                int32_t* ao = p.acc_out[g];
#pragma unroll
                for (int m = 0; m < kTok; ++m) {
                    if (m >= p.M) break;
                    if (ao) ao[(size_t)m * rows + row] = ai[m];
                    if (y) y[(size_t)m * rows + row] = __float2half_rn((float)ai[m] * sw * __ldg(p.x_scale + m));
                }
            } else {
#pragma unroll
                for (int m = 0; m < kTok; ++m) {
                    if (m >= p.M) break;
                    y[(size_t)m * rows + row] =
                        __float2half_rn(F == Q_W4A8 ? __ldg(p.x_scale + m) * a[m] : a[m]);
                }
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(T::kTmemCols)
                     : "memory");
}

// ---- host side -------------------------------------------------------------------------

namespace {

int qfmt_of(Fmt f) { return f == F_I8 ? Q_W8A8 : f == F_W4A16 ? Q_W4A16 : Q_W4A8; }

template <int F, int RS>
cudaError_t launch_tcq(TcqParams& p, int grid, cudaStream_t s) {
    const void* fn = reinterpret_cast<const void*>(k_gemv_tcq<F, RS>);
    const size_t smem = QTraits<F>::smem();
    cudaError_t e = smem_attr_once(fn, smem);
    if (e != cudaSuccess) return e;
    void* args[] = {&p};
    return launch_pdl(fn, dim3((unsigned)grid), dim3(QTraits<F>::kThreads), smem, s, args);
}

// The int4 kernels by MMAs per group (groups of 32, 64, 128 or 256 k).
template <int F>
cudaError_t launch_tcq_group(TcqParams& p, int grid, cudaStream_t s) {
    switch (p.seg_k) {
        case 32: return launch_tcq<F, 2>(p, grid, s);
        case 64: return launch_tcq<F, 4>(p, grid, s);
        case 128: return launch_tcq<F, 8>(p, grid, s);
        default: return launch_tcq<F, 16>(p, grid, s);
    }
}

}  // namespace

bool gemv_tcq_supported(const GemvParams& p, Fmt f) {
    if (f != F_I8 && f != F_W4A16 && f != F_W4A8) return false;
    if (p.a.M < 1 || p.a.M > kTok || p.t.pair || p.t.res || !have_encoder()) return false;
    const int KS = f == F_I8 ? 128 : 256;
    if (p.a.K % KS) return false;
    if (f != F_I8) {  // groups within one box; scale rows read in 16-byte windows
        if (KS % p.group || p.group < 32 || (p.group & (p.group - 1)) || (p.a.K / p.group) % 8) return false;
        for (int g = 0; g < p.t.nseg; ++g)
            if (reinterpret_cast<uintptr_t>(p.t.seg[g].scale) & 15) return false;
    }
    const void* x = f == F_W4A16 ? p.a.x : static_cast<const void*>(p.a.xq);
    if (!x || (reinterpret_cast<uintptr_t>(x) & 15)) return false;
    int tiles = 0;
    for (int g = 0; g < p.t.nseg; ++g) {
        if (reinterpret_cast<uintptr_t>(p.t.seg[g].W) & 15) return false;
        tiles += (p.t.seg[g].rows + kRows - 1) / kRows;
    }
    return tiles <= kMaxTiles;
}

cudaError_t gemv_tcq(const GemvParams& gp, Fmt f, unsigned spin, int grid_req, cudaStream_t s,
                     bool* launched) {
    *launched = false;
    Scratch scr;
    if (!scratch(s, &scr)) return cudaSuccess;
    TcqParams p;
    memset(&p, 0, sizeof p);
    const int F = qfmt_of(f);
    const int KS = F == Q_W8A8 ? 128 : 256;
    const int K = gp.a.K;
    const long long row_bytes = F == Q_W8A8 ? K : K / 2;
    p.nseg = gp.t.nseg;
    p.M = gp.a.M;
    p.K = K;
    p.nkb = K / KS;
    p.seg_k = F == Q_W8A8 ? kQRun8 : gp.group;
    p.ngroups = F == Q_W8A8 ? 0 : K / gp.group;
    p.x_scale = gp.a.x_scale;
    int tiles = 0;
    for (int g = 0; g < p.nseg; ++g) {
        const Segment& sg = gp.t.seg[g];
        if (!encode_2d(&p.wmap[g], sg.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, row_bytes, sg.rows, 128,
                       kRows, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaSuccess;
        if (F != Q_W8A8 && !encode_2d(&p.smap[g], sg.scale, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K / gp.group,
                                      sg.rows, kQScWin, kRows, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaSuccess;
        p.y[g] = sg.y;
        p.acc_out[g] = sg.acc_out;
        p.scale[g] = sg.scale;
        p.rows[g] = sg.rows;
        p.tile_begin[g] = tiles;
        tiles += (sg.rows + kRows - 1) / kRows;
    }
    p.tile_begin[p.nseg] = tiles;
    const bool ok = F == Q_W4A16
                        ? encode_2d(&p.xmap, gp.a.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K, gp.a.M, 64,
                                    kTok, CU_TENSOR_MAP_SWIZZLE_128B)
                        : encode_2d(&p.xmap, gp.a.xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, gp.a.M, KS,
                                    kTok, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return cudaSuccess;
    p.total = (long long)tiles * p.nkb;
    p.part = scr.part;
    p.count = scr.count;
    p.err = device_error_word();
    p.spin = spin;
    if (!p.err) return cudaSuccess;
    long long grid = grid_req > 0 ? grid_req : sm_count();
    if (grid > kMaxCtas) grid = kMaxCtas;
    if (grid > p.total) grid = p.total;
    if (grid < 1) grid = 1;
    cudaError_t e;
    switch (F) {
        case Q_W8A8: e = launch_tcq<Q_W8A8, 8>(p, (int)grid, s); break;
        case Q_W4A16: e = launch_tcq_group<Q_W4A16>(p, (int)grid, s); break;
        default: e = launch_tcq_group<Q_W4A8>(p, (int)grid, s); break;
    }
    if (e == cudaSuccess) *launched = true;
    return e;
}

}  // namespace dg
