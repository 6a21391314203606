// fp16 / bf16 weights for 2..16 tokens on the 5th-generation tensor cores
// (tcgen05), the weight stream moved by the Tensor Memory Accelerator.
//
// With several tokens the skinny product is a dense contraction, so each
// weight byte is read once by TMA and multiplied against all tokens by one
// tcgen05.mma:  D[128 weight rows][16 tokens] += W[128][64 k] x[16][64 k]^T,
// the 128 x 16 fp32 accumulator living in tensor memory (TMEM).  Tokens past
// M, rows past a matrix's end and k past K are read as zeros by TMA.
//
// Work split (stream-K): the (row tile, 64-wide k block) pairs of the launch,
// tile-major, are cut into gridDim.x equal contiguous ranges, one per CTA, so
// every SM streams the same number of weight bytes whatever N and K are.  A
// CTA runs one continuous TMA -> MMA pipeline over its range; a tile that its
// range covers whole is rounded and stored by the CTA itself; a tile cut
// between CTAs is finished by whichever of its CTAs arrives last, which adds
// the pieces' fp32 partial sums in CTA order (so the result does not depend on
// arrival order).  No CTA ever waits for another one.  A CTA whose range ends
// inside a tile processes that tile first, so the pieces of a cut tile are
// published early and the CTA holding its last k block, which takes that
// piece last, usually finds them all there: one acquire load tells it so, and
// it finishes the tile without publishing its own piece (measured on a
// 14336 x 4096 launch at 16 tokens: 26.3 -> 25.2 us).
//
// CTA roles (6 warps): warp 0 lane 0 issues TMA loads into a ring of stages of
// NB 64-k boxes (16 KB of weights + 2 KB of tokens per box, 128-byte swizzle;
// by default 4 stages of 2 boxes, 8 MMAs per stage); warp 1 owns
// the TMEM allocation and its lane 0 issues the MMAs; warps 2-5 drain the two
// TMEM accumulators (double-buffered, so a tile's epilogue overlaps the next
// tile's MMAs), each warp reading the 32 TMEM lanes (weight rows) its warp
// index may access.  Every wait is bounded; on a timeout the kernel records
// the library's timeout error, lets its copies and MMAs land, frees TMEM and
// returns.
#include <map>
#include <mutex>
#include <utility>

#include "tc_common.cuh"

namespace dg {

using namespace tc;

namespace {

constexpr int kTcRows = kRows;
constexpr int kTcTok = kTok;
constexpr int kTcBK = 64;                          // k per stage (one 128-byte swizzle row)
constexpr int kTcABytes = kTcRows * kTcBK * 2;     // 16 KB
constexpr int kTcBBytes = kTcTok * kTcBK * 2;      // 2 KB
constexpr int kTcThreads = 192;
constexpr int kTcPiece = kPiece;
constexpr int kTcMaxCtas = kMaxCtas;
// A stage holds NB 64-k boxes (NB MMAs x 4 per commit).
constexpr size_t tc_smem(int stages, int nb) {
    return (size_t)stages * nb * (kTcABytes + kTcBBytes) + 1024 + 256;
}

struct TcParams {
    CUtensorMap wmap[kMaxSeg];   // per matrix: {K, rows} fp16 / bf16, box {64, 128}
    CUtensorMap xmap;            // tokens: {K, M}, box {64, 16}
    void* y[kMaxSeg];            // [M][rows]
    int rows[kMaxSeg];
    int tile_begin[kMaxSeg + 1]; // first tile of each matrix (tiles never straddle two)
    int nseg, nkb, M;
    long long total;             // tiles * nkb
    float* part;                 // [2 * gridDim.x][kTcPiece] partial tiles
    unsigned* count;             // [tiles] pieces arrived; zero between launches
    int* err;
    unsigned spin;               // bound on every mbarrier wait (polls)
    int prefetch;                // weight boxes prefetched to L2 before the dependency wait
};


__device__ __forceinline__ int seg_of_tile(const TcParams& p, int tile) {
    int g = 0;
    while (g + 1 < p.nseg && tile >= p.tile_begin[g + 1]) ++g;
    return g;
}

// This CTA's tiles in processing order.  A range that ends inside a tile
// takes that tile first: its piece is the start of the tile, whose other
// pieces belong to later CTAs, and those take their cut tile ends last; so the
// pieces of a cut tile are published early, and its last piece (whose CTA
// finishes the tile when it finds all the others there) ends the range.
struct TileOrder {
    int t0, t1, kb_first, kb_end, nkb;  // kb_end: one past the last k block of t1
    bool rot;
    __device__ TileOrder(long long b0, long long b1, int nkb_) : nkb(nkb_) {
        t0 = (int)(b0 / nkb);
        kb_first = (int)(b0 % nkb);
        t1 = (int)((b1 - 1) / nkb);
        kb_end = (int)((b1 - 1) % nkb) + 1;
        rot = t1 > t0 && kb_end < nkb;
    }
    __device__ int count() const { return t1 - t0 + 1; }
    __device__ int tile(int i) const { return rot ? (i == 0 ? t1 : t0 + i - 1) : t0 + i; }
    __device__ int kb_lo(int t) const { return t == t0 ? kb_first : 0; }
    __device__ int kb_hi(int t) const { return t == t1 ? kb_end : nkb; }
};

template <bool BF16>
__device__ __forceinline__ void store_tokens(const TcParams& p, int g, int row, const float (&a)[16]) {
    if (row >= p.rows[g]) return;
    const size_t rows = (size_t)p.rows[g];
    if (BF16) {
        __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y[g]);
#pragma unroll
        for (int m = 0; m < kTcTok; ++m)
            if (m < p.M) y[(size_t)m * rows + row] = __float2bfloat16_rn(a[m]);
    } else {
        __half* y = static_cast<__half*>(p.y[g]);
#pragma unroll
        for (int m = 0; m < kTcTok; ++m)
            if (m < p.M) y[(size_t)m * rows + row] = __float2half_rn(a[m]);
    }
}

}  // namespace

template <bool BF16, int kTcStages, int NB>
__global__ void __launch_bounds__(kTcThreads, 1) k_gemv_tc(const __grid_constant__ TcParams p) {
    constexpr int kStA = NB * kTcABytes, kStB = NB * kTcBBytes, kBlkK = NB * kTcBK;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char* sA = smem;                                   // [stage][128 rows][128 B]
    unsigned char* sB = smem + kTcStages * kStA;                // [stage][NB][16 tokens][128 B]
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + kTcStages * kStB);
    uint64_t* empty = full + kTcStages;
    uint64_t* acc_full = empty + kTcStages;                     // [2]
    uint64_t* acc_empty = acc_full + 2;                         // [2]
    uint64_t* mma_done = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    int* last_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long G = gridDim.x, c = blockIdx.x;
    const long long b0 = range_begin(c, p.total, G), b1 = range_begin(c + 1, p.total, G);
    const int nkb = p.nkb;

    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int g = 0; g < p.nseg; ++g)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.wmap[g]))
                         : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.xmap))
                     : "memory");
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            mbar_init(smem_addr(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&acc_full[i]), 1);
            mbar_init(smem_addr(&acc_empty[i]), 128);
        }
        mbar_init(smem_addr(mma_done), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // warm L2 with this CTA's first weight boxes while the previous launch
        // drains (a prefetch never changes what a later load returns)
        if (p.prefetch) {
            const TileOrder ord(b0, b1, nkb);
            int n = 0;
            for (int i = 0; i < ord.count() && n < p.prefetch; ++i) {
                const int tile = ord.tile(i), g = seg_of_tile(p, tile);
                for (int kb = ord.kb_lo(tile); kb < ord.kb_hi(tile) && n < p.prefetch; ++kb, ++n) {
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(
                                         reinterpret_cast<uint64_t>(&p.wmap[g])),
                                     "r"(kb * kBlkK + kTcBK * b), "r"((tile - p.tile_begin[g]) * kTcRows)
                                     : "memory");
                }
            }
        }
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" ::"r"(
                smem_addr(tmem_slot))
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_wait();  // the tokens (and the outputs) belong to the previous launch until here

    const TileOrder ord(b0, b1, nkb);
    if (warp == 0 && lane == 0) {
        // ---- TMA producer ----
        int s = 0, issued = 0;
        uint32_t ph = 0;  // parity of the ring's current lap
        bool ok = true;
        for (int i = 0; i < ord.count() && ok; ++i) {
            const int tile = ord.tile(i), g = seg_of_tile(p, tile);
            for (int kb = ord.kb_lo(tile); kb < ord.kb_hi(tile); ++kb) {
                if (issued >= kTcStages && !mbar_wait(smem_addr(&empty[s]), ph ^ 1u, p.spin, p.err)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(smem_addr(&full[s]), kStA + kStB);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    tma_load_2d(smem_addr(sA + s * kStA + b * kTcABytes), &p.wmap[g], kb * kBlkK + kTcBK * b,
                                (tile - p.tile_begin[g]) * kTcRows, smem_addr(&full[s]));
                    tma_load_2d(smem_addr(sB + s * kStB + b * kTcBBytes), &p.xmap, kb * kBlkK + kTcBK * b, 0,
                                smem_addr(&full[s]));
                }
                ++issued;
                if (++s == kTcStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        // the copies still in flight land before the CTA can leave
        for (int j = issued > kTcStages ? issued - kTcStages : 0; j < issued; ++j)
            mbar_wait(smem_addr(&full[j % kTcStages]), (uint32_t)((j / kTcStages) & 1), p.spin, p.err);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        constexpr uint32_t idesc = idesc_f16<BF16>();
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int i = 0; i < ord.count() && ok; ++i) {  // i: tiles started by this CTA
            const int tile = ord.tile(i), buf = i & 1;
            const int lo = ord.kb_lo(tile), hi = ord.kb_hi(tile);
            if (i >= 2 && !mbar_wait(smem_addr(&acc_empty[buf]), (uint32_t)((i / 2 - 1) & 1), p.spin, p.err))
                break;
            for (int kb = lo; kb < hi; ++kb) {
                if (!mbar_wait(smem_addr(&full[s]), ph, p.spin, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t da = sw128_desc(smem_addr(sA + s * kStA)), db = sw128_desc(smem_addr(sB + s * kStB));
#pragma unroll
                for (int kk = 0; kk < 4 * NB; ++kk)  // box kk / 4, 32 bytes per 16-k step inside it
                    tc_mma(tmem + (uint32_t)(buf * kTcTok),
                           da + (uint64_t)(((kk >> 2) * kTcABytes + (kk & 3) * 32) >> 4),
                           db + (uint64_t)(((kk >> 2) * kTcBBytes + (kk & 3) * 32) >> 4), idesc,
                           (kb == lo && kk == 0) ? 0u : 1u);
                tc_commit(smem_addr(&empty[s]));
                if (kb == hi - 1) tc_commit(smem_addr(&acc_full[buf]));
                if (++s == kTcStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        tc_commit(smem_addr(mma_done));
        mbar_wait(smem_addr(mma_done), 0, p.spin, p.err);
    } else if (warp >= 2) {
        // ---- epilogue: 128 threads, thread <-> weight row of the tile ----
        const int q = warp & 3;                 // TMEM lanes 32q .. 32q + 31
        const int rl = 32 * q + lane;           // row within the tile
        for (int i = 0; i < ord.count(); ++i) {
            const int tile = ord.tile(i), buf = i & 1;
            float a[16];
            if (mbar_wait_sleep(smem_addr(&acc_full[buf]), (uint32_t)((i / 2) & 1), p.spin, p.err)) {
                tc_fence_after();
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kTcTok), a);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) a[j] = 0.f;
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&acc_empty[buf]));
            const int g = seg_of_tile(p, tile);
            const int row = (tile - p.tile_begin[g]) * kTcRows + rl;
            const long long tb = (long long)tile * nkb, te = tb + nkb;
            if (b0 <= tb && b1 >= te) {  // the whole tile is this CTA's
                store_tokens<BF16>(p, g, row, a);
                continue;
            }
            // A piece of a tile shared with other CTAs.  The CTA holding the
            // tile's last k block first looks whether every other piece has
            // arrived (one acquire load); if so it finishes the tile without
            // publishing its own.  Otherwise it publishes its piece (one release
            // by one thread after the epilogue's barrier covers the 128 threads'
            // stores) and the last of the tile's CTAs to arrive finishes it.
            // Either way the pieces are added in CTA order.
            const int fc = cta_of_block(tb, p.total, G), lc = cta_of_block(te - 1, p.total, G);
            asm volatile("bar.sync 1, 128;" ::: "memory");  // every thread has read the last flag
            if (threadIdx.x == 64) {
                int mode = 0;
                if (b1 >= te) {
                    unsigned arrived;
                    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];"
                                 : "=r"(arrived)
                                 : "l"(p.count + tile)
                                 : "memory");
                    mode = arrived == (unsigned)(lc - fc) ? 2 : 0;
                }
                *last_flag = mode;
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            int mode = *last_flag;
            if (mode == 0) {
                float4* dst = reinterpret_cast<float4*>(
                    p.part + ((size_t)(2 * c + (tile == ord.t0 ? 0 : 1)) * kTcPiece + (size_t)rl * kTcTok));
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    __stcg(dst + j, make_float4(a[4 * j], a[4 * j + 1], a[4 * j + 2], a[4 * j + 3]));
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (threadIdx.x == 64) {
                    unsigned old;
                    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                                 : "=r"(old)
                                 : "l"(p.count + tile)
                                 : "memory");
                    *last_flag = old == (unsigned)(lc - fc) ? 1 : 0;
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
                mode = *last_flag;
            }
            if (mode) {
                float own[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    own[j] = a[j];
                    a[j] = 0.f;
                }
                for (int c0 = fc; c0 <= lc; c0 += 4) {  // four pieces in flight at a time
                    float4 v[4][4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int cc = c0 + u;
                        if (cc > lc) break;
                        if (cc == (int)c) {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                v[u][j] = make_float4(own[4 * j], own[4 * j + 1], own[4 * j + 2], own[4 * j + 3]);
                            continue;
                        }
                        const int first_tile = (int)(range_begin(cc, p.total, G) / nkb);
                        const float4* src = reinterpret_cast<const float4*>(
                            p.part + ((size_t)(2 * cc + (tile == first_tile ? 0 : 1)) * kTcPiece +
                                      (size_t)rl * kTcTok));
#pragma unroll
                        for (int j = 0; j < 4; ++j) v[u][j] = __ldcg(src + j);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (c0 + u > lc) break;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            a[4 * j] += v[u][j].x;
                            a[4 * j + 1] += v[u][j].y;
                            a[4 * j + 2] += v[u][j].z;
                            a[4 * j + 3] += v[u][j].w;
                        }
                    }
                }
                store_tokens<BF16>(p, g, row, a);
                if (threadIdx.x == 64) p.count[tile] = 0u;  // ready for the next launch
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(tmem) : "memory");
}

// ---- host side ---------------------------------------------------------------------

namespace tc {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

bool have_encoder() { return encode_fn() != nullptr; }

bool encode_2d(CUtensorMap* m, const void* base, CUtensorMapDataType type, int elem_bytes,
               long long inner, long long outer, int box_inner, int box_outer,
               CUtensorMapSwizzle swizzle) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    const cuuint64_t strides[1] = {(cuuint64_t)inner * (cuuint64_t)elem_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, type, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Allocated on a stream's first use (outside stream capture), counters zeroed
// on that stream; every launch leaves them zero.
bool scratch(cudaStream_t s, Scratch* out) {
    static std::mutex mu;
    static std::map<std::pair<int, cudaStream_t>, Scratch> table;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> g(mu);
    auto it = table.find({dev, s});
    if (it != table.end()) {
        *out = it->second;
        return true;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return false;
    }
    Scratch t;
    if (cudaMalloc(&t.part, (size_t)2 * kMaxCtas * kPiece * sizeof(float)) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (cudaMalloc(&t.count, (size_t)kMaxTiles * sizeof(unsigned)) != cudaSuccess ||
        cudaMemsetAsync(t.count, 0, (size_t)kMaxTiles * sizeof(unsigned), s) != cudaSuccess) {
        cudaFree(t.part);
        if (t.count) cudaFree(t.count);
        cudaGetLastError();
        return false;
    }
    table[{dev, s}] = t;
    *out = t;
    return true;
}

cudaError_t smem_attr_once(const void* fn, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, size_t> done;  // the largest opt-in set so far
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> g(mu);
    auto it = done.find({dev, fn});
    if (it != done.end() && it->second >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) done[{dev, fn}] = smem;
    return e;
}

}  // namespace tc

namespace {

template <bool BF16>
const void* tc_kernel(int stages, int nb) {
    if (nb == 2) {
        switch (stages) {
            case 4: return reinterpret_cast<const void*>(k_gemv_tc<BF16, 4, 2>);
            case 6: return reinterpret_cast<const void*>(k_gemv_tc<BF16, 6, 2>);
            default: return reinterpret_cast<const void*>(k_gemv_tc<BF16, 3, 2>);
        }
    }
    switch (stages) {
        case 8: return reinterpret_cast<const void*>(k_gemv_tc<BF16, 8, 1>);
        case 12: return reinterpret_cast<const void*>(k_gemv_tc<BF16, 12, 1>);
        default: return reinterpret_cast<const void*>(k_gemv_tc<BF16, 6, 1>);
    }
}

}  // namespace

bool gemv_tc_supported(const GemvParams& p) {
    if (p.a.M < 1 || p.a.M > kTcTok || p.a.K % 8 || !have_encoder()) return false;
    if (reinterpret_cast<uintptr_t>(p.a.x) & 15) return false;
    int tiles = 0;
    for (int g = 0; g < p.t.nseg; ++g) {
        if (reinterpret_cast<uintptr_t>(p.t.seg[g].W) & 15) return false;
        tiles += (p.t.seg[g].rows + kTcRows - 1) / kTcRows;
    }
    return tiles <= kMaxTiles && p.t.nseg <= kMaxSeg && !p.t.pair && !p.t.res;
}

size_t gemv_tc_smem() { return tc_smem(6, 1); }

cudaError_t gemv_tc(const GemvParams& gp, bool bf16, unsigned spin, int grid_req, int stages,
                    int nb, int prefetch, cudaStream_t s, bool* launched) {
    *launched = false;
    Scratch scr;
    if (!scratch(s, &scr)) return cudaSuccess;
    TcParams p;
    memset(&p, 0, sizeof p);
    const int K = gp.a.K;
    p.nseg = gp.t.nseg;
    p.M = gp.a.M;
    if (nb != 2) nb = 1;
    p.nkb = (K + nb * kTcBK - 1) / (nb * kTcBK);
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    int tiles = 0;
    for (int g = 0; g < p.nseg; ++g) {
        const Segment& sg = gp.t.seg[g];
        if (!encode_2d(&p.wmap[g], sg.W, dt, 2, K, sg.rows, kTcBK, kTcRows, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaSuccess;
        p.y[g] = sg.y;
        p.rows[g] = sg.rows;
        p.tile_begin[g] = tiles;
        tiles += (sg.rows + kTcRows - 1) / kTcRows;
    }
    p.tile_begin[p.nseg] = tiles;
    if (!encode_2d(&p.xmap, gp.a.x, dt, 2, K, gp.a.M, kTcBK, kTcTok, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaSuccess;
    p.total = (long long)tiles * p.nkb;
    p.part = scr.part;
    p.count = scr.count;
    p.err = device_error_word();
    p.spin = spin;
    p.prefetch = prefetch;
    if (!p.err) return cudaSuccess;
    long long grid = grid_req > 0 ? grid_req : sm_count();
    if (grid > kTcMaxCtas) grid = kTcMaxCtas;
    if (grid > p.total) grid = p.total;
    if (grid < 1) grid = 1;
    if (nb == 2 ? (stages != 4 && stages != 6) : (stages != 8 && stages != 12)) stages = nb == 2 ? 3 : 6;
    const void* fn = bf16 ? tc_kernel<true>(stages, nb) : tc_kernel<false>(stages, nb);
    const size_t smem = tc_smem(stages, nb);
    cudaError_t e = smem_attr_once(fn, smem);
    if (e != cudaSuccess) return e;
    void* args[] = {&p};
    e = launch_pdl(fn, dim3((unsigned)grid), dim3(kTcThreads), smem, s, args);
    if (e == cudaSuccess) *launched = true;
    return e;
}

}  // namespace dg
