// W8A8 for 8..16 tokens (draft / verify blocks) on the tensor cores.
//
// With M >= 8 the skinny product is a real dense contraction: 16 tokens share
// every weight byte.  The integer tensor-core instruction available on sm_103a
// is the warp-level mma.sync m16n8k32 s8 x s8 -> s32 (tcgen05 has no int8 kind
// on this target), and its int32 accumulation is exact, so acc_out stays
// bit-exact.
//
// One warp owns a tile of 16 weight rows and all 16 (zero-padded) tokens:
// D[16 rows][16 tokens] = W[16][K] x[16][K]^T as two n8 halves.  Each 64-wide
// k block is two k32 MMA steps.  Thread (g = lane/4, t = lane%4) loads the 16
// bytes of rows g and g+8 at k0 + 16t; word i of those bytes feeds MMA step
// i/2: the MMA's logical k (4t..4t+3, 16+4t..16+4t+3) maps to physical
// k0 + 16t + 8(i/2) + (0..7), the same map is used for the activations, and an
// integer dot product does not depend on the order of k.  Every physical k of
// the block is used exactly once.
#include <climits>

#include "gemv_core.cuh"

namespace dg {

__device__ __forceinline__ void mma_s8_16816_32(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kMmaUnroll = 4;  // 64-wide k blocks loaded ahead

// p.a.xq: int8 [M][K], M <= 16; K a multiple of 64 * ks.  A CTA's 8 warps
// take 8 / ks tiles, ks warps per tile, each warp a contiguous 1/ks of K; the
// slices' int32 tiles are added in shared memory (exact in any order).
// Grid-stride over tile groups.
__global__ void __launch_bounds__(kThreads) k_w8a8_mma(const __grid_constant__ GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int K = p.a.K, M = p.a.M;
    const int ks = p.ksplit;
    const int tiles_per_cta = kWarps / ks;
    const int kw = warp % ks, slot = warp / ks;

    griddep_launch_dependents();
    griddep_wait();

    // activations: 16 tokens x K int8 (tokens >= M zero), rows padded by 64
    // bytes so the 8 quads of a warp read from different banks
    const int xstride = K + 64;
    {
        const int per_row = K / 16;
        const uint4* src = reinterpret_cast<const uint4*>(p.a.xq);
        for (int i = threadIdx.x; i < 16 * per_row; i += blockDim.x) {
            const int m = i / per_row, c = i - m * per_row;
            *reinterpret_cast<uint4*>(smem + (size_t)m * xstride + 16 * c) =
                m < M ? src[i] : make_uint4(0, 0, 0, 0);
        }
    }
    int* part = reinterpret_cast<int*>(smem + (size_t)16 * xstride);  // [warp][8][32]
    __syncthreads();

    const int n_tiles = (p.t.N + 15) / 16;
    const int nblk = K / 64 / ks;  // 64-wide k blocks per warp
    const int groups = (n_tiles + tiles_per_cta - 1) / tiles_per_cta;
    for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        const int tile = grp * tiles_per_cta + slot;
        const bool active = tile < n_tiles;
        const int r0 = (active ? tile : 0) * 16;
        RowRef z{};
        const RowRef first = locate(p.t, r0, (size_t)K, z);
        RowRef rlo = locate(p.t, r0 + g, (size_t)K, first);
        RowRef rhi = locate(p.t, r0 + g + 8, (size_t)K, first);
        const size_t k0 = (size_t)kw * nblk * 64 + 16 * t;
        const unsigned char* wlo = (rlo.valid ? rlo.w : first.w) + k0;
        const unsigned char* whi = (rhi.valid ? rhi.w : first.w) + k0;
        const unsigned char* xlo = smem + (size_t)g * xstride + k0;        // token g
        const unsigned char* xhi = smem + (size_t)(g + 8) * xstride + k0;  // token g + 8
        int d0[4] = {0, 0, 0, 0}, d1[4] = {0, 0, 0, 0};  // tokens 0..7, 8..15

        for (int kb = 0; active && kb < nblk; kb += kMmaUnroll) {
            uint4 alo[kMmaUnroll], ahi[kMmaUnroll];
#pragma unroll
            for (int u = 0; u < kMmaUnroll; ++u)
                if (kb + u < nblk) {
                    alo[u] = ld_stream16(wlo + (size_t)(kb + u) * 64);
                    ahi[u] = ld_stream16(whi + (size_t)(kb + u) * 64);
                }
#pragma unroll
            for (int u = 0; u < kMmaUnroll; ++u)
                if (kb + u < nblk) {
                    const uint4 bl = *reinterpret_cast<const uint4*>(xlo + (size_t)(kb + u) * 64);
                    const uint4 bh = *reinterpret_cast<const uint4*>(xhi + (size_t)(kb + u) * 64);
                    mma_s8_16816_32(d0, alo[u].x, ahi[u].x, alo[u].y, ahi[u].y, bl.x, bl.y);
                    mma_s8_16816_32(d1, alo[u].x, ahi[u].x, alo[u].y, ahi[u].y, bh.x, bh.y);
                    mma_s8_16816_32(d0, alo[u].z, ahi[u].z, alo[u].w, ahi[u].w, bl.z, bl.w);
                    mma_s8_16816_32(d1, alo[u].z, ahi[u].z, alo[u].w, ahi[u].w, bh.z, bh.w);
                }
        }
        if (ks > 1) {  // slices 1..ks-1 hand their tiles to slice 0 of the slot
            int* mine = part + (size_t)warp * 8 * 32;
            if (kw != 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    mine[j * 32 + lane] = d0[j];
                    mine[(4 + j) * 32 + lane] = d1[j];
                }
            }
            asm volatile("bar.sync %0, %1;" ::"r"(1 + slot), "r"(ks * 32) : "memory");
            if (kw == 0)
                for (int w = 1; w < ks; ++w) {
                    const int* o = part + (size_t)(warp + w) * 8 * 32;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        d0[j] += o[j * 32 + lane];
                        d1[j] += o[(4 + j) * 32 + lane];
                    }
                }
            asm volatile("bar.sync %0, %1;" ::"r"(1 + slot), "r"(ks * 32) : "memory");
        }
        if (kw != 0 || !active) continue;
        // d[0], d[1]: row g, tokens 2t, 2t+1 (+8 for d1); d[2], d[3]: row g + 8
        const int tok[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
        const int val_lo[4] = {d0[0], d0[1], d1[0], d1[1]};
        const int val_hi[4] = {d0[2], d0[3], d1[2], d1[3]};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = tok[j];
            if (m >= M) continue;
            const float sx = __ldg(p.a.x_scale + m);
            if (rlo.valid) PolicyI8::store(rlo, m, val_lo[j], sx);
            if (rhi.valid) PolicyI8::store(rhi, m, val_hi[j], sx);
        }
    }
}

size_t gemv_i8_mma_smem(int K) { return (size_t)16 * (K + 64) + (size_t)kWarps * 8 * 32 * 4; }

cudaError_t gemv_i8_mma(const GemvParams* p, int K, int grid, cudaStream_t s, int* occ) {
    const size_t smem = gemv_i8_mma_smem(K);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_w8a8_mma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k_w8a8_mma, kThreads, smem);
    void* args[] = {const_cast<GemvParams*>(p)};
    return launch_pdl(reinterpret_cast<const void*>(k_w8a8_mma), dim3(grid), dim3(kThreads), smem,
                      s, args);
}

}  // namespace dg
