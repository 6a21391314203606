// fp16 / bf16 weights for 8..16 tokens (draft / verify blocks) on the tensor
// cores.  With M >= 8 the skinny product is a real dense contraction: 16
// tokens share every weight byte.  mma.sync m16n8k16 takes the fp16 / bf16
// operands as they are and accumulates in fp32.
//
// One warp owns a tile of 16 weight rows and all 16 (zero-padded) tokens:
// D[16 rows][16 tokens] = W[16][K] x[16][K]^T as two n8 halves; the tokens'
// values are read from global memory through L1 (no staging, so two CTAs fit
// an SM and K is unbounded).  Thread
// (g = lane/4, t = lane%4) loads 16 bytes (8 values) of rows g and g+8 at
// k0 + 8t of each 32-wide k block; k16 step s (s = 0, 1) takes values
// 8t + 4s .. 8t + 4s + 3: logical k 2t, 2t+1 <- +0, +1 and 2t+8, 2t+9 <- +2,
// +3, the activations mapped the same way (a dot product does not depend on
// the order of k, and the map covers every k of the block once).  K is split
// over ks warps of a CTA (fp32 partials added in warp order); ks follows K
// alone, so a row's result does not depend on N or on the row's offset.
#include "gemv_core.cuh"

namespace dg {

namespace {

template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    if (BF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kFpMmaUnroll = 4;  // 32-wide k blocks loaded ahead

}  // namespace

// p.a.x: fp16 / bf16 [M][K], 8 <= M <= 16; K a multiple of 32 * ks.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) k_fp_mma(const __grid_constant__ GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    using P = PolicyFP<BF16>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int K = p.a.K, M = p.a.M;
    const int ks = p.ksplit;
    const int tiles_per_cta = kWarps / ks;
    const int kw = warp % ks, slot = warp / ks;

    griddep_launch_dependents();
    griddep_wait();

    // activations are read from global memory through L1 (every warp of an
    // SM reads the same 16 x K values); tokens >= M read as zeros
    float* part = reinterpret_cast<float*>(smem);  // [warp][8][32]
    const unsigned char* xg = static_cast<const unsigned char*>(p.a.x);

    const int n_tiles = (p.t.N + 15) / 16;
    const int nblk = K / 32 / ks;  // 32-wide k blocks per warp
    const int groups = (n_tiles + tiles_per_cta - 1) / tiles_per_cta;
    for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        const int tile = grp * tiles_per_cta + slot;
        const bool active = tile < n_tiles;
        const int r0 = (active ? tile : 0) * 16;
        RowRef z{};
        const RowRef first = locate(p.t, r0, (size_t)K * 2, z);
        const RowRef rlo = locate(p.t, r0 + g, (size_t)K * 2, first);
        const RowRef rhi = locate(p.t, r0 + g + 8, (size_t)K * 2, first);
        const size_t k0 = ((size_t)kw * nblk * 32 + 8 * t) * 2;  // bytes
        const unsigned char* wlo = (rlo.valid ? rlo.w : first.w) + k0;
        const unsigned char* whi = (rhi.valid ? rhi.w : first.w) + k0;
        const unsigned char* xlo = xg + (size_t)g * K * 2 + k0;        // token g
        const unsigned char* xhi = xg + (size_t)(g + 8) * K * 2 + k0;  // token g + 8
        const bool has_lo = g < M, has_hi = g + 8 < M;
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};  // tokens 0..7, 8..15

        for (int kb = 0; active && kb < nblk; kb += kFpMmaUnroll) {
            uint4 alo[kFpMmaUnroll], ahi[kFpMmaUnroll], blv[kFpMmaUnroll], bhv[kFpMmaUnroll];
#pragma unroll
            for (int u = 0; u < kFpMmaUnroll; ++u)
                if (kb + u < nblk) {
                    alo[u] = ld_stream16(wlo + (size_t)(kb + u) * 64);
                    ahi[u] = ld_stream16(whi + (size_t)(kb + u) * 64);
                    blv[u] = has_lo ? ld_nc16(xlo + (size_t)(kb + u) * 64) : make_uint4(0, 0, 0, 0);
                    bhv[u] = has_hi ? ld_nc16(xhi + (size_t)(kb + u) * 64) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
            for (int u = 0; u < kFpMmaUnroll; ++u)
                if (kb + u < nblk) {
                    const uint4 bl = blv[u], bh = bhv[u];
                    // step 0: values +0..+3 (words x, y); step 1: +4..+7 (z, w)
                    mma_16816<BF16>(d0, alo[u].x, ahi[u].x, alo[u].y, ahi[u].y, bl.x, bl.y);
                    mma_16816<BF16>(d1, alo[u].x, ahi[u].x, alo[u].y, ahi[u].y, bh.x, bh.y);
                    mma_16816<BF16>(d0, alo[u].z, ahi[u].z, alo[u].w, ahi[u].w, bl.z, bl.w);
                    mma_16816<BF16>(d1, alo[u].z, ahi[u].z, alo[u].w, ahi[u].w, bh.z, bh.w);
                }
        }
        if (ks > 1) {  // slices 1..ks-1 hand their tiles to slice 0 of the slot
            float* mine = part + (size_t)warp * 8 * 32;
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
                    const float* o = part + (size_t)(warp + w) * 8 * 32;
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
        const float val_lo[4] = {d0[0], d0[1], d1[0], d1[1]};
        const float val_hi[4] = {d0[2], d0[3], d1[2], d1[3]};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = tok[j];
            if (m >= M) continue;
            if (rlo.valid) P::store(rlo, m, val_lo[j], 1.f);
            if (rhi.valid) P::store(rhi, m, val_hi[j], 1.f);
        }
    }
}

size_t gemv_fp_mma_smem(int) { return (size_t)kWarps * 8 * 32 * 4; }

cudaError_t gemv_fp_mma(const GemvParams* p, bool bf16, int K, int grid, cudaStream_t s, int* occ) {
    const size_t smem = gemv_fp_mma_smem(K);
    const void* fn = bf16 ? reinterpret_cast<const void*>(k_fp_mma<true>)
                          : reinterpret_cast<const void*>(k_fp_mma<false>);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, kThreads, smem);
    void* args[] = {const_cast<GemvParams*>(p)};
    return launch_pdl(fn, dim3(grid), dim3(kThreads), smem, s, args);
}

}  // namespace dg
