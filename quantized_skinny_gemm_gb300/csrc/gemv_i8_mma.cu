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

    // activations are read from global memory through L1 (every warp of an
    // SM reads the same 16 x K codes); tokens >= M read as zeros
    int* part = reinterpret_cast<int*>(smem);  // [warp][8][32]
    const unsigned char* xg = reinterpret_cast<const unsigned char*>(p.a.xq);

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
        const unsigned char* xlo = xg + (size_t)g * K + k0;        // token g
        const unsigned char* xhi = xg + (size_t)(g + 8) * K + k0;  // token g + 8
        const bool has_lo = g < M, has_hi = g + 8 < M;
        int d0[4] = {0, 0, 0, 0}, d1[4] = {0, 0, 0, 0};  // tokens 0..7, 8..15

        for (int kb = 0; active && kb < nblk; kb += kMmaUnroll) {
            uint4 alo[kMmaUnroll], ahi[kMmaUnroll], blv[kMmaUnroll], bhv[kMmaUnroll];
#pragma unroll
            for (int u = 0; u < kMmaUnroll; ++u)
                if (kb + u < nblk) {
                    alo[u] = ld_stream16(wlo + (size_t)(kb + u) * 64);
                    ahi[u] = ld_stream16(whi + (size_t)(kb + u) * 64);
                    blv[u] = has_lo ? ld_nc16(xlo + (size_t)(kb + u) * 64) : make_uint4(0, 0, 0, 0);
                    bhv[u] = has_hi ? ld_nc16(xhi + (size_t)(kb + u) * 64) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
            for (int u = 0; u < kMmaUnroll; ++u)
                if (kb + u < nblk) {
                    const uint4 bl = blv[u], bh = bhv[u];
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

// ---- the same tile on the fp16 tensor path, exactly -------------------------
// int8 values are exact in fp16 (|v| <= 128), their products exact in fp32,
// and integer sums stay exact in fp32 while they are below 2^24: the MMA
// accumulates at most 512 k per thread-slice (|sum| <= 512 * 128 * 128 =
// 2^23) before the fp32 fragment is converted to int32 (exact) and added to
// int32 accumulators.  acc_out therefore stays bit-exact.  Each code v is
// widened with one PRMT into the fp16 pattern of 1024 + (v + 128) (the byte
// XOR 0x80 gives v + 128) and one HSUB2 of 1152, both exact.  Thread
// (g, t)'s 16 bytes of a row at k0 + 16t feed k16 step s (s = 0..3) with
// bytes 16t + 4s .. 16t + 4s + 3: logical k 2t, 2t+1 <- bytes +0, +1 and
// 2t+8, 2t+9 <- bytes +2, +3, the activations mapped the same way.

__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t biased, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(biased), "r"(0x64646464u), "r"(sel));
    return h2_as_u32(__hsub2(u32_as_h2(r), __floats2half2_rn(1152.f, 1152.f)));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kF16FlushBlocks = 8;  // 64-wide k blocks between int32 flushes (512 k)

__global__ void __launch_bounds__(kThreads) k_w8a8_mma_f16(const __grid_constant__ GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int K = p.a.K, M = p.a.M;
    const int ks = p.ksplit;
    const int tiles_per_cta = kWarps / ks;
    const int kw = warp % ks, slot = warp / ks;

    griddep_launch_dependents();
    griddep_wait();

    // activations are read from global memory through L1 (every warp of an
    // SM reads the same 16 x K codes); tokens >= M read as zeros
    int* part = reinterpret_cast<int*>(smem);  // [warp][8][32]
    const unsigned char* xg = reinterpret_cast<const unsigned char*>(p.a.xq);

    const int n_tiles = (p.t.N + 15) / 16;
    const int nblk = K / 64 / ks;
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
        const unsigned char* xlo = xg + (size_t)g * K + k0;
        const unsigned char* xhi = xg + (size_t)(g + 8) * K + k0;
        const bool has_lo = g < M, has_hi = g + 8 < M;
        int i0[4] = {0, 0, 0, 0}, i1[4] = {0, 0, 0, 0};  // tokens 0..7, 8..15

        for (int kb0 = 0; active && kb0 < nblk; kb0 += kF16FlushBlocks) {
            float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
            const int kb1 = min(nblk, kb0 + kF16FlushBlocks);
            for (int kb = kb0; kb < kb1; kb += kMmaUnroll) {
                uint4 alo[kMmaUnroll], ahi[kMmaUnroll], blv[kMmaUnroll], bhv[kMmaUnroll];
#pragma unroll
                for (int u = 0; u < kMmaUnroll; ++u)
                    if (kb + u < kb1) {
                        alo[u] = ld_stream16(wlo + (size_t)(kb + u) * 64);
                        ahi[u] = ld_stream16(whi + (size_t)(kb + u) * 64);
                        blv[u] = has_lo ? ld_nc16(xlo + (size_t)(kb + u) * 64) : make_uint4(0, 0, 0, 0);
                        bhv[u] = has_hi ? ld_nc16(xhi + (size_t)(kb + u) * 64) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                for (int u = 0; u < kMmaUnroll; ++u)
                    if (kb + u < kb1) {
                        const uint4 bl = blv[u], bh = bhv[u];
                        const uint32_t wl[4] = {alo[u].x, alo[u].y, alo[u].z, alo[u].w};
                        const uint32_t wh[4] = {ahi[u].x, ahi[u].y, ahi[u].z, ahi[u].w};
                        const uint32_t xl[4] = {bl.x, bl.y, bl.z, bl.w};
                        const uint32_t xh[4] = {bh.x, bh.y, bh.z, bh.w};
#pragma unroll
                        for (int st = 0; st < 4; ++st) {
                            const uint32_t ql = wl[st] ^ 0x80808080u, qh = wh[st] ^ 0x80808080u;
                            const uint32_t a0 = i8x2_to_f16x2(ql, 0x4140u), a1 = i8x2_to_f16x2(ql, 0x4342u);
                            const uint32_t a2 = i8x2_to_f16x2(qh, 0x4140u), a3 = i8x2_to_f16x2(qh, 0x4342u);
                            const uint32_t yl = xl[st] ^ 0x80808080u, yh = xh[st] ^ 0x80808080u;
                            mma_f16_16816(d0, a0, a2, a1, a3, i8x2_to_f16x2(yl, 0x4140u),
                                          i8x2_to_f16x2(yl, 0x4342u));
                            mma_f16_16816(d1, a0, a2, a1, a3, i8x2_to_f16x2(yh, 0x4140u),
                                          i8x2_to_f16x2(yh, 0x4342u));
                        }
                    }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // exact: integers below 2^24
                i0[j] += __float2int_rn(d0[j]);
                i1[j] += __float2int_rn(d1[j]);
            }
        }
        if (ks > 1) {  // slices 1..ks-1 hand their tiles to slice 0 of the slot
            int* mine = part + (size_t)warp * 8 * 32;
            if (kw != 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    mine[j * 32 + lane] = i0[j];
                    mine[(4 + j) * 32 + lane] = i1[j];
                }
            }
            asm volatile("bar.sync %0, %1;" ::"r"(1 + slot), "r"(ks * 32) : "memory");
            if (kw == 0)
                for (int w = 1; w < ks; ++w) {
                    const int* o = part + (size_t)(warp + w) * 8 * 32;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        i0[j] += o[j * 32 + lane];
                        i1[j] += o[(4 + j) * 32 + lane];
                    }
                }
            asm volatile("bar.sync %0, %1;" ::"r"(1 + slot), "r"(ks * 32) : "memory");
        }
        if (kw != 0 || !active) continue;
        const int tok[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
        const int val_lo[4] = {i0[0], i0[1], i1[0], i1[1]};
        const int val_hi[4] = {i0[2], i0[3], i1[2], i1[3]};
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

size_t gemv_i8_mma_smem(int) { return (size_t)kWarps * 8 * 32 * 4; }

// f16: the fp16 tensor path (exact as above); else the int8 one.
cudaError_t gemv_i8_mma(const GemvParams* p, int K, int grid, cudaStream_t s, int* occ, bool f16) {
    const size_t smem = gemv_i8_mma_smem(K);
    const void* fn = f16 ? reinterpret_cast<const void*>(k_w8a8_mma_f16)
                         : reinterpret_cast<const void*>(k_w8a8_mma);
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
