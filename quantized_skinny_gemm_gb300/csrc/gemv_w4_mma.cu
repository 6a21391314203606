// Groupwise int4 weights for 8..16 tokens (draft / verify blocks) on the
// tensor cores.  With M >= 8 the skinny product is a real dense contraction:
// 16 tokens share every weight byte.  mma.sync m16n8k16 takes fp16 operands
// and accumulates in fp32: the int4 codes are unpacked exactly to fp16 (the
// same nibble-in-mantissa arithmetic as the CUDA-core path), the activations
// are fp16 (W4A16) or int8 codes widened exactly to fp16 (W4A8).
//
// One warp owns 16 weight rows and all 16 (zero-padded) tokens.  Per 32-code
// block (one scale group, or a part of one), quad thread t holds the block's
// codes 8t .. 8t + 7 of rows g and g + 8 (one 32-bit word each), unpacked
// into the pairs (c_j, c_j+4); k16 step s takes pairs 2s and 2s + 1, and the
// activations sit in shared memory as the matching pairs (x_j, x_j+4), so the
// B fragments are read as they lie.  The MMAs of a block start from zero and
// its partial sums are scaled by the block's group scale in fp32: every
// product is exact, and for W4A8 the integer sum of a block (at most
// 32 * 8 * 127 < 2^24) is exact in fp32 as well.  K is split over ks warps of
// a CTA by a rule on K alone (fp32 partials added in warp order), so a row's
// result does not depend on N or on the row's offset.  A CTA runs 16 warps
// and each thread keeps 8 blocks' words of both its rows in flight, so an SM
// has about 32 KB of weight loads outstanding.
#include "gemv_core.cuh"

namespace dg {

namespace {

__device__ __forceinline__ void mma_f16_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ void mma_f16_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t ld_word(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

constexpr int kW4MmaUnroll = 8;  // 32-code blocks loaded ahead (two words each)

// int8 code pair -> fp16 pair (exact)
__device__ __forceinline__ uint32_t i8pair_to_h2(int a, int b) {
    return h2_as_u32(__floats2half2_rn((float)a, (float)b));
}

}  // namespace

// A8: activations are int8 codes (p.a.xq) with per-token scales; else fp16 (p.a.x).
template <bool A8>
__global__ void __launch_bounds__(kW4MmaWarps * 32) k_w4_mma(const __grid_constant__ GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int K = p.a.K, M = p.a.M;
    const int ks = p.ksplit;
    const int tiles_per_cta = kW4MmaWarps / ks;
    const int kw = warp % ks, slot = warp / ks;
    const int cpg = p.group / 32, cps = log2_or_neg(cpg), gk = K / p.group;

    griddep_launch_dependents();
    griddep_wait();

    // activations: 16 tokens x K values as fp16 pairs (x_j, x_j+4) per block
    // of eight, tokens >= M zero; rows padded by 64 bytes (the 8 quads of a
    // warp read different banks)
    const size_t xstride = (size_t)K * 2 + 64;
    {
        const int per_row = K / 8;
        for (int i = threadIdx.x; i < 16 * per_row; i += blockDim.x) {
            const int m = i / per_row, b = i - m * per_row;
            uint4 o = make_uint4(0, 0, 0, 0);
            if (m < M) {
                if constexpr (A8) {
                    const uint2 v = reinterpret_cast<const uint2*>(p.a.xq)[(size_t)m * per_row + b];
                    const int8_t* c = reinterpret_cast<const int8_t*>(&v);
                    o = make_uint4(i8pair_to_h2(c[0], c[4]), i8pair_to_h2(c[1], c[5]),
                                   i8pair_to_h2(c[2], c[6]), i8pair_to_h2(c[3], c[7]));
                } else {
                    const uint4 v = static_cast<const uint4*>(p.a.x)[(size_t)m * per_row + b];
                    o = make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                                   __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
                }
            }
            *reinterpret_cast<uint4*>(smem + (size_t)m * xstride + 16 * b) = o;
        }
    }
    float* part = reinterpret_cast<float*>(smem + 16 * xstride);  // [warp][8][32]
    __syncthreads();

    const int n_tiles = (p.t.N + 15) / 16;
    const int nblk = K / 32 / ks;  // 32-code blocks per warp
    const int groups = (n_tiles + tiles_per_cta - 1) / tiles_per_cta;
    for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        const int tile = grp * tiles_per_cta + slot;
        const bool active = tile < n_tiles;
        const int r0 = (active ? tile : 0) * 16;
        RowRef z{};
        const RowRef first = locate(p.t, r0, (size_t)K / 2, z);
        const RowRef rlo = locate(p.t, r0 + g, (size_t)K / 2, first);
        const RowRef rhi = locate(p.t, r0 + g + 8, (size_t)K / 2, first);
        const RowRef& alo_row = rlo.valid ? rlo : first;
        const RowRef& ahi_row = rhi.valid ? rhi : first;
        const int kb0 = kw * nblk;
        const unsigned char* wlo = alo_row.w + (size_t)kb0 * 16 + 4 * t;
        const unsigned char* whi = ahi_row.w + (size_t)kb0 * 16 + 4 * t;
        const uint16_t* slo = static_cast<const uint16_t*>(alo_row.scale) + (size_t)alo_row.local * gk;
        const uint16_t* shi = static_cast<const uint16_t*>(ahi_row.scale) + (size_t)ahi_row.local * gk;
        const unsigned char* xlo = smem + (size_t)g * xstride + ((size_t)kb0 * 4 + t) * 16;
        const unsigned char* xhi = smem + (size_t)(g + 8) * xstride + ((size_t)kb0 * 4 + t) * 16;
        // one scale per block (groups of 32) and 16-byte aligned runs of eight:
        // scales arrive as one vector per row and batch
        const bool vec_scales = cpg == 1 && (gk % 8) == 0 && (kb0 % 8) == 0 &&
                                ((reinterpret_cast<uintptr_t>(alo_row.scale) |
                                  reinterpret_cast<uintptr_t>(ahi_row.scale)) & 15) == 0;
        // y[row g / g+8][token 2t, 2t+1, 8+2t, 9+2t]
        float ylo[4] = {0.f, 0.f, 0.f, 0.f}, yhi[4] = {0.f, 0.f, 0.f, 0.f};

        for (int kb = 0; active && kb < nblk; kb += kW4MmaUnroll) {
            uint32_t wl[kW4MmaUnroll], wh[kW4MmaUnroll];
            uint16_t sl16[kW4MmaUnroll], sh16[kW4MmaUnroll];
#pragma unroll
            for (int u = 0; u < kW4MmaUnroll; ++u)
                if (kb + u < nblk) {
                    wl[u] = ld_word(wlo + (size_t)(kb + u) * 16);
                    wh[u] = ld_word(whi + (size_t)(kb + u) * 16);
                }
            if (vec_scales && kb + kW4MmaUnroll <= nblk) {
                // one scale per block, eight consecutive ones: one 16-byte load per row
                const uint4 a = *reinterpret_cast<const uint4*>(slo + kb0 + kb);
                const uint4 b = *reinterpret_cast<const uint4*>(shi + kb0 + kb);
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int u = 0; u < kW4MmaUnroll; ++u) {
                    sl16[u] = (u & 1) ? hi16(aw[u >> 1]) : lo16(aw[u >> 1]);
                    sh16[u] = (u & 1) ? hi16(bw[u >> 1]) : lo16(bw[u >> 1]);
                }
            } else {
#pragma unroll
                for (int u = 0; u < kW4MmaUnroll; ++u)
                    if (kb + u < nblk) {
                        const int sg = group_of_chunk(kb0 + kb + u, cpg, cps);
                        sl16[u] = ld_stream_u16(slo + sg);
                        sh16[u] = ld_stream_u16(shi + sg);
                    }
            }
#pragma unroll
            for (int u = 0; u < kW4MmaUnroll; ++u)
                if (kb + u < nblk) {
                    uint32_t ql[4], qh[4];
                    unpack_int4x8_f16(wl[u], ql);
                    unpack_int4x8_f16(wh[u], qh);
                    const uint4 bl = *reinterpret_cast<const uint4*>(xlo + (size_t)(kb + u) * 64);
                    const uint4 bh = *reinterpret_cast<const uint4*>(xhi + (size_t)(kb + u) * 64);
                    float d0[4], d1[4];  // tokens 0..7, 8..15
                    mma_f16_zero(d0, ql[0], qh[0], ql[1], qh[1], bl.x, bl.y);
                    mma_f16_zero(d1, ql[0], qh[0], ql[1], qh[1], bh.x, bh.y);
                    mma_f16_acc(d0, ql[2], qh[2], ql[3], qh[3], bl.z, bl.w);
                    mma_f16_acc(d1, ql[2], qh[2], ql[3], qh[3], bh.z, bh.w);
                    const float sl = __half2float(__ushort_as_half(sl16[u]));
                    const float sh = __half2float(__ushort_as_half(sh16[u]));
                    ylo[0] = fmaf(d0[0], sl, ylo[0]);
                    ylo[1] = fmaf(d0[1], sl, ylo[1]);
                    ylo[2] = fmaf(d1[0], sl, ylo[2]);
                    ylo[3] = fmaf(d1[1], sl, ylo[3]);
                    yhi[0] = fmaf(d0[2], sh, yhi[0]);
                    yhi[1] = fmaf(d0[3], sh, yhi[1]);
                    yhi[2] = fmaf(d1[2], sh, yhi[2]);
                    yhi[3] = fmaf(d1[3], sh, yhi[3]);
                }
        }
        if (ks > 1) {  // slices 1..ks-1 hand their sums to slice 0 of the slot
            float* mine = part + (size_t)warp * 8 * 32;
            if (kw != 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    mine[j * 32 + lane] = ylo[j];
                    mine[(4 + j) * 32 + lane] = yhi[j];
                }
            }
            asm volatile("bar.sync %0, %1;" ::"r"(1 + slot), "r"(ks * 32) : "memory");
            if (kw == 0)
                for (int w = 1; w < ks; ++w) {
                    const float* o = part + (size_t)(warp + w) * 8 * 32;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        ylo[j] += o[j * 32 + lane];
                        yhi[j] += o[(4 + j) * 32 + lane];
                    }
                }
            asm volatile("bar.sync %0, %1;" ::"r"(1 + slot), "r"(ks * 32) : "memory");
        }
        if (kw != 0 || !active) continue;
        const int tok[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = tok[j];
            if (m >= M) continue;
            const float sx = A8 ? __ldg(p.a.x_scale + m) : 1.f;
            if (rlo.valid) write_out<false>(rlo, m, A8 ? sx * ylo[j] : ylo[j]);
            if (rhi.valid) write_out<false>(rhi, m, A8 ? sx * yhi[j] : yhi[j]);
        }
    }
}

size_t gemv_w4_mma_smem(int K) {
    return (size_t)16 * ((size_t)K * 2 + 64) + (size_t)kW4MmaWarps * 8 * 32 * 4;
}

cudaError_t gemv_w4_mma(const GemvParams* p, bool a8, int K, int grid, cudaStream_t s, int* occ) {
    const size_t smem = gemv_w4_mma_smem(K);
    const void* fn = a8 ? reinterpret_cast<const void*>(k_w4_mma<true>)
                        : reinterpret_cast<const void*>(k_w4_mma<false>);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, kW4MmaWarps * 32, smem);
    void* args[] = {const_cast<GemvParams*>(p)};
    return launch_pdl(fn, dim3(grid), dim3(kW4MmaWarps * 32), smem, s, args);
}

}  // namespace dg
