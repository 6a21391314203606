// Weight-streaming skinny GEMV: the per-row arithmetic shared by every kernel
// (one policy per weight format), and the per-launch kernel k_gemv.
//
// Work decomposition.  `ksplit` consecutive warps of a CTA form a slot that
// owns one row group of R rows; the slot's warps split the row's 16-byte
// chunks: warp kw of the slot, lane l, visits chunks
//     c_j = (j * ksplit + kw) * 32 + l,   j = 0, 1, ...
// so each warp-wide load reads 512 contiguous bytes of a weight row, and one
// lane accumulates its chunks in ascending j.  Lane sums meet in a fixed
// xor-butterfly, then the slot's warps add in kw order.  The order depends
// only on K and ksplit (which the host picks from K alone), never on N, the
// row's offset, the grid or the kernel (k_gemv or the persistent step kernel),
// so a row slice of W reproduces the full matrix's rows bit for bit (the
// 16-slice lm_head split of the Orange Pi AIPro post holds exactly), and a
// decode step gives bitwise the results of the per-op calls.
//
// Activations are staged once per CTA in shared memory (permuted where the
// int4 unpack wants it); weights bypass L1 and are read with 16-byte vector
// loads, U chunks per lane in flight per row.
#pragma once

#include <climits>
#include <cmath>
#include <type_traits>

#include "dg_internal.cuh"

namespace dg {

// ---- per-row addressing -------------------------------------------------------

struct RowRef {
    const unsigned char* w;   // weight row
    const void* scale;        // segment scale base
    void* y;                  // segment output base
    int32_t* acc_out;
    int local;                // row index inside its segment
    int seg_rows;             // rows of its segment (output row stride)
    int global;               // row index over all segments
    bool valid;
};

__device__ __forceinline__ RowRef locate(const SegTable& t, int r, size_t row_bytes,
                                         const RowRef& fallback) {
    RowRef rr = fallback;
    rr.valid = false;
    if (r >= t.N) return rr;
    int s = 0;
#pragma unroll
    for (int i = 1; i < kMaxSeg; ++i)
        if (i < t.nseg && r >= t.seg[i].row_begin) s = i;
    const Segment& sg = t.seg[s];
    rr.local = r - sg.row_begin;
    rr.w = static_cast<const unsigned char*>(sg.W) + (size_t)rr.local * row_bytes;
    rr.scale = sg.scale;
    rr.y = sg.y;
    rr.acc_out = sg.acc_out;
    rr.seg_rows = sg.rows;
    rr.global = r;
    rr.valid = true;
    return rr;
}

template <typename T>
__device__ __forceinline__ int to_bits(T v);
template <>
__device__ __forceinline__ int to_bits<float>(float v) { return __float_as_int(v); }
template <>
__device__ __forceinline__ int to_bits<int>(int v) { return v; }
template <typename T>
__device__ __forceinline__ T from_bits(int v);
template <>
__device__ __forceinline__ float from_bits<float>(int v) { return __int_as_float(v); }
template <>
__device__ __forceinline__ int from_bits<int>(int v) { return v; }

// ---- format policies ------------------------------------------------------------
// stage_x fills the CTA's activation area from `a`; the int8 policies read
// their codes from `a.xq`, which may point to global or shared memory.

// Two fp16 (or bf16) values of a packed word, converted exactly to fp32.
template <bool BF16>
__device__ __forceinline__ float2 unpack2_f32(uint32_t w) {
    if (BF16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    return __half22float2(u32_as_h2(w));
}

// fp16 / bf16 weights and activations; 8 elements per chunk.  Each product
// of two 11-bit (8-bit) significands is exact in fp32 and one FMA with fp32
// accumulation rounds once, in ascending k.  With one token the activations
// are read straight from global memory (16 bytes per chunk, L1-cached: every
// warp of an SM reads the same vector); with more tokens they are staged in
// shared memory.
template <bool BF16>
struct PolicyFP {
    static constexpr int kElems = 8;
    static constexpr bool kIntAct = false;
    static constexpr bool kDirectX = true;  // M = 1 reads x from global memory
    using Acc = float;
    struct Chunk { uint4 w; };

    __host__ __device__ static size_t row_bytes(int K) { return (size_t)K * 2; }
    __host__ __device__ static size_t x_bytes(int MT, int K) { return (size_t)MT * K * 2; }

    __device__ static void stage_x(const ActIn& a, unsigned char* xs, int MT) {
        const int per_row = a.K / 8;
        const uint4* src = static_cast<const uint4*>(a.x);
        uint4* dst = reinterpret_cast<uint4*>(xs);
        for (int i = threadIdx.x; i < MT * per_row; i += blockDim.x) {
            const int m = i / per_row;
            dst[i] = m < a.M ? src[i] : make_uint4(0, 0, 0, 0);
        }
    }
    __device__ __forceinline__ static void load(Chunk& ch, const RowRef& r, int c, int, int) {
        ch.w = ld_stream16(r.w + (size_t)c * 16);
    }
    __device__ __forceinline__ static float mac2(uint32_t w, uint32_t x, float a) {
        if (BF16) {
            a = fma_bf16(lo16(w), lo16(x), a);
            return fma_bf16(hi16(w), hi16(x), a);
        }
        a = fma_f16(lo16(w), lo16(x), a);
        return fma_f16(hi16(w), hi16(x), a);
    }
    __device__ __forceinline__ static float mac8(const uint4& w, const uint4& xv, float a) {
        a = mac2(w.x, xv.x, a);
        a = mac2(w.y, xv.y, a);
        a = mac2(w.z, xv.z, a);
        return mac2(w.w, xv.w, a);
    }
    template <int MT>
    __device__ __forceinline__ static void mac(Acc (&acc)[MT], const Chunk& ch,
                                               const unsigned char* xs, int c, int K) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
            acc[m] = mac8(ch.w, *reinterpret_cast<const uint4*>(xs + ((size_t)m * K + (size_t)c * 8) * 2),
                          acc[m]);
    }
    // One token, activations from global memory (loaded with the weights,
    // see row_group): the chunk's eight products go into two independent
    // chains of four, merged into the row sum once per chunk.
    __device__ __forceinline__ static uint4 load_x(const void* x, int c, bool coherent) {
        const unsigned char* p = static_cast<const unsigned char*>(x) + (size_t)c * 16;
        return coherent ? ld_cg16(p) : ld_nc16(p);
    }
    __device__ __forceinline__ static void mac_direct(Acc (&acc)[1], const Chunk& ch, const uint4& xv) {
        float s0 = mac2(ch.w.x, xv.x, 0.f);
        float s1 = mac2(ch.w.z, xv.z, 0.f);
        s0 = mac2(ch.w.y, xv.y, s0);
        s1 = mac2(ch.w.w, xv.w, s1);
        acc[0] += s0 + s1;
    }
    __device__ static float finish(const RowRef&, Acc a, float) { return a; }
    __device__ static void store(const RowRef& r, int m, Acc a, float) {
        const size_t o = (size_t)m * r.seg_rows + r.local;
        if (BF16)
            static_cast<__nv_bfloat16*>(r.y)[o] = __float2bfloat16_rn(a);
        else
            static_cast<__half*>(r.y)[o] = __float2half_rn(a);
    }
};

// int8 weights x int8 activations, exact int32 sums; 16 elements per chunk.
struct PolicyI8 {
    static constexpr int kElems = 16;
    static constexpr bool kIntAct = true;
    static constexpr bool kDirectX = false;
    using Acc = int;
    struct Chunk { uint4 w; };

    __host__ __device__ static size_t row_bytes(int K) { return (size_t)K; }
    __host__ __device__ static size_t x_bytes(int MT, int K) { return (size_t)MT * K; }

    __device__ static void stage_x(const ActIn& a, unsigned char* xs, int MT) {
        const int per_row = a.K / 16;
        const uint4* src = reinterpret_cast<const uint4*>(a.xq);
        uint4* dst = reinterpret_cast<uint4*>(xs);
        for (int i = threadIdx.x; i < MT * per_row; i += blockDim.x) {
            const int m = i / per_row;
            dst[i] = m < a.M ? src[i] : make_uint4(0, 0, 0, 0);
        }
    }
    __device__ __forceinline__ static void load(Chunk& ch, const RowRef& r, int c, int, int) {
        ch.w = ld_stream16(r.w + (size_t)c * 16);
    }
    template <int MT>
    __device__ __forceinline__ static void mac(Acc (&acc)[MT], const Chunk& ch,
                                               const unsigned char* xs, int c, int K) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)m * K + (size_t)c * 16);
            int a = acc[m];
            a = dp4a_ss(ch.w.x, xv.x, a);
            a = dp4a_ss(ch.w.y, xv.y, a);
            a = dp4a_ss(ch.w.z, xv.z, a);
            a = dp4a_ss(ch.w.w, xv.w, a);
            acc[m] = a;
        }
    }
    __device__ static float finish(const RowRef& r, Acc a, float sx) {
        const float sw = __ldg(static_cast<const float*>(r.scale) + r.local);
        return (float)a * sw * sx;
    }
    __device__ static void store(const RowRef& r, int m, Acc a, float sx) {
        const size_t o = (size_t)m * r.seg_rows + r.local;
        if (r.acc_out) r.acc_out[o] = a;
        if (r.y) static_cast<__half*>(r.y)[o] = __float2half_rn(finish(r, a, sx));
    }
};

// Unpacks one word of 8 int4 codes (k0..k7: byte j holds k = 2j in bits 0-3
// and k = 2j+1 in bits 4-7) into four fp16 pairs (c0,c4) (c1,c5) (c2,c6)
// (c3,c7), exactly.  A nibble n stands for c = n - 16*(n >= 8), so n ^ 8 =
// c + 8 in [0, 15].  Placing n ^ 8 in the low mantissa bits of the fp16 1024
// gives 1024 + (c + 8); subtracting 1032 leaves c.  For the nibbles in bits
// 4-7 of a half the mantissa holds 16 * (c + 8), so (1024 + 16(c+8)) / 16 - 72
// = c, computed by one fused multiply-add with an exact result.
__device__ __forceinline__ void unpack_int4x8_f16(uint32_t w, uint32_t (&q)[4]) {
    const uint32_t w8 = w >> 8;
    const __half2 k1032 = __floats2half2_rn(1032.f, 1032.f);
    const __half2 k16th = __floats2half2_rn(0.0625f, 0.0625f);
    const __half2 k72 = __floats2half2_rn(-72.f, -72.f);
    q[0] = h2_as_u32(__hsub2(u32_as_h2(and_xor(w, 0x000F000Fu, 0x64086408u)), k1032));
    q[1] = h2_as_u32(__hfma2(u32_as_h2(and_xor(w, 0x00F000F0u, 0x64806480u)), k16th, k72));
    q[2] = h2_as_u32(__hsub2(u32_as_h2(and_xor(w8, 0x000F000Fu, 0x64086408u)), k1032));
    q[3] = h2_as_u32(__hfma2(u32_as_h2(and_xor(w8, 0x00F000F0u, 0x64806480u)), k16th, k72));
}

// Shared-memory layout of int4 activations: chunk c (32 codes) of a token is
// cut into 16-byte pieces, and piece i of chunk c sits at
//     ((c / 32) * pieces + i) * 512 + (c % 32) * 16
// so the 32 lanes of a warp, which always hold chunks with c % 32 = lane,
// read 32 consecutive 16-byte words: no bank conflicts.  A token's area is
// padded to a multiple of 32 chunks.
__host__ __device__ __forceinline__ size_t int4_x_token_bytes(int K, int piece_bytes_per_chunk) {
    const size_t nch = (size_t)(K / 32);
    return ((nch + 31) / 32) * 32 * (size_t)piece_bytes_per_chunk;
}
// Scale group of chunk c when cpg chunks share a scale (no division in the
// common case of one 32-code group per chunk).
__device__ __forceinline__ int group_of_chunk(int c, int cpg) { return cpg == 1 ? c : c / cpg; }

__device__ __forceinline__ size_t int4_x_piece(int c, int i, int pieces) {
    return ((size_t)(c >> 5) * pieces + i) * 512 + (size_t)(c & 31) * 16;
}

// Groupwise int4 weights with fp16 activations; 32 codes per chunk.  Chunk c
// covers codes [32c, 32c + 32) of the row and uses the scale of group c / cpg
// (cpg = group / 32).  Activations are staged as fp16 in the interleaved
// layout, four 16-byte pieces per chunk: piece i holds the pairs (x0,x4)
// (x1,x5) (x2,x6) (x3,x7) of the chunk's i-th block of eight, lined up with the
// unpacked code pairs.  Each code (exact in fp16) meets its activation in one
// mixed-precision FMA (fp16 x fp16 + fp32: the product of a 4-bit code and an
// 11-bit significand is exact, one rounding), in four chains, one per block.
struct PolicyW4A16 {
    static constexpr int kElems = 32;
    static constexpr bool kIntAct = false;
    static constexpr bool kDirectX = false;
    using Acc = float;
    struct Chunk { uint4 w; uint16_t s; };

    __host__ __device__ static size_t row_bytes(int K) { return (size_t)K / 2; }
    __host__ __device__ static size_t token_bytes(int K) { return int4_x_token_bytes(K, 64); }
    __host__ __device__ static size_t x_bytes(int MT, int K) { return (size_t)MT * token_bytes(K); }

    __device__ static void stage_x(const ActIn& a, unsigned char* xs, int MT) {
        const int per_row = a.K / 8;  // 16-byte blocks (8 halves) of one token
        const uint4* src = static_cast<const uint4*>(a.x);
        const size_t tb = token_bytes(a.K);
        for (int i = threadIdx.x; i < MT * per_row; i += blockDim.x) {
            const int m = i / per_row, blk = i - m * per_row;
            const uint4 v = m < a.M ? src[i] : make_uint4(0, 0, 0, 0);
            // v = (x0,x1) (x2,x3) (x4,x5) (x6,x7) -> (x0,x4) (x1,x5) (x2,x6) (x3,x7)
            const uint4 o = make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                                       __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
            // block blk = word blk % 4 of chunk blk / 4
            *reinterpret_cast<uint4*>(xs + m * tb + int4_x_piece(blk >> 2, blk & 3, 4)) = o;
        }
    }
    __device__ __forceinline__ static void load(Chunk& ch, const RowRef& r, int c, int gk, int cpg) {
        ch.w = ld_stream16(r.w + (size_t)c * 16);
        ch.s = ld_stream_u16(static_cast<const uint16_t*>(r.scale) + (size_t)r.local * gk +
                             group_of_chunk(c, cpg));
    }
    template <int MT>
    __device__ __forceinline__ static void mac(Acc (&acc)[MT], const Chunk& ch,
                                               const unsigned char* xs, int c, int K) {
        uint32_t q[4][4];
        unpack_int4x8_f16(ch.w.x, q[0]);
        unpack_int4x8_f16(ch.w.y, q[1]);
        unpack_int4x8_f16(ch.w.z, q[2]);
        unpack_int4x8_f16(ch.w.w, q[3]);
        const float s = __half2float(__ushort_as_half(ch.s));
        const size_t tb = token_bytes(K);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const unsigned char* xb = xs + m * tb;
            float P[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 xp = *reinterpret_cast<const uint4*>(xb + int4_x_piece(c, i, 4));
                const uint32_t xv[4] = {xp.x, xp.y, xp.z, xp.w};
                float a = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {  // (c_j, c_j+4) against (x_j, x_j+4)
                    a = fma_f16(lo16(q[i][j]), lo16(xv[j]), a);
                    a = fma_f16(hi16(q[i][j]), hi16(xv[j]), a);
                }
                P[i] = a;
            }
            acc[m] = fmaf((P[0] + P[1]) + (P[2] + P[3]), s, acc[m]);
        }
    }
    __device__ static float finish(const RowRef&, Acc a, float) { return a; }
    __device__ static void store(const RowRef& r, int m, Acc a, float) {
        static_cast<__half*>(r.y)[(size_t)m * r.seg_rows + r.local] = __float2half_rn(a);
    }
};

// Groupwise int4 weights with int8 activations.  Codes are biased to c + 8 in
// [0, 15] (one LOP3 per four codes) and multiplied with dp4a (unsigned x
// signed); the bias is removed exactly with the chunk's activation sum:
// sum (c+8) x - 8 sum x = sum c x.  Activations use the interleaved layout
// above (two 16-byte pieces per chunk), each 8-byte block ordered
// x0 x2 x4 x6 | x1 x3 x5 x7 (even codes sit in low nibbles), followed by the
// int32 sum of each 32-chunk.
struct PolicyW4A8 {
    static constexpr int kElems = 32;
    static constexpr bool kIntAct = true;
    static constexpr bool kDirectX = false;
    using Acc = float;
    struct Chunk { uint4 w; uint16_t s; };

    __host__ __device__ static size_t row_bytes(int K) { return (size_t)K / 2; }
    __host__ __device__ static size_t token_bytes(int K) { return int4_x_token_bytes(K, 32); }
    __host__ __device__ static size_t x_bytes(int MT, int K) {
        return (size_t)MT * token_bytes(K) + (size_t)MT * (K / 32) * 4;
    }

    __device__ static void stage_x(const ActIn& a, unsigned char* xs, int MT) {
        const int K = a.K;
        const int per_row = K / 8;  // 8-byte blocks of one token
        const uint2* src = reinterpret_cast<const uint2*>(a.xq);
        const size_t tb = token_bytes(K);
        for (int i = threadIdx.x; i < MT * per_row; i += blockDim.x) {
            const int m = i / per_row, blk = i - m * per_row;
            uint2 v = m < a.M ? src[i] : make_uint2(0, 0);
            uint2 o;
            o.x = __byte_perm(v.x, v.y, 0x6420);  // x0 x2 x4 x6
            o.y = __byte_perm(v.x, v.y, 0x7531);  // x1 x3 x5 x7
            // block blk: chunk blk / 4, 16-byte piece (blk % 4) / 2, half blk % 2
            *reinterpret_cast<uint2*>(xs + m * tb + int4_x_piece(blk >> 2, (blk >> 1) & 1, 2) +
                                      (blk & 1) * 8) = o;
        }
        int* xsum = reinterpret_cast<int*>(xs + (size_t)MT * tb);
        const int nch = K / 32;
        const uint4* src16 = reinterpret_cast<const uint4*>(a.xq);
        for (int i = threadIdx.x; i < MT * nch; i += blockDim.x) {
            const int m = i / nch;
            int s = 0;
            if (m < a.M) {
                const uint4 p = src16[2 * i], q = src16[2 * i + 1];
                s = dp4a_ss(p.x, 0x01010101u, s);
                s = dp4a_ss(p.y, 0x01010101u, s);
                s = dp4a_ss(p.z, 0x01010101u, s);
                s = dp4a_ss(p.w, 0x01010101u, s);
                s = dp4a_ss(q.x, 0x01010101u, s);
                s = dp4a_ss(q.y, 0x01010101u, s);
                s = dp4a_ss(q.z, 0x01010101u, s);
                s = dp4a_ss(q.w, 0x01010101u, s);
            }
            xsum[i] = s;
        }
    }
    __device__ __forceinline__ static void load(Chunk& ch, const RowRef& r, int c, int gk, int cpg) {
        ch.w = ld_stream16(r.w + (size_t)c * 16);
        ch.s = ld_stream_u16(static_cast<const uint16_t*>(r.scale) + (size_t)r.local * gk +
                             group_of_chunk(c, cpg));
    }
    template <int MT>
    __device__ __forceinline__ static void mac(Acc (&acc)[MT], const Chunk& ch,
                                               const unsigned char* xs, int c, int K) {
        uint32_t lo[4], hi[4];
        const uint32_t wv[4] = {ch.w.x, ch.w.y, ch.w.z, ch.w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = and_xor(wv[i], 0x0F0F0F0Fu, 0x08080808u);
            hi[i] = and_xor(wv[i] >> 4, 0x0F0F0F0Fu, 0x08080808u);
        }
        const float s = __half2float(__ushort_as_half(ch.s));
        const size_t tb = token_bytes(K);
        const int* xsum = reinterpret_cast<const int*>(xs + (size_t)MT * tb);
        const int nch = K / 32;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const unsigned char* xb = xs + m * tb;
            const uint4 x0 = *reinterpret_cast<const uint4*>(xb + int4_x_piece(c, 0, 2));
            const uint4 x1 = *reinterpret_cast<const uint4*>(xb + int4_x_piece(c, 1, 2));
            int a = -8 * xsum[m * nch + c];
            a = dp4a_us(lo[0], x0.x, a);
            a = dp4a_us(hi[0], x0.y, a);
            a = dp4a_us(lo[1], x0.z, a);
            a = dp4a_us(hi[1], x0.w, a);
            a = dp4a_us(lo[2], x1.x, a);
            a = dp4a_us(hi[2], x1.y, a);
            a = dp4a_us(lo[3], x1.z, a);
            a = dp4a_us(hi[3], x1.w, a);
            acc[m] = fmaf((float)a, s, acc[m]);
        }
    }
    __device__ static float finish(const RowRef&, Acc a, float sx) { return sx * a; }
    __device__ static void store(const RowRef& r, int m, Acc a, float sx) {
        static_cast<__half*>(r.y)[(size_t)m * r.seg_rows + r.local] = __float2half_rn(sx * a);
    }
};

// Named barrier of warp `warp`'s slot when ks = 2, 4 or 8 warps share a row.
// In a persistent kernel warps move through phases independently, so phases
// with different ks can be live at once, and a named barrier must never be
// used with two thread counts at the same time: the splits take disjoint ids,
// ks = 2 from 1 upward (1..8), ks = 8 at 9..10 and ks = 4 from 14 downward
// (14..11), for up to 16 warps; 0 is __syncthreads, 15 the weight ring's
// consumer barrier.
__device__ __forceinline__ int slot_barrier(int warp, int ks) {
    return ks == 4 ? 14 - warp / 4 : ks == 8 ? 9 + warp / 8 : 1 + warp / ks;
}

// ---- W4A16 at one token on the tensor cores ---------------------------------------
//
// On the CUDA cores each int4 weight with an fp16 activation costs about four
// issued instructions (unpack, mixed FMA, activation load, loop), which holds
// the stream far below HBM speed.  mma.sync m16n8k16 (fp16 operands, fp32
// accumulation) takes the products and their sums off the FMA pipe: 16 weight
// rows form the A operand, and the activations a B operand whose column n
// collects chunk n (32 codes) of a 256-code segment, so that D[row][n] is the
// chunk's partial sum; its group scale is applied afterwards in fp32.
//
// Thread (g = lane / 4, t = lane % 4) streams rows g and g + 8 of the tile
// and, of every segment, chunks t and t + 4 (so one warp-wide copy reads 64
// contiguous bytes of each of 8 rows).  In each of a segment's 16 MMAs its k
// values 2t, 2t+1 are a code pair (c_j, c_j+4) of chunk t and its k values
// 2t+8, 2t+9 the same pair of chunk t + 4 (the pairs unpack_int4x8_f16
// yields).  Column n of B is then non-zero only in thread (g = n, t = n % 4),
// fragment b0 for n < 4 and b1 for n >= 4, which holds the activations of that
// pair in the interleaved layout; every other thread feeds zeros.  Thread
// (g, t) finds D[g][2t], D[g][2t+1], D[g+8][2t], D[g+8][2t+1] in its
// accumulator: the partials of chunks 2t and 2t + 1 of rows g and g + 8.  A
// 4-bit code times an fp16 activation is exact; four independent MMA chains
// (one per code pair) sum a chunk and are added in a fixed order; the lane
// adds its scaled chunks in ascending order; a fixed xor butterfly joins the
// quad.  The order follows K alone, never the row's place in the
// tile, N or the grid.
//
// The host takes this path only on request: on the int4 decoder it measured
// slower than the CUDA-core policy (PolicyW4A16) in every variant tried.
//
// Weights travel through a per-warp ring of kW4MmaStages segments in shared
// memory, filled with cp.async kW4MmaStages - 1 segments ahead of use, so the
// bytes in flight do not occupy registers.  Each thread reads back only the
// 16-byte slots it copied itself: the copies' own completion (wait_group) is
// the only ordering needed, and nothing waits on another thread.

__device__ __forceinline__ void mma_m16n8k16_f16(float (&d)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kW4MmaStages = 3;                     // segments in a warp's ring
constexpr int kW4MmaStageBytes = 4 * 32 * 16;       // 4 slots of 16 B per lane
constexpr int kW4MmaRingBytes = kW4MmaStages * kW4MmaStageBytes;  // per warp

// wg / wh: codes of rows g and g + 8 (K / 2 bytes each); sg / sh: their fp16
// group scales; xs: the activations in the interleaved layout (shared or
// global memory); segments [sbeg, send); cpg = group / 32; ring: this warp's
// kW4MmaRingBytes of shared memory.  Returns the sums of rows g (.x) and
// g + 8 (.y), complete in all four lanes of the quad.
__device__ __forceinline__ float2 w4a16_mma_rows(const unsigned char* wg, const unsigned char* wh,
                                                 const uint16_t* sg, const uint16_t* sh,
                                                 const unsigned char* xs, int sbeg, int send,
                                                 int cpg, unsigned char* ring) {
    constexpr int S = kW4MmaStages;
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const bool own_e = g == t, own_o = g == t + 4;
    unsigned char* slot = ring + lane * 16;  // slot j of stage st: + (st * 4 + j) * 512
    uint16_t sc[S][4];                       // group scales of the segments in flight

    // segment s into stage st: its four 16-byte pieces (rows g, g + 8;
    // chunks t, t + 4) and, into registers, the scales of chunks 2t, 2t + 1
    auto issue = [&](int s, int st) {
        const size_t off = (size_t)s * (kW4MmaSeg / 2) + (size_t)t * 16;
        unsigned char* d = slot + st * kW4MmaStageBytes;
        cp_async16(d, wg + off);
        cp_async16(d + 512, wg + off + 64);
        cp_async16(d + 1024, wh + off);
        cp_async16(d + 1536, wh + off + 64);
        const int c0 = s * 8 + 2 * t;
        const int ga = group_of_chunk(c0, cpg), gb = group_of_chunk(c0 + 1, cpg);
        sc[st][0] = ld_stream_u16(sg + ga);
        sc[st][1] = ld_stream_u16(sg + gb);
        sc[st][2] = ld_stream_u16(sh + ga);
        sc[st][3] = ld_stream_u16(sh + gb);
    };

    uint4 xe = make_uint4(0u, 0u, 0u, 0u), xo = xe;  // B fragments: owners only
    float yg = 0.f, yh = 0.f;
#pragma unroll
    for (int u = 0; u < S - 1; ++u) {
        if (sbeg + u < send) issue(sbeg + u, u);
        cp_async_commit();
    }
    for (int s0 = sbeg; s0 < send; s0 += S) {
#pragma unroll
        for (int u = 0; u < S; ++u) {
            const int s = s0 + u;
            if (s < send) {
                if (s + S - 1 < send) issue(s + S - 1, (u + S - 1) % S);
                cp_async_commit();
                cp_async_wait<S - 1>();  // segment s (this thread's copies) has landed
                const unsigned char* st = slot + u * kW4MmaStageBytes;
                const uint4 w0 = *reinterpret_cast<const uint4*>(st);         // row g, chunk t
                const uint4 w1 = *reinterpret_cast<const uint4*>(st + 512);   // row g, chunk t + 4
                const uint4 w2 = *reinterpret_cast<const uint4*>(st + 1024);  // row g + 8, chunk t
                const uint4 w3 = *reinterpret_cast<const uint4*>(st + 1536);  // row g + 8, chunk t + 4
                const int ce = s * 8 + t;  // chunk t of the segment
                // four accumulators (one per code pair j): MMA chains of four
                // instead of sixteen dependent MMAs per segment
                float acc[4][4] = {};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (own_e) xe = *reinterpret_cast<const uint4*>(xs + int4_x_piece(ce, i, 4));
                    if (own_o) xo = *reinterpret_cast<const uint4*>(xs + int4_x_piece(ce + 4, i, 4));
                    uint32_t qa[4], qb[4], qc[4], qd[4];
                    unpack_int4x8_f16(word_of(w0, i), qa);
                    unpack_int4x8_f16(word_of(w1, i), qb);
                    unpack_int4x8_f16(word_of(w2, i), qc);
                    unpack_int4x8_f16(word_of(w3, i), qd);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_m16n8k16_f16(acc[j], qa[j], qc[j], qb[j], qd[j], word_of(xe, j),
                                         word_of(xo, j));
                }
                float d[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) d[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
                yg = fmaf(d[0], __half2float(__ushort_as_half(sc[u][0])), yg);
                yg = fmaf(d[1], __half2float(__ushort_as_half(sc[u][1])), yg);
                yh = fmaf(d[2], __half2float(__ushort_as_half(sc[u][2])), yh);
                yh = fmaf(d[3], __half2float(__ushort_as_half(sc[u][3])), yh);
            }
        }
    }
    cp_async_wait<0>();  // (only empty groups remain; the ring is free for reuse)
    yg += __shfl_xor_sync(0xffffffffu, yg, 1);
    yh += __shfl_xor_sync(0xffffffffu, yh, 1);
    yg += __shfl_xor_sync(0xffffffffu, yg, 2);
    yh += __shfl_xor_sync(0xffffffffu, yh, 2);
    return make_float2(yg, yh);
}

// Where k_gemv's warps' weight rings begin (after its activations, row-group
// partials and argmax candidates).
template <class P>
__host__ __device__ size_t w4_ring_offset(int MT, int K) {
    const bool direct = P::kDirectX && MT == 1;
    size_t x = direct ? 0 : (P::x_bytes(MT, K) + 15) & ~(size_t)15;
    return (x + (size_t)kWarps * 4 * MT * 4 + (size_t)kWarps * sizeof(ArgPart) + 15) &
           ~(size_t)15;
}

// The per-launch kernel takes this path for W4A16, one token, R = 16.
template <class P, int MT, int R>
struct W4Mma {
    static constexpr bool v = std::is_same<P, PolicyW4A16>::value && MT == 1 && R == kW4MmaRows;
};

// ---- the row-group computation shared by all kernels ------------------------------

// Chunks per row loaded ahead of use: about eight loads in flight per lane.
template <int MT, int R>
struct Unroll {
    static constexpr int v = (MT * R <= 1) ? 8 : (MT * R <= 2 ? 4 : 2);
};

// Geometry of one launch or phase, uniform over the CTA.
struct RowGeom {
    int K, nchunks, gk, cpg, ks;
    size_t rb;
};

template <class P>
__device__ __forceinline__ RowGeom row_geom_gk(int K, int group, int ks, int gk) {
    RowGeom g;
    g.K = K;
    g.nchunks = K / P::kElems;
    g.gk = gk;
    g.cpg = group / 32;
    g.ks = ks;
    g.rb = P::row_bytes(K);
    return g;
}

template <class P>
__device__ __forceinline__ RowGeom row_geom(int K, int group, int ks) {
    RowGeom g;
    g.K = K;
    g.nchunks = K / P::kElems;
    g.gk = K / group;
    g.cpg = group / 32;
    g.ks = ks;
    g.rb = P::row_bytes(K);
    return g;
}

// Fills rows[] for row group rg of table t; invalid rows alias the first row
// (loaded but dropped) so every load stays in bounds.
template <int R>
__device__ __forceinline__ void rows_of(const SegTable& t, int rg, bool active, size_t rb,
                                        RowRef (&rows)[R]) {
    RowRef z{};
    const RowRef first = active ? locate(t, rg * R, rb, z) : z;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        rows[r] = active ? locate(t, rg * R + r, rb, first) : first;
        if (!rows[r].valid) rows[r].w = first.w;
    }
}

// Streams R rows for this lane and returns the per-row sums, complete in every
// lane of the slot's first warp (kw == 0).  With ks > 1 the slot's warps meet
// at the slot's named barrier, so all of them must call it; inactive slots pass
// active = false.
// DX: one token, activations read from global memory at `xs` (coherent:
// bypassing L1); otherwise `xs` is the staged shared-memory copy.
// [cbeg, cend): the row's chunks to visit (a multiple of ks * 32 and the
// row's end by default; split-K launches give each CTA one such range).
template <class P, int MT, int R, bool DX = false, int UOVR = 0>
__device__ __forceinline__ void row_group(const RowRef (&rows)[R], bool active, const RowGeom& g,
                                          const unsigned char* xs, int* red,
                                          typename P::Acc (&acc)[R][MT], bool coherent = false,
                                          int cbeg = 0, int cend = -1) {
    using Acc = typename P::Acc;
    constexpr int U = UOVR > 0 ? UOVR : Unroll<MT, R>::v;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = g.ks;
    const int kw = warp % ks;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = Acc(0);

    if (active) {
        // Batches of U chunks per row, all loads of a batch issued before any
        // use (chunks past the row's end are skipped), so a short row costs one
        // memory round trip; the sums still run in ascending chunk order.
        const int step = ks * 32;
        const int ce = cend < 0 ? g.nchunks : cend;
        for (int c = cbeg + kw * 32 + lane; c < ce; c += U * step) {
            typename P::Chunk ch[U][R];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (c + u * step < ce)
#pragma unroll
                    for (int r = 0; r < R; ++r) P::load(ch[u][r], rows[r], c + u * step, g.gk, g.cpg);
            if constexpr (DX) {
                // one activation chunk (an L1 hit, mostly) kept in flight ahead of the MACs
                uint4 xn = P::load_x(xs, c, coherent);
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (c + u * step < ce) {
                        const uint4 xv = xn;
                        if (u + 1 < U && c + (u + 1) * step < ce)
                            xn = P::load_x(xs, c + (u + 1) * step, coherent);
#pragma unroll
                        for (int r = 0; r < R; ++r) P::mac_direct(acc[r], ch[u][r], xv);
                    }
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (c + u * step < ce)
#pragma unroll
                        for (int r = 0; r < R; ++r)
                            P::template mac<MT>(acc[r], ch[u][r], xs, c + u * step, g.K);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = warp_sum(acc[r][m]);

    if (ks > 1) {
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) red[(warp * R + r) * MT + m] = to_bits(acc[r][m]);
        }
        // only the slot's warps meet (its named barrier, ks warps)
        const int bar = slot_barrier(warp, ks);
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(ks * 32) : "memory");
        if (kw == 0) {
            for (int j = 1; j < ks; ++j) {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        acc[r][m] += from_bits<Acc>(red[((warp + j) * R + r) * MT + m]);
            }
        }
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(ks * 32) : "memory");
    }
}

// ---- the per-launch kernel ---------------------------------------------------------

// SPLIT: a split-K launch (grid = row-group blocks x p.kparts K ranges); the
// unsplit instantiation carries none of its bookkeeping.
template <class P, int MT, int R, bool ARGMAX, bool SPLIT>
__global__ void __launch_bounds__(kThreads) k_gemv(const __grid_constant__ GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    using Acc = typename P::Acc;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = p.ksplit;
    const int slots = kWarps / ks;
    const int slot = warp / ks, kw = warp - slot * ks;
    const RowGeom g = row_geom<P>(p.a.K, p.group, ks);
    const int n_rg = (p.t.N + R - 1) / R;
    // split-K across CTAs: CTA (sidx, bx) takes K range sidx of row groups bx,
    // bx + gx, ...: the lane chunk indices j in [J sidx / S, J (sidx + 1) / S)
    const int S = SPLIT ? p.kparts : 1;
    const int gx = SPLIT ? (int)gridDim.x / S : (int)gridDim.x;
    const int sidx = SPLIT ? (int)blockIdx.x / gx : 0;
    const int bx = (int)blockIdx.x - sidx * gx;
    int cbeg = 0, cend = -1;
    if constexpr (SPLIT) {
        const int stepc = ks * 32, J = (g.nchunks + stepc - 1) / stepc;
        cbeg = (int)((long long)J * sidx / S) * stepc;
        cend = min(g.nchunks, (int)((long long)J * (sidx + 1) / S) * stepc);
    }

    // Weights do not depend on the previous kernel: warm L2 with the rows this
    // CTA streams first while that kernel drains.
    if (!SPLIT && p.prefetch_bytes > 0 && threadIdx.x < slots * R) {
        const int r = blockIdx.x * slots * R + threadIdx.x;
        RowRef z{};
        const RowRef rr = locate(p.t, r, g.rb, z);
        if (rr.valid) {
            const size_t cap = (size_t)p.prefetch_bytes / (size_t)(slots * R);
            uint32_t n = (uint32_t)(g.rb < cap ? g.rb : cap);
            n &= ~15u;
            if (n) prefetch_l2(rr.w, n);
        }
    }
    griddep_launch_dependents();
    griddep_wait();

    constexpr bool DX = P::kDirectX && MT == 1;
    if constexpr (!DX) {
        P::stage_x(p.a, smem, MT);
        __syncthreads();
    }
    int* red = reinterpret_cast<int*>(smem + (DX ? 0 : ((P::x_bytes(MT, g.K) + 15) & ~(size_t)15)));
    const unsigned char* xsrc = DX ? static_cast<const unsigned char*>(p.a.x) : smem;

    float best_v = NAN;
    int best_i = INT_MAX;

    if constexpr (W4Mma<P, MT, R>::v) {
        // one warp per tile of 16 rows (ksplit = 1), on the tensor cores
        const int nseg = g.K / kW4MmaSeg;
        int sbeg = 0, send = nseg;
        if constexpr (SPLIT) {
            sbeg = (int)((long long)nseg * sidx / S);
            send = (int)((long long)nseg * (sidx + 1) / S);
        }
        const int q = lane >> 2, t = lane & 3;
        unsigned char* ring = smem + w4_ring_offset<P>(1, g.K) + (size_t)warp * kW4MmaRingBytes;
        for (int it = 0; it < p.iters; ++it) {
            const int tile = (it * gx + bx) * slots + slot;
            if (tile >= n_rg) continue;
            const int r0 = tile * kW4MmaRows;
            RowRef z{};
            const RowRef first = locate(p.t, r0, g.rb, z);
            // rows past the end alias the tile's first row (loaded, dropped)
            const RowRef ra = locate(p.t, r0 + q, g.rb, first);
            const RowRef rb = locate(p.t, r0 + q + 8, g.rb, first);
            const float2 y = w4a16_mma_rows(
                ra.w, rb.w, static_cast<const uint16_t*>(ra.scale) + (size_t)ra.local * g.gk,
                static_cast<const uint16_t*>(rb.scale) + (size_t)rb.local * g.gk, xsrc, sbeg, send,
                g.cpg, ring);
            if constexpr (ARGMAX) {
                float v = NAN;
                int i = INT_MAX;
                if (t == 0) {
                    if (ra.valid) {
                        p.logits[ra.global] = y.x;
                        v = y.x;
                        i = ra.global;
                    }
                    if (rb.valid) {
                        p.logits[rb.global] = y.y;
                        if (arg_better(y.y, rb.global, v, i)) {
                            v = y.y;
                            i = rb.global;
                        }
                    }
                }
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
                    if (arg_better(ov, oi, v, i)) {
                        v = ov;
                        i = oi;
                    }
                }
                if (lane == 0 && arg_better(v, i, best_v, best_i)) {
                    best_v = v;
                    best_i = i;
                }
            } else if constexpr (SPLIT) {
                int* part = static_cast<int*>(p.kpart) + (size_t)sidx * p.t.N;
                if (t == 0 && ra.valid) part[ra.global] = to_bits(y.x);
                if (t == 1 && rb.valid) part[rb.global] = to_bits(y.y);
            } else {
                if (t == 0 && ra.valid) P::store(ra, 0, y.x, 1.f);
                if (t == 1 && rb.valid) P::store(rb, 0, y.y, 1.f);
            }
        }
    } else {
    for (int it = 0; it < p.iters; ++it) {
        const int rg = (it * gx + bx) * slots + slot;
        const bool active = rg < n_rg;
        RowRef rows[R];
        rows_of<R>(p.t, rg, active, g.rb, rows);
        Acc acc[R][MT];
        row_group<P, MT, R, DX>(rows, active, g, xsrc, red, acc, false, cbeg, cend);

        if (kw == 0 && active) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (!rows[r].valid) continue;
                if (ARGMAX) {
                    const float sx = p.a.x_scale ? __ldg(p.a.x_scale) : 1.f;
                    const float v = P::finish(rows[r], acc[r][0], sx);
                    if (lane == 0) {
                        p.logits[rows[r].global] = v;
                        if (arg_better(v, rows[r].global, best_v, best_i)) {
                            best_v = v;
                            best_i = rows[r].global;
                        }
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        if (m < p.a.M && lane == ((r * MT + m) & 31)) {
                            if constexpr (SPLIT) {  // this K range's partial sum, for pass 2
                                static_cast<int*>(p.kpart)[((size_t)sidx * p.a.M + m) * p.t.N +
                                                           rows[r].global] = to_bits(acc[r][m]);
                            } else {
                                const float sx = p.a.x_scale ? __ldg(p.a.x_scale + m) : 1.f;
                                P::store(rows[r], m, acc[r][m], sx);
                            }
                        }
                }
            }
        }
    }
    }

    if (ARGMAX) {
        ArgPart* cta = reinterpret_cast<ArgPart*>(red + kWarps * 4 * MT);
        if (lane == 0) {
            cta[warp].v = best_v;
            cta[warp].i = best_i;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float bv = NAN;
            int bi = INT_MAX;
            for (int w = 0; w < kWarps; ++w)
                if (arg_better(cta[w].v, cta[w].i, bv, bi)) {
                    bv = cta[w].v;
                    bi = cta[w].i;
                }
            p.part[blockIdx.x].v = bv;
            p.part[blockIdx.x].i = bi;
        }
    }
}

// Split-K pass 2: adds each output's K-range partials in range order and
// applies the format's epilogue, one thread per output.  int32 partials
// (W8A8) add exactly, so those outputs equal the unsplit ones bit for bit.
template <class P>
__global__ void __launch_bounds__(256) k_split_finish(const __grid_constant__ GemvParams p) {
    using Acc = typename P::Acc;
    griddep_launch_dependents();
    griddep_wait();
    const int N = p.t.N, M = p.a.M, S = p.kparts;
    const int* part = static_cast<const int*>(p.kpart);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < M * N; i += gridDim.x * blockDim.x) {
        const int m = i / N, row = i - m * N;
        Acc acc = from_bits<Acc>(part[(size_t)m * N + row]);
        for (int s = 1; s < S; ++s) acc += from_bits<Acc>(part[((size_t)s * M + m) * N + row]);
        RowRef z{};
        const RowRef rr = locate(p.t, row, 0, z);
        const float sx = p.a.x_scale ? __ldg(p.a.x_scale + m) : 1.f;
        P::store(rr, m, acc, sx);
    }
}

// Shared memory of k_gemv: staged activations | row-group partials | per-warp
// argmax candidates | (W4A16 tensor-core tiles, R = kW4MmaRows) the warps'
// weight rings from w4_ring_offset on.
template <class P>
size_t smem_bytes_for(int MT, int K, int R = 0) {
    const bool direct = P::kDirectX && MT == 1;
    size_t x = direct ? 0 : (P::x_bytes(MT, K) + 15) & ~(size_t)15;
    if (std::is_same<P, PolicyW4A16>::value && MT == 1 && R == kW4MmaRows)
        return w4_ring_offset<P>(MT, K) + (size_t)kWarps * kW4MmaRingBytes;
    return x + (size_t)kWarps * 4 * MT * 4 + (size_t)kWarps * sizeof(ArgPart);
}

// Launches one instantiation, or (occ != nullptr) reports how many of its CTAs
// fit on one SM with this much dynamic shared memory.
template <class P, int MT, int R, bool ARGMAX>
cudaError_t run_one(const GemvParams* p, int grid, size_t smem, cudaStream_t s, int* occ) {
    const bool split = !ARGMAX && p && p->kparts > 1;
    auto fn = split ? k_gemv<P, MT, R, ARGMAX, !ARGMAX> : k_gemv<P, MT, R, ARGMAX, false>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, kThreads, smem);
    void* args[] = {const_cast<GemvParams*>(p)};
    return launch_pdl(reinterpret_cast<const void*>(fn), dim3(grid), dim3(kThreads), smem, s, args);
}

template <class P, int MT, bool ARGMAX>
cudaError_t run_r(int R, const GemvParams* p, int grid, size_t smem, cudaStream_t s, int* occ) {
    switch (R) {
        case 1: return run_one<P, MT, 1, ARGMAX>(p, grid, smem, s, occ);
        case 2: return run_one<P, MT, 2, ARGMAX>(p, grid, smem, s, occ);
        case 4: return run_one<P, MT, 4, ARGMAX>(p, grid, smem, s, occ);
        case kW4MmaRows:  // W4A16 at one token: tiles on the tensor cores
            if constexpr (W4Mma<P, MT, kW4MmaRows>::v)
                return run_one<P, MT, kW4MmaRows, ARGMAX>(p, grid, smem, s, occ);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

// The instantiations the launch heuristic can pick.
template <class P>
cudaError_t run_family_main(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ) {
    const size_t smem = smem_bytes_for<P>(L.MT, L.K, L.R);
    if (L.argmax) {
        if constexpr (P::kIntAct && P::kElems == 16) {
            return cudaErrorInvalidValue;  // no int8 lm_head
        } else {
            return L.MT == 1 ? run_r<P, 1, true>(L.R, p, L.grid, smem, s, occ)
                             : cudaErrorInvalidValue;
        }
    }
    switch (L.MT) {
        case 1: return run_r<P, 1, false>(L.R, p, L.grid, smem, s, occ);
        case 2: return run_r<P, 2, false>(L.R, p, L.grid, smem, s, occ);
        case 4: return run_r<P, 4, false>(L.R, p, L.grid, smem, s, occ);
        case 8:
            return L.R == 1 ? run_one<P, 8, 1, false>(p, L.grid, smem, s, occ)
                            : run_one<P, 8, 2, false>(p, L.grid, smem, s, occ);
        case 16:
            if constexpr (P::kElems == 16) {
                if (L.R == 4) return run_one<P, 16, 4, false>(p, L.grid, smem, s, occ);
            }
            return run_one<P, 16, 1, false>(p, L.grid, smem, s, occ);
        default: return cudaErrorInvalidValue;
    }
}

// Launches the main kernel, and with split-K its pass 2 behind it.
template <class P>
cudaError_t run_family(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ) {
    cudaError_t e = run_family_main<P>(L, p, s, occ);
    if (e != cudaSuccess || occ || !p || p->kparts <= 1 || L.argmax) return e;
    const int total = p->a.M * p->t.N;
    void* args[] = {const_cast<GemvParams*>(p)};
    return launch_pdl(reinterpret_cast<const void*>(k_split_finish<P>), dim3((total + 255) / 256),
                      dim3(256), 0, s, args);
}

}  // namespace dg
