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

// Segment of global row r and the row's index inside it: by position, or for
// a SwiGLU pair table by parity (row 2i is gate row i, 2i + 1 up row i).
__device__ __forceinline__ int seg_of_row(const SegTable& t, int r, int* local) {
    if (t.pair) {
        *local = r >> 1;
        return r & 1;
    }
    int s = 0;
#pragma unroll
    for (int i = 1; i < kMaxSeg; ++i)
        if (i < t.nseg && r >= t.seg[i].row_begin) s = i;
    *local = r - t.seg[s].row_begin;
    return s;
}

__device__ __forceinline__ RowRef locate(const SegTable& t, int r, size_t row_bytes,
                                         const RowRef& fallback) {
    RowRef rr = fallback;
    rr.valid = false;
    if (r >= t.N) return rr;
    const int s = seg_of_row(t, r, &rr.local);
    const Segment& sg = t.seg[s];
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

// Writes an op's final fp32 value for token m of row r into its output, as
// fp16 (bf16 for the bf16 format), round to nearest even.
template <bool BF16>
__device__ __forceinline__ void write_out(const RowRef& r, int m, float v) {
    const size_t o = (size_t)m * r.seg_rows + r.local;
    if (BF16)
        static_cast<__nv_bfloat16*>(r.y)[o] = __float2bfloat16_rn(v);
    else
        static_cast<__half*>(r.y)[o] = __float2half_rn(v);
}
template <bool BF16>
__device__ __forceinline__ float read_res(const void* res, size_t o) {
    return BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(res)[o])
                : __half2float(static_cast<const __half*>(res)[o]);
}

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
    static constexpr bool kBF16 = BF16;
    static constexpr int kElems = 8;
    static constexpr bool kMacRows = false;  // one row per mac() call
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
    __device__ __forceinline__ static void load(Chunk& ch, const unsigned char* wrow, const uint16_t*,
                                                int c, int) {
        ch.w = ld_stream16(wrow + (unsigned)c * 16u);
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
    static constexpr bool kBF16 = false;
    static constexpr int kElems = 16;
    static constexpr bool kMacRows = false;  // one row per mac() call
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
    __device__ __forceinline__ static void load(Chunk& ch, const unsigned char* wrow, const uint16_t*,
                                                int c, int) {
        ch.w = ld_stream16(wrow + (unsigned)c * 16u);
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

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
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
// Scale group of chunk c when cpg chunks share a scale: a shift when cpg is a
// power of two (cps = log2 cpg), a division otherwise (cps < 0).
__device__ __forceinline__ int group_of_chunk(int c, int cpg, int cps) {
    return cps >= 0 ? c >> cps : c / cpg;
}

__device__ __forceinline__ unsigned int4_x_piece(int c, int i, int pieces) {
    return ((unsigned)(c >> 5) * (unsigned)pieces + (unsigned)i) * 512u + (unsigned)(c & 31) * 16u;
}

// Groupwise int4 weights with fp16 activations; 32 codes per chunk.  Chunk c
// covers codes [32c, 32c + 32) of the row and uses the scale of group c / cpg
// (cpg = group / 32).  Activations are staged as fp16 in the interleaved
// layout, four 16-byte pieces per chunk: piece i holds the pairs (x0,x4)
// (x1,x5) (x2,x6) (x3,x7) of the chunk's i-th block of eight, lined up with the
// unpacked code pairs.  Each code (exact in fp16) meets its activation in one
// mixed-precision FMA (fp16 x fp16 + fp32: the product of a 4-bit code and an
// 11-bit significand is exact, one rounding).  Per row and token a chunk runs
// two chains (blocks 0 and 2, blocks 1 and 3, in ascending k), which meet once
// before the group scale is applied.  All rows of a slot go through one call,
// so each activation piece is loaded once for all of them.
struct PolicyW4A16 {
    static constexpr bool kBF16 = false;
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
    // wrow: the row's codes; srow: the row's group scales; grp: chunk c's group
    __device__ __forceinline__ static void load(Chunk& ch, const unsigned char* wrow,
                                                const uint16_t* srow, int c, int grp) {
        ch.w = ld_stream16(wrow + (unsigned)c * 16u);
        ch.s = ld_stream_u16(srow + grp);
    }
    static constexpr bool kMacRows = true;  // mac_rows() takes the whole slot
    template <int MT, int R>
    __device__ __forceinline__ static void mac_rows(Acc (&acc)[R][MT], const Chunk (&ch)[R],
                                                    const unsigned char* xs, int c, int K) {
        mac_rows_at<MT, R>(acc, ch, xs + int4_x_piece(c, 0, 4), token_bytes(K));
    }
    // xc: piece 0 of the chunk's activations of token 0 (piece i at + 512 i,
    // token m at + m tb)
    template <int MT, int R>
    __device__ __forceinline__ static void mac_rows_at(Acc (&acc)[R][MT], const Chunk (&ch)[R],
                                                       const unsigned char* xc, size_t tb) {
        float a[R][MT][2];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) a[r][m][0] = a[r][m][1] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // block i of the chunk: codes 8i .. 8i + 7
            uint32_t q[R][4];
#pragma unroll
            for (int r = 0; r < R; ++r) unpack_int4x8_f16(word_of(ch[r].w, i), q[r]);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 xp = *reinterpret_cast<const uint4*>(xc + m * tb + i * 512);
                const uint32_t xv[4] = {xp.x, xp.y, xp.z, xp.w};
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float& ar = a[r][m][i & 1];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {  // (c_j, c_j+4) against (x_j, x_j+4)
                        ar = fma_f16(lo16(q[r][j]), lo16(xv[j]), ar);
                        ar = fma_f16(hi16(q[r][j]), hi16(xv[j]), ar);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float s = __half2float(__ushort_as_half(ch[r].s));
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] = fmaf(a[r][m][0] + a[r][m][1], s, acc[r][m]);
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
    static constexpr bool kBF16 = false;
    static constexpr int kElems = 32;
    static constexpr bool kMacRows = false;  // one row per mac() call
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
    // wrow: the row's codes; srow: the row's group scales; grp: chunk c's group
    __device__ __forceinline__ static void load(Chunk& ch, const unsigned char* wrow,
                                                const uint16_t* srow, int c, int grp) {
        ch.w = ld_stream16(wrow + (unsigned)c * 16u);
        ch.s = ld_stream_u16(srow + grp);
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

// Stores token m of row r: the plain store, or with an epilogue the fp32
// result plus the residual (res, [M][rows] of the output type), or for a
// SwiGLU pair silu(gate) * up with `up` the pair's second row.
template <class P>
__device__ __forceinline__ void store_row(const RowRef& r, int m, typename P::Acc a, float sx,
                                          const void* res, bool pair, const RowRef& up,
                                          typename P::Acc au) {
    if (!res && !pair) {
        P::store(r, m, a, sx);
        return;
    }
    float v = P::finish(r, a, sx);
    if (res) v += read_res<P::kBF16>(res, (size_t)m * r.seg_rows + r.local);
    if (pair) v = silu_f32(v) * P::finish(up, au, sx);
    write_out<P::kBF16>(r, m, v);
}

// Named barrier of warp `warp`'s slot when ks = 2, 4 or 8 warps share a row.
// In a persistent kernel warps move through phases independently, so phases
// with different ks can be live at once, and a named barrier must never be
// used with two thread counts at the same time: the splits take disjoint ids,
// ks = 2 from 1 upward (1..8), ks = 8 at 9..10 and ks = 4 from 14 downward
// (14..11), for up to 16 warps; 0 is __syncthreads.
__device__ __forceinline__ int slot_barrier(int warp, int ks) {
    return ks == 4 ? 14 - warp / 4 : ks == 8 ? 9 + warp / 8 : 1 + warp / ks;
}

// ---- the row-group computation shared by all kernels ------------------------------

// Chunks per row loaded ahead of use: about eight loads in flight per lane.
template <int MT, int R>
struct Unroll {
    static constexpr int v = (MT * R <= 1) ? 8 : (MT * R <= 2 ? 4 : 2);
};

// Geometry of one launch or phase, uniform over the CTA.
struct RowGeom {
    int K, nchunks, gk, cpg, cps, ks;   // cps: log2(cpg), or -1 if cpg is no power of two
    size_t rb;
};

__device__ __forceinline__ int log2_or_neg(int v) { return (v & (v - 1)) == 0 ? __ffs(v) - 1 : -1; }

template <class P>
__device__ __forceinline__ RowGeom row_geom_gk(int K, int group, int ks, int gk) {
    RowGeom g;
    g.K = K;
    g.nchunks = K / P::kElems;
    g.gk = gk;
    g.cpg = group / 32;
    g.cps = log2_or_neg(g.cpg);
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
    g.cps = log2_or_neg(g.cpg);
    g.ks = ks;
    g.rb = P::row_bytes(K);
    return g;
}

// Fills rows[] for row group rg of table t; invalid rows alias the first row
// (loaded but dropped) so every load stays in bounds.
// When the group's rows all lie in the first row's matrix (segments are
// contiguous; SwiGLU pairs interleave two), the next rows follow from it.
template <int R>
__device__ __forceinline__ void rows_of(const SegTable& t, int rg, bool active, size_t rb,
                                        RowRef (&rows)[R]) {
    RowRef z{};
    const RowRef first = active ? locate(t, rg * R, rb, z) : z;
    const bool one_seg = R > 1 && active && first.valid && !t.pair && first.local + R <= first.seg_rows;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (one_seg) {
            rows[r] = first;
            rows[r].w = first.w + (size_t)r * rb;
            rows[r].local = first.local + r;
            rows[r].global = first.global + r;
        } else {
            rows[r] = active ? locate(t, rg * R + r, rb, first) : first;
        }
        if (!rows[r].valid) rows[r].w = first.w;
    }
}

// The slot loop of W4A16 at one token when one warp owns a row (ks = 1), the
// whole row is summed (no split-K) and a scale group spans a power of two of
// chunks, at most 32 (group <= 1024): lane l visits chunks l, l + 32, ... in
// ascending order, U of them per batch, through row pointers advanced by
// constant strides.  Same loads and the same arithmetic, in the same order,
// as row_group, so the two give identical bits; this one issues fewer
// integer instructions per chunk.
template <class P, int R, int U>
__device__ __forceinline__ void row_group_w4_ks1(const RowRef (&rows)[R], const RowGeom& g,
                                                 const unsigned char* xs, float (&acc)[R][1]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r][0] = 0.f;
    const int nj = (g.nchunks - lane + 31) >> 5;   // this lane's chunks
    const int sstep = 32 >> g.cps;                  // scale groups per 32 chunks
    const unsigned char* wp[R];
    const uint16_t* sp[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        wp[r] = rows[r].w + lane * 16;
        sp[r] = static_cast<const uint16_t*>(rows[r].scale) + (size_t)rows[r].local * g.gk +
                (lane >> g.cps);
    }
    const unsigned char* xp = xs + lane * 16;       // chunk lane + 32 j: + 2048 j
    int j = 0;
    for (; j + U <= nj; j += U) {
        typename P::Chunk ch[U][R];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int r = 0; r < R; ++r) {
                ch[u][r].w = ld_stream16(wp[r] + u * 512);
                ch[u][r].s = ld_stream_u16(sp[r] + u * sstep);
            }
#pragma unroll
        for (int u = 0; u < U; ++u) P::template mac_rows_at<1, R>(acc, ch[u], xp + u * 2048, 0);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            wp[r] += U * 512;
            sp[r] += U * sstep;
        }
        xp += U * 2048;
    }
    for (; j < nj; ++j) {
        typename P::Chunk ch[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            ch[r].w = ld_stream16(wp[r]);
            ch[r].s = ld_stream_u16(sp[r]);
            wp[r] += 512;
            sp[r] += sstep;
        }
        P::template mac_rows_at<1, R>(acc, ch, xp, 0);
        xp += 2048;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r][0] = warp_sum(acc[r][0]);
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
    constexpr int UB = UOVR > 0 ? UOVR : Unroll<MT, R>::v;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = g.ks;
    const int kw = warp % ks;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = Acc(0);

    if constexpr (P::kMacRows && MT == 1 && !DX) {
        if (ks == 1 && cbeg == 0 && cend < 0 && g.cps >= 0 && g.cps <= 5) {
            if (active) row_group_w4_ks1<P, R, UB>(rows, g, xs, acc);
            return;
        }
    }
    if (active) {
        // Batches of U chunks per row, all loads of a batch issued before any
        // use (chunks past the row's end are skipped), so a short row costs one
        // memory round trip; the sums still run in ascending chunk order.
        // W4A16 at one token reaches this general loop only for rare shapes
        // (split rows, split-K, odd group sizes): one chunk per batch there
        // keeps its registers below the fast loop's
        constexpr int U = (P::kMacRows && MT == 1) ? 1 : UB;
        const int step = ks * 32;
        const int ce = cend < 0 ? g.nchunks : cend;
        // per-row bases, once per row group: codes, and (int4) the group scales
        const unsigned char* wrow[R];
        const uint16_t* srow[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            wrow[r] = rows[r].w;
            srow[r] = P::kElems == 32 ? static_cast<const uint16_t*>(rows[r].scale) +
                                            (size_t)rows[r].local * g.gk
                                      : nullptr;
        }
        for (int c = cbeg + kw * 32 + lane; c < ce; c += U * step) {
            typename P::Chunk ch[U][R];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (c + u * step < ce) {
                    const int grp = P::kElems == 32 ? group_of_chunk(c + u * step, g.cpg, g.cps) : 0;
#pragma unroll
                    for (int r = 0; r < R; ++r) P::load(ch[u][r], wrow[r], srow[r], c + u * step, grp);
                }
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
            } else if constexpr (P::kMacRows) {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (c + u * step < ce) P::template mac_rows<MT, R>(acc, ch[u], xs, c + u * step, g.K);
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

    {
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
                    if (p.t.pair && (r & 1)) continue;  // stored with its gate row
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        if (m < p.a.M && lane == ((r * MT + m) & 31)) {
                            if constexpr (SPLIT) {  // this K range's partial sum, for pass 2
                                static_cast<int*>(p.kpart)[((size_t)sidx * p.a.M + m) * p.t.N +
                                                           rows[r].global] = to_bits(acc[r][m]);
                            } else {
                                const float sx = p.a.x_scale ? __ldg(p.a.x_scale + m) : 1.f;
                                const int ru = r + 1 < R ? r + 1 : r;  // (pairs: R is even)
                                store_row<P>(rows[r], m, acc[r][m], sx, p.t.res, p.t.pair != 0,
                                             rows[ru], acc[ru][m]);
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
// argmax candidates.
template <class P>
size_t smem_bytes_for(int MT, int K) {
    const bool direct = P::kDirectX && MT == 1;
    size_t x = direct ? 0 : (P::x_bytes(MT, K) + 15) & ~(size_t)15;
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
        default: return cudaErrorInvalidValue;
    }
}

// The instantiations the launch heuristic can pick.
template <class P>
cudaError_t run_family_main(const GemvLaunch& L, const GemvParams* p, cudaStream_t s, int* occ) {
    const size_t smem = smem_bytes_for<P>(L.MT, L.K);
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
            } else {
                if (L.R == 2) return run_one<P, 16, 2, false>(p, L.grid, smem, s, occ);  // SwiGLU pairs
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
