// Kernels around the weight stream that are not weight-streaming GEMVs: the
// causal-conv1d decode step, the load-time weight quantizers / packers, and
// the elementwise SwiGLU and residual add that a decoder runs when they are
// not fused into the stream's epilogue.
#include <cmath>

#include "dg_internal.cuh"

namespace dg {

// ---- elementwise epilogues ---------------------------------------------------------
// Eight fp16 elements per thread (one 16-byte vector each way), fp32 arithmetic,
// one rounding into fp16.
__global__ void __launch_bounds__(256) k_swiglu(const uint4* __restrict__ g,
                                                const uint4* __restrict__ u, uint4* h, int n8) {
    griddep_launch_dependents();
    griddep_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += gridDim.x * blockDim.x) {
        const uint4 a = g[i], b = u[i];
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 fa = __half22float2(u32_as_h2(av[j])), fb = __half22float2(u32_as_h2(bv[j]));
            o[j] = h2_as_u32(__floats2half2_rn(silu_f32(fa.x) * fb.x, silu_f32(fa.y) * fb.y));
        }
        h[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void __launch_bounds__(256) k_residual_add(const uint4* __restrict__ a,
                                                      const uint4* __restrict__ b, uint4* out,
                                                      int n8) {
    griddep_launch_dependents();
    griddep_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += gridDim.x * blockDim.x) {
        const uint4 x = a[i], r = b[i];
        const uint32_t xv[4] = {x.x, x.y, x.z, x.w}, rv[4] = {r.x, r.y, r.z, r.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 fa = __half22float2(u32_as_h2(xv[j])), fb = __half22float2(u32_as_h2(rv[j]));
            o[j] = h2_as_u32(__floats2half2_rn(fa.x + fb.x, fa.y + fb.y));
        }
        out[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

static int elementwise_grid(int n8) {
    const int need = (n8 + 255) / 256, cap = sm_count() * 8;
    return need < cap ? (need > 0 ? need : 1) : cap;
}

cudaError_t launch_swiglu(const void* g, const void* u, void* h, int n, cudaStream_t s) {
    int n8 = n / 8;
    const uint4 *pg = static_cast<const uint4*>(g), *pu = static_cast<const uint4*>(u);
    uint4* ph = static_cast<uint4*>(h);
    void* args[] = {&pg, &pu, &ph, &n8};
    return launch_pdl(reinterpret_cast<const void*>(k_swiglu), dim3(elementwise_grid(n8)),
                      dim3(256), 0, s, args);
}

cudaError_t launch_residual_add(const void* a, const void* b, void* out, int n, cudaStream_t s) {
    int n8 = n / 8;
    const uint4 *pa = static_cast<const uint4*>(a), *pb = static_cast<const uint4*>(b);
    uint4* po = static_cast<uint4*>(out);
    void* args[] = {&pa, &pb, &po, &n8};
    return launch_pdl(reinterpret_cast<const void*>(k_residual_add), dim3(elementwise_grid(n8)),
                      dim3(256), 0, s, args);
}

// ---- causal-conv1d decode step ------------------------------------------------------
// One thread per token and group of eight channels: the group's window
// (8 x (W-1) halves, contiguous), taps (8 x W halves), input and bias arrive
// as 16-byte vectors; per channel v = bias + sum_j w[j] u[j] with exact fp16 x
// fp16 products and one fp32 rounding per term, j ascending; the window then
// shifts by one input.
template <int W>
__global__ void __launch_bounds__(256) k_conv1d_update(const __half* __restrict__ x, __half* state,
                                                       const __half* __restrict__ w,
                                                       const __half* __restrict__ bias,
                                                       __half* __restrict__ y, int M, int C,
                                                       int silu) {
    griddep_launch_dependents();
    griddep_wait();
    const int groups = C / 8;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= M * groups) return;
    const int m = t / groups, c0 = (t - m * groups) * 8;
    constexpr int S = W - 1;  // window inputs kept per channel
    // window: 8 channels x S halves = S 16-byte vectors
    uint16_t st[8 * S];
    __half* sp = state + ((size_t)m * C + c0) * S;
#pragma unroll
    for (int q = 0; q < S; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(sp + 8 * q);
        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            st[8 * q + 2 * h] = lo16(vv[h]);
            st[8 * q + 2 * h + 1] = hi16(vv[h]);
        }
    }
    uint16_t tp[8 * W];
    const __half* wp = w + (size_t)c0 * W;
#pragma unroll
    for (int q = 0; q < W; ++q) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(wp + 8 * q));
        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            tp[8 * q + 2 * h] = lo16(vv[h]);
            tp[8 * q + 2 * h + 1] = hi16(vv[h]);
        }
    }
    const uint4 xv = *reinterpret_cast<const uint4*>(x + (size_t)m * C + c0);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    uint32_t bw[4] = {0, 0, 0, 0};
    if (bias) {
        const uint4 bv = __ldg(reinterpret_cast<const uint4*>(bias + c0));
        bw[0] = bv.x, bw[1] = bv.y, bw[2] = bv.z, bw[3] = bv.w;
    }
    uint16_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint16_t xi = (i & 1) ? hi16(xw[i >> 1]) : lo16(xw[i >> 1]);
        const uint16_t bi = (i & 1) ? hi16(bw[i >> 1]) : lo16(bw[i >> 1]);
        float v = __half2float(__ushort_as_half(bi));
#pragma unroll
        for (int j = 0; j < S; ++j) v = fma_f16(tp[i * W + j], st[i * S + j], v);
        v = fma_f16(tp[i * W + S], xi, v);
        if (silu) v = silu_f32(v);
        out[i] = __half_as_ushort(__float2half_rn(v));
    }
    *reinterpret_cast<uint4*>(y + (size_t)m * C + c0) =
        make_uint4((uint32_t)out[0] | ((uint32_t)out[1] << 16), (uint32_t)out[2] | ((uint32_t)out[3] << 16),
                   (uint32_t)out[4] | ((uint32_t)out[5] << 16), (uint32_t)out[6] | ((uint32_t)out[7] << 16));
    // shifted window: channel i keeps inputs 1 .. S-1 and appends x_i
    uint16_t ns[8 * S];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int j = 0; j + 1 < S; ++j) ns[i * S + j] = st[i * S + j + 1];
        ns[i * S + S - 1] = (i & 1) ? hi16(xw[i >> 1]) : lo16(xw[i >> 1]);
    }
#pragma unroll
    for (int q = 0; q < S; ++q) {
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 4; ++h)
            o[h] = (uint32_t)ns[8 * q + 2 * h] | ((uint32_t)ns[8 * q + 2 * h + 1] << 16);
        *reinterpret_cast<uint4*>(sp + 8 * q) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int W>
static cudaError_t launch_conv1d_w(const void* x, void* state, const void* w, const void* bias,
                                   void* y, int M, int C, int silu, cudaStream_t s) {
    const __half* px = static_cast<const __half*>(x);
    __half* ps = static_cast<__half*>(state);
    const __half* pw = static_cast<const __half*>(w);
    const __half* pb = static_cast<const __half*>(bias);
    __half* py = static_cast<__half*>(y);
    const int threads = M * (C / 8);
    void* args[] = {&px, &ps, &pw, &pb, &py, &M, &C, &silu};
    return launch_pdl(reinterpret_cast<const void*>(k_conv1d_update<W>), dim3((threads + 255) / 256),
                      dim3(256), 0, s, args);
}

cudaError_t launch_conv1d_update(const void* x, void* state, const void* w, const void* bias,
                                 void* y, int M, int C, int width, int silu, cudaStream_t s) {
    switch (width) {
        case 2: return launch_conv1d_w<2>(x, state, w, bias, y, M, C, silu, s);
        case 3: return launch_conv1d_w<3>(x, state, w, bias, y, M, C, silu, s);
        case 4: return launch_conv1d_w<4>(x, state, w, bias, y, M, C, silu, s);
        case 5: return launch_conv1d_w<5>(x, state, w, bias, y, M, C, silu, s);
        case 6: return launch_conv1d_w<6>(x, state, w, bias, y, M, C, silu, s);
        case 7: return launch_conv1d_w<7>(x, state, w, bias, y, M, C, silu, s);
        case 8: return launch_conv1d_w<8>(x, state, w, bias, y, M, C, silu, s);
    }
    return cudaErrorInvalidValue;
}

// ---- load-time weight quantizers -----------------------------------------------------
// Per-output-channel int8: one warp per row.  amax = max |w| (fp32, exact),
// s = amax / 127 (IEEE fp32) or 1 for an all-zero row, q = clamp(rne(w / s)).
__global__ void __launch_bounds__(256) k_quant_w8(const __half* __restrict__ W, int8_t* Wq,
                                                  float* s_out, int N, int K) {
    const int lane = threadIdx.x & 31;
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= N) return;
    const __half* wr = W + (size_t)row * K;
    float amax = 0.f;
    for (int k = lane * 8; k < K; k += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(wr + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(u32_as_h2(w[i]));
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.f ? __fdiv_rn(amax, 127.f) : 1.f;
    if (lane == 0) s_out[row] = s;
    int8_t* qr = Wq + (size_t)row * K;
    for (int k = lane * 8; k < K; k += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(wr + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(u32_as_h2(w[i]));
            const int q0 = max(-127, min(127, __float2int_rn(__fdiv_rn(f.x, s))));
            const int q1 = max(-127, min(127, __float2int_rn(__fdiv_rn(f.y, s))));
            out[i >> 1] |= ((uint32_t)(q0 & 0xFF) | ((uint32_t)(q1 & 0xFF) << 8)) << ((i & 1) * 16);
        }
        *reinterpret_cast<uint2*>(qr + k) = make_uint2(out[0], out[1]);
    }
}

// Groupwise int4: one thread per group of G consecutive k of a row.
// s = fp16(amax / 7) (IEEE fp32 division, then round to nearest even fp16),
// raised to the smallest fp16 subnormal if that rounds to 0, or 1 for an
// all-zero group; code = clamp(rne(w / s), -7, 7) with s widened to fp32;
// two codes per byte, the even k in the low nibble (two's complement).
__global__ void __launch_bounds__(256) k_quant_w4(const __half* __restrict__ W, uint8_t* Wq,
                                                  __half* scales, int N, int K, int G) {
    const int gk = K / G;
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (long long)N * gk) return;
    const int row = (int)(t / gk), grp = (int)(t - (long long)row * gk);
    const __half* wg = W + (size_t)row * K + (size_t)grp * G;
    float amax = 0.f;
    for (int k = 0; k < G; k += 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(wg + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(u32_as_h2(w[i]));
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
    __half s16 = __float2half_rn(1.f);
    if (amax > 0.f) {
        s16 = __float2half_rn(__fdiv_rn(amax, 7.f));
        if (__half2float(s16) < 5.9604644775390625e-08f) s16 = __ushort_as_half((uint16_t)1);  // 2^-24
    }
    scales[(size_t)row * gk + grp] = s16;
    const float s = __half2float(s16);
    uint8_t* qg = Wq + ((size_t)row * K + (size_t)grp * G) / 2;
    for (int k = 0; k < G; k += 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(wg + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(u32_as_h2(w[i]));
            const int q0 = max(-7, min(7, __float2int_rn(__fdiv_rn(f.x, s))));
            const int q1 = max(-7, min(7, __float2int_rn(__fdiv_rn(f.y, s))));
            packed |= ((uint32_t)(q0 & 0xF) | ((uint32_t)(q1 & 0xF) << 4)) << (8 * i);
        }
        *reinterpret_cast<uint32_t*>(qg + k / 2) = packed;
    }
}

cudaError_t launch_quant_w8(const void* W, int8_t* Wq, float* s, int N, int K, cudaStream_t st) {
    const long long threads = (long long)N * 32;
    k_quant_w8<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(static_cast<const __half*>(W), Wq,
                                                                   s, N, K);
    return cudaGetLastError();
}

cudaError_t launch_quant_w4(const void* W, uint8_t* Wq, void* scales, int N, int K, int G,
                            cudaStream_t st) {
    const long long threads = (long long)N * (K / G);
    k_quant_w4<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
        static_cast<const __half*>(W), Wq, static_cast<__half*>(scales), N, K, G);
    return cudaGetLastError();
}

}  // namespace dg
