// Small kernels around the weight stream: the second level of the greedy
// argmax, per-token int8 activation quantization, and the HBM probes.
#include <climits>
#include <cmath>

#include "dg_internal.cuh"

namespace dg {

// ---- argmax level 2 ---------------------------------------------------------------
// One CTA reduces the per-CTA (value, index) partials of the lm_head kernel
// under the total order of arg_better (larger value, then lower index).  The
// maximum of a total order does not depend on the reduction tree, so any
// fixed tree gives the same token.
__global__ void __launch_bounds__(1024) k_argmax_pass2(const ArgPart* __restrict__ part,
                                                       int nparts, int32_t* __restrict__ token) {
    griddep_launch_dependents();
    griddep_wait();
    float bv = NAN;
    int bi = INT_MAX;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) {
        const ArgPart a = part[i];
        if (arg_better(a.v, a.i, bv, bi)) {
            bv = a.v;
            bi = a.i;
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
    __shared__ float sv[32];
    __shared__ int si[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        sv[warp] = bv;
        si[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            if (arg_better(sv[w], si[w], bv, bi)) {
                bv = sv[w];
                bi = si[w];
            }
        *token = bi == INT_MAX ? -1 : bi;
    }
}

cudaError_t launch_argmax_pass2(const ArgPart* part, int nparts, int32_t* token, cudaStream_t s) {
    void* args[] = {const_cast<ArgPart**>(&part), &nparts, &token};
    return launch_pdl(reinterpret_cast<const void*>(k_argmax_pass2), dim3(1), dim3(1024), 0, s, args);
}

// ---- per-token int8 activations -----------------------------------------------------
// One CTA per token: amax = max |x|, s = amax / 127 (IEEE fp32 division),
// q = clamp(rne(x / s), -127, 127); s = 1, q = 0 for an all-zero token.
__global__ void __launch_bounds__(256) k_quant_act(const __half* __restrict__ x,
                                                   int8_t* __restrict__ xq,
                                                   float* __restrict__ xs, int K) {
    griddep_launch_dependents();
    griddep_wait();
    const __half* xr = x + (size_t)blockIdx.x * K;
    int8_t* qr = xq + (size_t)blockIdx.x * K;
    float amax = 0.f;
    for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(u32_as_h2(w[i]));
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, red[w]);
    const float s = amax > 0.f ? __fdiv_rn(amax, 127.f) : 1.f;
    if (threadIdx.x == 0) xs[blockIdx.x] = s;
    for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(u32_as_h2(w[i]));
            int q0 = 0, q1 = 0;
            if (amax > 0.f) {
                q0 = max(-127, min(127, __float2int_rn(__fdiv_rn(f.x, s))));
                q1 = max(-127, min(127, __float2int_rn(__fdiv_rn(f.y, s))));
            }
            out[i >> 1] |= ((uint32_t)(q0 & 0xFF) | ((uint32_t)(q1 & 0xFF) << 8)) << ((i & 1) * 16);
        }
        *reinterpret_cast<uint2*>(qr + k) = make_uint2(out[0], out[1]);
    }
}

cudaError_t launch_quant_act(const __half* x, int8_t* xq, float* s, int M, int K, cudaStream_t st) {
    void* args[] = {const_cast<__half**>(&x), &xq, &s, &K};
    return launch_pdl(reinterpret_cast<const void*>(k_quant_act), dim3(M), dim3(256), 0, st, args);
}

// ---- HBM probes -------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_probe_copy(const uint4* __restrict__ src,
                                                    uint4* __restrict__ dst, size_t n) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 a = ld_stream16(src + i), b = ld_stream16(src + i + stride);
        const uint4 c = ld_stream16(src + i + 2 * stride), d = ld_stream16(src + i + 3 * stride);
        __stcs(dst + i, a);
        __stcs(dst + i + stride, b);
        __stcs(dst + i + 2 * stride, c);
        __stcs(dst + i + 3 * stride, d);
    }
    for (; i < n; i += stride) __stcs(dst + i, ld_stream16(src + i));
}

__global__ void __launch_bounds__(256) k_probe_read(const uint4* __restrict__ src, size_t n,
                                                    uint32_t* __restrict__ sink) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 a = ld_stream16(src + i), b = ld_stream16(src + i + stride);
        const uint4 c = ld_stream16(src + i + 2 * stride), d = ld_stream16(src + i + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w;
        acc ^= c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < n; i += stride) {
        const uint4 a = ld_stream16(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) atomicXor(sink + (blockIdx.x & 1023), acc);
}

static int probe_grid() { return sm_count() * 8; }

cudaError_t launch_probe_copy(const void* src, void* dst, size_t bytes, cudaStream_t s) {
    k_probe_copy<<<probe_grid(), 256, 0, s>>>(static_cast<const uint4*>(src),
                                              static_cast<uint4*>(dst), bytes / 16);
    return cudaGetLastError();
}

cudaError_t launch_probe_read(const void* src, size_t bytes, uint32_t* sink, cudaStream_t s) {
    k_probe_read<<<probe_grid(), 256, 0, s>>>(static_cast<const uint4*>(src), bytes / 16, sink);
    return cudaGetLastError();
}

}  // namespace dg
