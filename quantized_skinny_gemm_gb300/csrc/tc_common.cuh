// Building blocks of the tcgen05 tiles (gemv_tc.cu, gemv_tcq.cu): mbarrier
// waits with a bound, TMA tile loads, shared-memory matrix descriptors,
// tcgen05 MMA / commit / TMEM load-store wrappers, the stream-K work split and
// the per-stream fixup scratch.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "dg_internal.cuh"

namespace dg {
namespace tc {

constexpr int kRows = 128;                 // MMA M: weight rows per tile (TMEM lanes)
constexpr int kTok = 16;                   // MMA N: tokens (zero-padded)
constexpr int kPiece = kRows * kTok;       // 4-byte words of one partial tile
constexpr int kMaxCtas = 256;              // fixup slots: 2 per CTA
constexpr int kMaxTiles = 65536;           // fixup counters

// Instruction descriptor of tcgen05.mma .kind::f16: fp32 accumulator, A and B
// fp16 (or bf16), both K-major, N = 16, M = 128.
template <bool BF16>
constexpr uint32_t idesc_f16() {
    return (1u << 4) | (BF16 ? (1u << 7) | (1u << 10) : 0u) | ((uint32_t)(kTok >> 3) << 17) |
           ((uint32_t)(kRows >> 4) << 24);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with this parity to complete, at most `limit`
// polls; false (and the timeout recorded) if it did not.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned limit,
                                          int* err) {
    for (unsigned n = 0; n < limit; ++n)
        if (mbar_try(bar, parity)) return true;
    atomicExch(err, kErrTimeout);
    return false;
}

// The same wait for threads off the critical path (epilogue, converters):
// a short sleep between polls leaves the scheduler's issue slots to the warps
// that feed the tensor core.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, unsigned limit,
                                                int* err) {
    for (unsigned n = 0; n < limit; ++n) {
        if (mbar_try(bar, parity)) return true;
        __nanosleep(32);
    }
    atomicExch(err, kErrTimeout);
    return false;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, rows of 128 bytes
// in groups of 8 rows 1024 bytes apart (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B).  The 16-wide k step s of a stage starts 32 * s
// bytes into the swizzle row.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Starts a 16-column TMEM load (this warp's lane quarter) into r; r may be
// read only after tmem_ld_wait(r).  Several loads may be in flight at once.
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Waits for this thread's TMEM loads.  r passes through the wait, so that no
// use of the loaded registers can be scheduled above it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

__device__ __forceinline__ long long range_begin(long long c, long long total, long long G) {
    return c * total / G;
}

// The CTA whose range holds block `blk`.
__device__ __forceinline__ int cta_of_block(long long blk, long long total, long long G) {
    long long c = blk * G / total;
    while (c > 0 && range_begin(c, total, G) > blk) --c;
    while (c + 1 < G && range_begin(c + 1, total, G) <= blk) ++c;
    return (int)c;
}


// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- host side (gemv_tc.cu) ----------------------------------------------------------

// 2-D map of a row-major [outer][inner] array of `elem_bytes`-byte elements.
bool encode_2d(CUtensorMap* m, const void* base, CUtensorMapDataType type, int elem_bytes,
               long long inner, long long outer, int box_inner, int box_outer,
               CUtensorMapSwizzle swizzle);
bool have_encoder();

// The fixup scratch of one (device, stream): launches on one stream run one
// after another, so they can share it; launches on different streams never do.
struct Scratch {
    float* part = nullptr;      // [2 * kMaxCtas][kPiece] partial tiles (fp32 or int32)
    unsigned* count = nullptr;  // [kMaxTiles] pieces arrived, zero between launches
};
bool scratch(cudaStream_t s, Scratch* out);

// The dynamic shared memory opt-in of a kernel on this device, raised when a
// launch needs more than any before.
cudaError_t smem_attr_once(const void* fn, size_t smem);

}  // namespace tc
}  // namespace dg
