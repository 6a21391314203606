// Persistent decode-step kernel with a TMA-fed weight ring (fp16 / bf16
// weights, one token): the same work as k_step (graph-accelerated decode of
// EdgeFM, section 2.C, one launch per step), with the weight stream decoupled
// from the arithmetic.
//
// A CTA's share of a phase is a contiguous row slice, and rows are stored one
// after another, so the slice is at most kMaxSeg contiguous byte ranges (one
// per fused matrix).  One producer thread walks the CTA's slices of all phases
// in order and copies them into a ring of shared-memory stages with
// cp.async.bulk (the Tensor Memory Accelerator's linear copy), packing each
// stage with consecutive rows across matrix and phase boundaries (a row is
// never split); each stage has a "full" mbarrier (transaction bytes of every
// copy into it, one arrival when the producer closes it) and an "empty" one
// (one arrival per consumer warp).  The bytes in flight are the
// ring's size, not what the registers of the computing warps can hold, and
// the producer runs ahead across grid barriers: weights never depend on the
// activations, so the ring is already full when the consumers pass a barrier.
//
// Consumer warps compute each row exactly as row_group does for one token
// (lane l of slot warp kw takes chunks (j * ks + kw) * 32 + l in ascending j,
// two four-product chains per chunk, the xor butterfly, then the slot's warps
// in kw order), reading the weights from the ring instead of global memory,
// so every output is bitwise what k_gemv and k_step return.  A lane's chunks
// are the same in every row of a phase, so when they number at most kXR their
// activations are loaded once per phase and kept in registers.
//
// Every wait is bounded: an mbarrier wait gives up after spin_limit * 64 ns,
// a grid-barrier poll after spin_limit polls; either records kErrTimeout and
// raises the CTA's abort flag, after which the consumers run through the rest
// of the work list without waiting, computing or storing (keeping every named
// barrier matched), and the producer stops issuing and waits (bounded) for
// the copies it has in flight before it exits.
#include "step_common.cuh"

namespace dg {

namespace {

constexpr int kXR = kRingXR;  // activation chunks per lane kept in registers
constexpr int kConsumerBar = 15;  // named barrier of the consumer warps
// Rows are dealt to slots in groups of group_rows(ks) consecutive rows (about
// 12 KB of fp16 weights), so a phase of a few rows per CTA occupies a few
// warps and each pays the phase's set-up once per group, not once per row.
constexpr int kGroupRows = 4;
__host__ __device__ constexpr int group_rows(int ks) { return ks < kGroupRows ? kGroupRows / ks : 1; }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
// A waiting thread is suspended until the phase completes or about 0.5 ms
// pass (so a wait costs a few instructions, not a spin).
__device__ __forceinline__ bool mbar_try_wait(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity), "r"(500000u)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
                 : "memory");
}
// Adds `bytes` to the transaction count of the current phase (no arrival).
__device__ __forceinline__ void mbar_add_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(bytes)
                 : "memory");
}
// Linear global -> shared copy completing `bytes` transaction bytes on the
// mbarrier; the weights are read once per step, so they go first out of L2.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t mbar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(mbar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint4 lds16(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ void consumers_sync(int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(kConsumerBar), "r"(nthreads) : "memory");
}

// Bounded wait for the completion of the mbarrier phase of parity `parity`.
// Gives up (false) when the CTA's abort flag is up or, after budget_ns, raises
// it and records the timeout.
__device__ __forceinline__ bool ring_wait(uint32_t a, uint32_t parity, uint64_t budget_ns,
                                          int* err, volatile int* abort) {
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(a, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > budget_ns) {
            atomicExch(err, kErrTimeout);
            *abort = 1;
            return false;
        }
    }
}

// Grid barrier among the consumer warps (the producer never joins one).
// bar[0] counts CTA arrivals over the launch; barrier e completes at e * G.
__device__ __forceinline__ void consumer_grid_barrier(const StepParams& sp, unsigned target,
                                                      int nthreads, volatile int* abort) {
    consumers_sync(nthreads);
    if (threadIdx.x == 0 && !*abort) {
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(sp.bar) : "memory");
        for (unsigned n = 0; ld_acquire_gpu(sp.bar) < target; ++n) {
            if (n >= sp.spin_limit) {
                atomicExch(sp.err, kErrTimeout);
                *abort = 1;
                break;
            }
            __nanosleep(32);
        }
        __threadfence();
    }
    consumers_sync(nthreads);
}

// Where rows land in the ring.  A CTA's rows form one stream (its slice of
// phase 0, then of phase 1, ...); stages are filled with consecutive rows of
// the stream across fused matrices and phases, a row never split: a row that
// does not fit the rest of a stage starts the next one.  `cs` is the index
// (over the launch) of the stage being filled and `used` its bytes so far.
// Producer and consumers evaluate the same closed forms.
struct Pack {
    unsigned cs;
    uint32_t used;
};

// Row q of a phase with row bytes rb, T = SB / rb rows per empty stage, whose
// first row goes after `pk`: stage index and byte offset in the stage.
__device__ __forceinline__ void row_pos(const Pack& pk, uint32_t SB, uint32_t rb, int T, int q,
                                        unsigned& stage, uint32_t& off) {
    const int cap0 = pk.used ? div_floor_small((int)(SB - pk.used), (int)rb) : T;  // rows left in stage cs
    if (q < cap0) {
        stage = pk.cs;
        off = pk.used + (uint32_t)q * rb;
    } else {
        const int q2 = q - cap0, k = div_floor_small(q2, T);
        stage = pk.cs + 1 + (unsigned)k;
        off = (uint32_t)(q2 - k * T) * rb;
    }
}

// The cursor after a phase of n rows.
__device__ __forceinline__ Pack pack_after(const Pack& pk, uint32_t SB, uint32_t rb, int T, int n) {
    if (n <= 0) return pk;
    unsigned st;
    uint32_t off;
    row_pos(pk, SB, rb, T, n - 1, st, off);
    return Pack{st, off + rb};
}

// A warp's rows of one phase are q = q0, q0 + slots, ...: their places in the
// ring advanced without division (row_pos once per phase).
struct RowWalk {
    unsigned st;   // stage of the current row
    int idx;       // row index within its stage's run of this phase's rows
    bool first;    // in the stage the phase started in (rows after `used`)
    int cap0, T, slots;
    uint32_t used, rb;

    __device__ __forceinline__ RowWalk(const Pack& pk, uint32_t SB, uint32_t rb_, int T_, int q0,
                                       int slots_)
        : T(T_), slots(slots_), used(pk.used), rb(rb_) {
        cap0 = pk.used ? div_floor_small((int)(SB - pk.used), (int)rb_) : T_;
        if (q0 < cap0) {
            st = pk.cs;
            idx = q0;
            first = true;
        } else {
            const int q2 = q0 - cap0, k = div_floor_small(q2, T_);
            st = pk.cs + 1 + (unsigned)k;
            idx = q2 - k * T_;
            first = false;
        }
    }
    __device__ __forceinline__ uint32_t off() const { return (first ? used : 0u) + (uint32_t)idx * rb; }
    __device__ __forceinline__ void next() {
        idx += slots;
        if (first) {
            if (idx < cap0) return;
            idx -= cap0;
            ++st;
            first = false;
        }
        while (idx >= T) {
            idx -= T;
            ++st;
        }
    }
};

// Stages a launch fills in total.
__device__ __forceinline__ unsigned pack_stages(const Pack& pk) { return pk.cs + (pk.used ? 1u : 0u); }

// The lane's share of one row (weights at shared address w), activations in
// registers: chunk j of the lane is (j * ks + kw) * 32 + lane, j < nl.
template <bool BF16>
__device__ __forceinline__ float row_dot_cached(uint32_t w, const uint4 (&xr)[kXR], int nl, int c0,
                                                int step) {
    using P = PolicyFP<BF16>;
    float acc[1] = {0.f};
    // three shared-memory loads in flight at a time (ascending j throughout)
#pragma unroll
    for (int jb = 0; jb < kXR; jb += 3) {
        typename P::Chunk ch[3];
#pragma unroll
        for (int u = 0; u < 3; ++u)
            if (jb + u < nl) ch[u].w = lds16(w + (uint32_t)(c0 + (jb + u) * step) * 16u);
#pragma unroll
        for (int u = 0; u < 3; ++u)
            if (jb + u < nl) P::mac_direct(acc, ch[u], xr[jb + u]);
    }
    return acc[0];
}

// The same for rows with more than kXR chunks per lane: activations read from
// global memory (L1) with the weights, four chunks at a time.
template <bool BF16>
__device__ __forceinline__ float row_dot_stream(uint32_t w, const void* x, bool coherent,
                                                int nchunks, int c0, int step) {
    using P = PolicyFP<BF16>;
    constexpr int U = 4;
    float acc[1] = {0.f};
    for (int c = c0; c < nchunks; c += U * step) {
        typename P::Chunk ch[U];
        uint4 xv[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (c + u * step < nchunks) {
                ch[u].w = lds16(w + (uint32_t)(c + u * step) * 16u);
                xv[u] = P::load_x(x, c + u * step, coherent);
            }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (c + u * step < nchunks) P::mac_direct(acc, ch[u], xv[u]);
    }
    return acc[0];
}

// Adds the slot's warps' row sums in kw order into warp kw == 0 (the order
// row_group uses).  Every warp of the slot calls it, whatever it computed.
__device__ __forceinline__ float slot_reduce(float acc, int* red, int warp, int ks, int kw,
                                             int lane) {
    if (ks == 1) return acc;
    if (lane == 0) red[warp] = __float_as_int(acc);
    const int bar = slot_barrier(warp, ks);
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(ks * 32) : "memory");
    if (kw == 0)
        for (int j = 1; j < ks; ++j) acc += __int_as_float(red[warp + j]);
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(ks * 32) : "memory");
    return acc;
}

// What a consumer warp needs to walk the ring (shared addresses).
struct RingView {
    uint32_t ring;   // stage 0
    uint32_t full;   // full[0]; full[s] at full + 8 s
    uint32_t empty;  // empty[0]
    int* red;        // slot reduction scratch
    volatile int* abort;
    uint32_t SB;
    int NS;
    uint64_t budget_ns;
};

// A consumer warp's place in the ring: every stage before `vs` is released;
// `have`: the warp has waited for stage vs (and `ok`: the wait succeeded).
// A warp visits every stage in order, waits for it to be full and arrives on
// its empty barrier exactly once, whether or not it had rows there.
// slot = vs % NS and par = (vs / NS) & 1 are kept incrementally.
struct Cursor {
    unsigned vs, slot, par;
    bool have, ok;
};

__device__ __forceinline__ bool cursor_wait(Cursor& c, const RingView& rv, int* err) {
    const bool ok = !*rv.abort && ring_wait(rv.full + 8u * c.slot, c.par, rv.budget_ns, err, rv.abort);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void cursor_release(Cursor& c, const RingView& rv, int* err) {
    if (!c.have) (void)cursor_wait(c, rv, err);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(rv.empty + 8u * c.slot);
    ++c.vs;
    if (++c.slot == (unsigned)rv.NS) {
        c.slot = 0;
        c.par ^= 1u;
    }
    c.have = false;
}

// Moves the cursor to stage `st` (releasing the stages before it) and waits
// for it; returns whether its data can be used.
__device__ __forceinline__ bool cursor_acquire(Cursor& c, unsigned st, const RingView& rv, int* err) {
    while (c.vs < st) cursor_release(c, rv, err);
    if (!c.have) {
        c.ok = cursor_wait(c, rv, err);
        c.have = true;
    }
    return c.ok;
}

// One consumer warp's rows of one phase: groups mine, mine + slots, ... of
// gr consecutive rows of the CTA's slice, each row read from its place in the
// ring.  CACHED: the phase's activation chunks of this lane live in xr: read
// from the ring (kPhaseXRing: the activation vector precedes the rows in the
// stream, as one more row) or loaded by the caller; otherwise they are read
// with the weights.
template <bool BF16, bool CACHED>
__device__ __forceinline__ void consume_phase(const StepParams& sp, const StepPhase& ph,
                                              const RingView& rv, Cursor& cur, const Pack& pk,
                                              int r0, int n, int gr, int mine, int slots, int warp,
                                              uint4 (&xr)[kXR], float& best_v, int& best_i) {
    using P = PolicyFP<BF16>;
    const int ng = (n + gr - 1) / gr;
    if (mine >= ng) return;
    const int lane = threadIdx.x & 31;
    const int ks = ph.ks, kw = warp % ks;
    const int nchunks = ph.K / 8, step = ks * 32, c0 = kw * 32 + lane;
    const int nl = c0 < nchunks ? (nchunks - c0 + step - 1) / step : 0;
    const bool coherent = (ph.flags & kPhaseXWritten) != 0;
    const bool head = (ph.flags & kPhaseHead) != 0;
    const uint32_t rb = (uint32_t)ph.K * 2u;
    const int T = div_floor_small((int)rv.SB, (int)rb);
    int xoff = 0;  // stream index of row 0
    if constexpr (CACHED) {
        if (ph.flags & kPhaseXRing) {
            unsigned st;
            uint32_t off;
            row_pos(pk, rv.SB, rb, T, 0, st, off);
            if (cursor_acquire(cur, st, rv, sp.err)) {
                const uint32_t xs = rv.ring + cur.slot * rv.SB + off + (uint32_t)c0 * 16u;
#pragma unroll
                for (int j = 0; j < kXR; ++j)
                    if (j < nl) xr[j] = lds16(xs + (uint32_t)(j * step) * 16u);
            }
            xoff = 1;
        }
    }
    // output segment of the current row (parameters read when it changes)
    int sg = 0, seg_end = ph.nseg > 1 ? ph.seg[1].row_begin : ph.N;
    for (int g = mine; g < ng; g += slots) {
        const int q0 = g * gr, q1 = min(n, q0 + gr);
        RowWalk rw(pk, rv.SB, rb, T, q0 + xoff, 1);
        for (int q = q0; q < q1; ++q) {
            const bool ok = cursor_acquire(cur, rw.st, rv, sp.err);
            const uint32_t w = rv.ring + cur.slot * rv.SB + rw.off();
            float acc = 0.f;
            if (ok) {
                if constexpr (CACHED)
                    acc = row_dot_cached<BF16>(w, xr, nl, c0, step);
                else
                    acc = row_dot_stream<BF16>(w, ph.x, coherent, nchunks, c0, step);
            }
            acc = warp_sum(acc);
            acc = slot_reduce(acc, rv.red, warp, ks, kw, lane);
            const int r = r0 + q;
            while (r >= seg_end) {
                ++sg;
                seg_end = sg + 1 < ph.nseg ? ph.seg[sg + 1].row_begin : ph.N;
            }
            if (ok && kw == 0 && lane == 0) {
                if (head) {
                    ph.logits[r] = acc;
                    if (arg_better(acc, r, best_v, best_i)) {
                        best_v = acc;
                        best_i = r;
                    }
                } else {
                    RowRef rr{};
                    rr.y = ph.seg[sg].y;
                    rr.local = r - ph.seg[sg].row_begin;
                    P::store(rr, 0, acc, 1.f);
                }
            }
            rw.next();
        }
    }
}

// What the producer needs of a phase, read from the kernel parameters two
// phases ahead of use: the first read of a phase's parameters on an SM misses
// the constant cache and waits for L2, in dependent rounds, which a small
// phase (a few rows per CTA) cannot hide.  Loading the next phases while the
// current one streams also warms the lines for the consumer warps (ks is read
// for that reason only).
struct PhaseDesc {
    const unsigned char* W[kMaxSeg];
    const void* x;
    int rbeg[kMaxSeg];
    int N, K, nseg, flags, ks;
};

// Element i of a descriptor array with constant indices only (the
// descriptors must stay in registers: a dynamic index would put them in local
// memory, and storing a parameter load there waits for it).
template <typename T>
__device__ __forceinline__ T pick(const T (&a)[kMaxSeg], int i) {
    return i == 0 ? a[0] : i == 1 ? a[1] : i == 2 ? a[2] : a[3];
}

__device__ __forceinline__ void load_desc(PhaseDesc& d, const StepPhase& ph) {
#pragma unroll
    for (int i = 0; i < kMaxSeg; ++i) {
        d.W[i] = static_cast<const unsigned char*>(ph.seg[i].W);
        d.rbeg[i] = ph.seg[i].row_begin;
    }
    d.x = ph.x;
    d.N = ph.N;
    d.K = ph.K;
    d.nseg = ph.nseg;
    d.flags = ph.flags;
    d.ks = ph.ks;
}

}  // namespace

template <bool BF16, int NC>
__global__ void __launch_bounds__((NC + 1) * 32, 1) k_step_ring(const __grid_constant__ StepParams sp) {
    using P = PolicyFP<BF16>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int NS = sp.nstage;
    const uint32_t SB = (uint32_t)sp.stage_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const uint64_t budget_ns = (uint64_t)sp.spin_limit * 64u;

    // shared memory: ring | phase table | full[NS] | empty[NS] | red[NC] |
    // best[NC] | abort
    const uint32_t ring = smem_addr(smem);
    PhaseSlice* table = reinterpret_cast<PhaseSlice*>(smem + (size_t)NS * SB);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * SB + kPhaseTableBytes);
    uint64_t* empty = full + NS;
    int* red = reinterpret_cast<int*>(empty + NS);
    ArgPart* cta_best = reinterpret_cast<ArgPart*>(red + NC);
    volatile int* abort = reinterpret_cast<volatile int*>(cta_best + NC);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_addr(full + s), 1);
            mbar_init(smem_addr(empty + s), NC);
        }
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // per-phase slices and the dealing of row groups (group_rows(ks) rows)
    plan_phases(sp, table, b, G,
                [](const StepPhase& ph, int n) { return (n + group_rows(ph.ks) - 1) / group_rows(ph.ks); });

    if (warp == NC) {
        // ---- producer: one thread copies the CTA's row stream into the ring,
        // one bulk copy per run of rows of one matrix within one stage; the
        // stage (cs), its slot and parity and the rows still fitting in it are
        // kept incrementally
        if (lane != 0) return;
        const uint64_t policy = evict_first_policy();
        unsigned cs = 0, slot = 0, par = 0;
        uint32_t used = 0;
        bool open = false, run = true;
        PhaseDesc d0{}, d1{}, d2{};  // phases p, p + 1, p + 2
        if (sp.nphase > 0) load_desc(d0, sp.ph[0]);
        if (sp.nphase > 1) load_desc(d1, sp.ph[1]);
        for (int p = 0; p < sp.nphase && run; ++p) {
            if (p + 2 < sp.nphase) load_desc(d2, sp.ph[p + 2]);
            const PhaseDesc& ph = d0;
            const int r0 = table[p].r0, n = table[p].n;
            const uint32_t rb = (uint32_t)ph.K * 2u;
            const int T = div_floor_small((int)SB, (int)rb);
            int left = open ? div_floor_small((int)(SB - used), (int)rb) : 0;  // rows that still fit
            // kPhaseXRing: the activation vector goes first, as one more row
            const int xoff = (ph.flags & kPhaseXRing) ? 1 : 0, nn = n > 0 ? n + xoff : 0;
            int sg = 0;
#pragma unroll
            for (int i = 1; i < kMaxSeg; ++i)
                if (i < ph.nseg && r0 >= ph.rbeg[i]) sg = i;
            int seg_end = sg + 1 < ph.nseg ? pick(ph.rbeg, sg + 1) : ph.N;
            const unsigned char* seg_w = pick(ph.W, sg) + (size_t)(r0 - pick(ph.rbeg, sg)) * rb;
            for (int q = 0; q < nn;) {
                if (left == 0) {  // close the stage, wait for the next slot
                    if (open) {
                        mbar_arrive(smem_addr(full + slot));
                        ++cs;
                        if (++slot == (unsigned)NS) {
                            slot = 0;
                            par ^= 1u;
                        }
                    }
                    if (!ring_wait(smem_addr(empty + slot), par ^ 1u, budget_ns, sp.err, abort)) {
                        open = false;
                        run = false;
                        break;
                    }
                    open = true;
                    used = 0;
                    left = T;
                }
                const uint32_t fb = smem_addr(full + slot);
                if (q < xoff) {  // the activations
                    mbar_add_tx(fb, rb);
                    bulk_copy_g2s(ring + slot * SB + used, ph.x, rb, fb, policy);
                    used += rb;
                    --left;
                    ++q;
                    continue;
                }
                const int r = r0 + q - xoff;
                if (r >= seg_end) {  // the next fused matrix
                    ++sg;
                    seg_end = sg + 1 < ph.nseg ? pick(ph.rbeg, sg + 1) : ph.N;
                    seg_w = pick(ph.W, sg);
                }
                const int rows = min(min(left, seg_end - r), nn - q);
                const uint32_t bytes = (uint32_t)rows * rb;
                mbar_add_tx(fb, bytes);
                bulk_copy_g2s(ring + slot * SB + used, seg_w, bytes, fb, policy);
                seg_w += bytes;
                used += bytes;
                left -= rows;
                q += rows;
            }
            d0 = d1;
            d1 = d2;
        }
        if (open) mbar_arrive(smem_addr(full + slot));
        // no copy may still be writing this CTA's shared memory when it exits:
        // wait for the last stage of every slot that received copies (after an
        // abort, stage cs was never acquired; stages before it all were)
        const unsigned filled = run ? (open ? cs + 1 : 0u) : cs;
        for (unsigned j = 0; j < (unsigned)NS && j < filled; ++j) {
            const unsigned last = filled - 1 - ((filled - 1 - j) % NS);  // last stage in slot j
            const uint32_t a = smem_addr(full + j);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(a, (last / NS) & 1u))
                if (global_ns() - t0 > budget_ns) {
                    atomicExch(sp.err, kErrTimeout);
                    break;
                }
        }
        return;
    }

    // ---- consumers
    const RingView rv{ring, smem_addr(full), smem_addr(empty), red, abort, SB, NS, budget_ns};
    const int nthreads = NC * 32;
    unsigned nbar = 0;
    Pack pk{0, 0};
    Cursor cur{0, 0, 0, false, false};
    for (int p = 0; p < sp.nphase; ++p) {
        const StepPhase& ph = sp.ph[p];
        if (p > 0 && (ph.flags & kPhaseBarrier)) {
            // stages before the cursor hold only earlier rows: release them
            // first, or the producer could wait on this warp while another warp
            // of the CTA waits for data before the barrier
            while (cur.vs < pk.cs) cursor_release(cur, rv, sp.err);
            ++nbar;
            consumer_grid_barrier(sp, nbar * G, nthreads, abort);
            if ((sp.ph[p - 1].flags & kPhaseHead) && b == 0 && warp == 0 && !*abort)
                reduce_token(sp.part, G, sp.ph[p - 1].token);
        }
        const int ks = ph.ks;
        const int slots = NC / ks;  // warps past slots * ks take no rows (ks = 8)
        const int slot = warp / ks, kw = warp - slot * ks;
        const bool idle = slot >= slots;
        const int nchunks = ph.K / 8, step = ks * 32, c0 = kw * 32 + lane;
        const PhaseSlice sl = table[p];
        const int r0 = sl.r0, n = sl.n;
        // groups of rows are dealt round-robin over the whole step (continuing
        // where the previous phase stopped) so every slot streams a fair share
        const int gr = group_rows(ks);
        const int lead = mod_slots<NC>(sl.deal0, ks);
        // an idle warp's first group is past the phase's last
        const int mine = idle ? (n + gr - 1) / gr : slot >= lead ? slot - lead : slot - lead + slots;
        const bool head = (ph.flags & kPhaseHead) != 0;
        float best_v = NAN;
        int best_i = INT_MAX;
        uint4 xr[kXR];
        if ((nchunks + step - 1) / step <= kXR) {
            if (!(ph.flags & kPhaseXRing) && !*abort && mine * gr < n) {
                const int nl = c0 < nchunks ? (nchunks - c0 + step - 1) / step : 0;
                const bool coherent = (ph.flags & kPhaseXWritten) != 0;
#pragma unroll
                for (int j = 0; j < kXR; ++j)
                    if (j < nl) xr[j] = P::load_x(ph.x, c0 + j * step, coherent);
            }
            consume_phase<BF16, true>(sp, ph, rv, cur, pk, r0, n, gr, mine, slots, warp, xr,
                                      best_v, best_i);
        } else {
            consume_phase<BF16, false>(sp, ph, rv, cur, pk, r0, n, gr, mine, slots, warp, xr,
                                       best_v, best_i);
        }
        const uint32_t rb = (uint32_t)ph.K * 2u;
        const int nn = n > 0 ? n + ((ph.flags & kPhaseXRing) ? 1 : 0) : 0;
        pk = pack_after(pk, SB, rb, div_floor_small((int)SB, (int)rb), nn);
        if (head) {
            while (cur.vs < pk.cs) cursor_release(cur, rv, sp.err);
            if (lane == 0) {
                cta_best[warp].v = best_v;
                cta_best[warp].i = best_i;
            }
            consumers_sync(nthreads);
            if (threadIdx.x == 0) {
                float bv = NAN;
                int bi = INT_MAX;
                for (int w = 0; w < NC; ++w)
                    if (arg_better(cta_best[w].v, cta_best[w].i, bv, bi)) {
                        bv = cta_best[w].v;
                        bi = cta_best[w].i;
                    }
                sp.part[b].v = bv;
                sp.part[b].i = bi;
            }
        }
    }
    // every warp releases the rest of the ring (the producer waits for it)
    const unsigned total = pack_stages(pk);
    while (cur.vs < total) cursor_release(cur, rv, sp.err);

    if (sp.ph[sp.nphase - 1].flags & kPhaseHead) {
        ++nbar;
        consumer_grid_barrier(sp, nbar * G, nthreads, abort);
        if (b == 0 && warp == 0 && !*abort) reduce_token(sp.part, G, sp.ph[sp.nphase - 1].token);
    }
}

size_t step_ring_overhead(int nc) {
    // phase table, full + empty barriers for up to 16 stages, red, best, abort
    return kPhaseTableBytes + (size_t)2 * 16 * 8 + (size_t)nc * 4 + (size_t)nc * sizeof(ArgPart) +
           16;
}

template <bool BF16, int NC>
static cudaError_t ring_run(const StepParams* sp, int grid, size_t smem, cudaStream_t s, int* occ) {
    auto fn = k_step_ring<BF16, NC>;
    constexpr int threads = (NC + 1) * 32;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, threads, smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<StepParams*>(sp)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(fn), args);
}

cudaError_t step_ring_launch(Fmt f, const StepParams* sp, int grid, size_t smem, cudaStream_t s,
                             int* occ, int nc) {
    const bool bf = f == F_BF16;
    if (f != F_F16 && f != F_BF16) return cudaErrorInvalidValue;
    if (nc == 8) return bf ? ring_run<true, 8>(sp, grid, smem, s, occ)
                           : ring_run<false, 8>(sp, grid, smem, s, occ);
    if (nc == 12) return bf ? ring_run<true, 12>(sp, grid, smem, s, occ)
                            : ring_run<false, 12>(sp, grid, smem, s, occ);
    return cudaErrorInvalidValue;
}

}  // namespace dg
