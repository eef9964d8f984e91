// pipeline.cuh -- the shared-memory pipeline machinery: bulk-copy (TMA)
// configuration, the library's device error word, the bounded mbarrier waits
// and their self-test kernel.
// Included by asr.cu inside its anonymous namespace (one translation unit).

// --------------------------------------------- bulk-copy pipelined kernel
//
// The same step, with the loads taken off the registers: a producer warp
// streams every tile's p, g, m and v into a ring of shared-memory stages with
// cp.async.bulk (the Blackwell/Hopper bulk-copy engine; completion counted on
// an mbarrier), while consumer warps compute from shared memory and store
// their results straight to global memory.  With several 48 KB stages in
// flight per SM the kernel keeps far more bytes outstanding than register
// occupancy allows.
//
// Every mbarrier wait is bounded by a %globaltimer limit; a wait that gives
// up sets a bit in g_device_error, the thread leaves its loop, and the
// producer still waits (bounded) for the copies it issued before exiting.

#ifndef ASR_TMA_STAGES
#define ASR_TMA_STAGES 4
#endif
#ifndef ASR_TMA_SMEM_KB
#define ASR_TMA_SMEM_KB 224
#endif
#ifndef ASR_TMA_EVICT_FIRST
#define ASR_TMA_EVICT_FIRST 1
#endif

// Pipeline shape per (param, grad) dtype: the number of consumer warps, the
// 8-element units per consumer thread per tile, and as many stages (at most
// four) as fit in a 224 KB shared-memory budget.  Measured on GB300 with the
// dynamic tile schedule, all shapes in the same run, two or three repetitions
// (GB/s; bf16/bf16 on the Llama-3-8B set, the others on one 268M-element
// tensor):
//   bf16/bf16: 16 warps x 2 units (8,192-element tiles), 2 stages of 96 KB:
//              7,179-7,183 (24 warps x 1 unit, 3 stages of 72 KB:
//              7,078-7,088; 14 x 2: 6,308; 18 x 2: 7,007; 10 x 3: 5,141;
//              8 x 4: 4,480; 20 x 1 in 200 KB: 6,866-6,905) -- the most
//              arithmetic per byte (Philox and rounding): two independent
//              units per thread beat more warps;
//   bf16/f32:  20 warps, 3 stages: 7,073-7,080 (16: 6,533-6,626; 24: 7,033-7,042);
//   f32/bf16:  16 warps, 4 stages: 7,021-7,031 (12: 6,962-6,968);
//   f32/f32:   12 warps, 4 stages: 7,066-7,075 (16: 7,022).
// Two units per thread lose for the other three (bf16/f32 10 x 2: 5,358,
// 12 x 2: 6,288, 16 x 2: 7,061 against 20 x 1: 7,091; f32/bf16 8 x 2: 5,999,
// 12 x 2: 7,013 against 16 x 1: 7,025; f32/f32 6 x 2: 4,886, 8 x 2: 6,378,
// 12 x 2: 7,004 against 12 x 1: 7,078).
#ifndef ASR_TMA_WARPS_BB
#define ASR_TMA_WARPS_BB 16             // bf16 params, bf16 grads (two units per thread)
#endif
#ifndef ASR_TMA_WARPS_BF
#define ASR_TMA_WARPS_BF 20             // bf16 params, f32 grads
#endif
#ifndef ASR_TMA_WARPS_FB
#define ASR_TMA_WARPS_FB 16             // f32 params, bf16 grads
#endif
#ifndef ASR_TMA_WARPS_FF
#define ASR_TMA_WARPS_FF 12             // f32 params, f32 grads
#endif
#ifndef ASR_TMA_UNITS_BB
#define ASR_TMA_UNITS_BB 2              // units per consumer thread, bf16 params and grads
#endif
#ifndef ASR_TMA_UNITS_BF
#define ASR_TMA_UNITS_BF 1
#endif
#ifndef ASR_TMA_UNITS_FB
#define ASR_TMA_UNITS_FB 1
#endif
#ifndef ASR_TMA_UNITS_FF
#define ASR_TMA_UNITS_FF 1
#endif
template <int PT, int GT>
struct TmaShape {
#ifdef ASR_TMA_WARPS
    static constexpr int kWarps = ASR_TMA_WARPS;            // one shape for all, for sweeps
#else
    static constexpr int kWarps = PT == ASR_BF16 ? (GT == ASR_BF16 ? ASR_TMA_WARPS_BB : ASR_TMA_WARPS_BF)
                                                 : (GT == ASR_BF16 ? ASR_TMA_WARPS_FB : ASR_TMA_WARPS_FF);
#endif
    static constexpr int kConsumers = kWarps * 32;
    static constexpr int kThreads = kConsumers + 32;        // + one producer warp
#ifdef ASR_TMA_UNITS
    static constexpr int kUnits = ASR_TMA_UNITS;            // one shape for all, for sweeps
#else
    // 8-element units per consumer thread per tile
    static constexpr int kUnits = PT == ASR_BF16 ? (GT == ASR_BF16 ? ASR_TMA_UNITS_BB : ASR_TMA_UNITS_BF)
                                                 : (GT == ASR_BF16 ? ASR_TMA_UNITS_FB : ASR_TMA_UNITS_FF);
#endif
    static constexpr int kTile = kConsumers * kVec * kUnits;
};

inline int tma_tile(int pdt, int gdt)
{
    if (pdt == ASR_BF16) return gdt == ASR_BF16 ? TmaShape<ASR_BF16, ASR_BF16>::kTile : TmaShape<ASR_BF16, ASR_F32>::kTile;
    return gdt == ASR_BF16 ? TmaShape<ASR_F32, ASR_BF16>::kTile : TmaShape<ASR_F32, ASR_F32>::kTile;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;       // 2 s: a healthy wait takes microseconds

constexpr uint32_t kErrWaitTimeout = 1u;

__device__ unsigned int g_device_error = 0;

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait until the phase with the given parity has completed, for at most
// limit_ns.  Returns false (and raises the device error bit) on timeout.
// A second guard caps the number of polls, so the wait ends even if the
// timer did not advance.
constexpr uint32_t kWaitMaxPolls = 1u << 26;

__device__ __noinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    const uint64_t t0 = global_ns();
    for (uint32_t polls = 0; !mbar_test(bar, parity); ++polls) {
        if (global_ns() - t0 > limit_ns || polls >= kWaitMaxPolls) {
            atomicOr(&g_device_error, kErrWaitTimeout);
            return false;
        }
    }
    return true;
}


__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_test(bar, parity)) return true;      // fast path: already complete
    return mbar_wait_bounded(bar, parity, limit_ns);
}

// Diagnostic: one thread waits, with the given limit, on a barrier that
// nothing arrives on, so the bounded wait must give up and raise the error
// bit.  Shows that a stuck pipeline ends with a readable status.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(b, 0, limit_ns);
}

// ------------------------------------------------- dynamic tile schedule
//
// Cluster launch control (sm_100 and later): the grid holds one CTA per tile,
// and a running CTA asks the hardware to cancel the launch of a CTA that has
// not started yet and takes that CTA's tile instead.  Each SM thus takes a
// new tile whenever it has room for one, so SMs that the memory system serves
// faster take more tiles, and every SM finishes within a few tiles of the
// others.  No global state is involved, and a tile is processed exactly once
// either way: by its own CTA if that one launches, or by the CTA that
// cancelled it.

// Asks for one not-yet-started CTA; the 16-byte answer lands at `buf` and
// completes 16 bytes of transaction count on `bar`.
__device__ __forceinline__ void clc_try_cancel(uint32_t buf, uint32_t bar)
{
    asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];"
                 ::"r"(buf), "r"(bar)
                 : "memory");
}

// Reads an answer: true, and the cancelled CTA's x index, if a launch was
// cancelled; false once no CTA is left to cancel.
__device__ __forceinline__ bool clc_answer(uint32_t buf, uint32_t &x)
{
    uint32_t ok, cx = 0;
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b128 r;\n\t"
        "ld.shared.b128 r, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t"
        "}"
        : "=r"(ok), "+r"(cx)
        : "r"(buf)
        : "memory");
    x = cx;
    return ok != 0;
}

__device__ __forceinline__ void st_shared_u64(uint32_t addr, uint64_t v)
{
    asm volatile("st.shared.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_shared_u64(uint32_t addr)
{
    uint64_t v;
    asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy)
{
#if ASR_TMA_EVICT_FIRST
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
#else
    (void)policy;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
#endif
}
