// asr.cu -- GB300 (sm_103a) kernels and C-ABI entry points for the fused AdamW
// step with Philox-keyed stochastic rounding to bf16.
//
// What is computed follows two pages:
//   "Add stochastic rounding and philox RNG helpers" (FlyDSL PR 907), section
//     Primitives: stochastic rounding f32 -> bf16 by adding random bits below
//     the kept mantissa and truncating; a Philox 4x32 counter-based generator
//     that feeds it from a global index and a seed.
//   "adamw-sr", introduction and sections Method / Correctness: decoupled
//     weight decay Adam fused into one memory pass per parameter, bf16
//     write-back by stochastic rounding, randomness keyed by (seed, step) and
//     indexed by the element's global parameter position, so shards carrying
//     a base_index give the same bits as the whole tensor.
//
// Design (GB300): the step is a streaming pass, 22 bytes per element for bf16
// params/grads with f32 moments, far below the ALU ridge, so the kernels are
// built for HBM bandwidth: 128-bit coalesced loads/stores, eight elements per
// thread-unit, two units in flight per thread, a persistent grid sized to the
// SM count times the resident CTAs per SM, grid-striding over tiles of a
// tensor table passed by value (__grid_constant__) so that one launch covers
// a whole model.  Philox runs in registers, one 10-round call per four
// elements, with the ten round keys precomputed on the host and read from the
// constant bank.  Every float operation is an explicitly rounded IEEE binary32
// intrinsic in a fixed order, so results are bit-reproducible.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <memory>
#include <mutex>
#include <unordered_map>

#include "asr.h"

namespace {

// ------------------------------------------------------------------ config

#ifndef ASR_THREADS
#define ASR_THREADS 128
#endif
#ifndef ASR_UNROLL
#define ASR_UNROLL 2
#endif
#ifndef ASR_MIN_BLOCKS
#define ASR_MIN_BLOCKS 1
#endif
constexpr int kThreads = ASR_THREADS;       // threads per CTA
constexpr int kVec = 8;                     // elements per unit (one 16 B bf16 vector)
constexpr int kUnroll = ASR_UNROLL;         // units per thread per tile
constexpr int kTile = kThreads * kVec * kUnroll;   // 2048 elements per tile
constexpr int kCapLarge = 512;              // descriptors per multi-tensor launch
constexpr int kCapSmall = 1;                // single-tensor launch

// Philox4x32-10 constants (Salmon et al., SC'11; cuRAND's Philox4_32_10).
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// --------------------------------------------------------- kernel params

// The ten round keys of one seed: round r uses (k0 + r*W0, k1 + r*W1).
struct RoundKeys {
    uint32_t k0[10];
    uint32_t k1[10];
};

struct StepScalars {
    float b1, b2, eps, decay, omb1, omb2, step_size, bc2s;
};

struct AdamParams {
    StepScalars s;
    RoundKeys keys;
    uint32_t step;
};

struct TensorEntry {
    void *p;
    const void *g;
    float *m;
    float *v;
    uint64_t n;
    uint64_t base;
    uint64_t tile_end;      // exclusive end of this tensor's tiles in the launch
};

template <int CAP>
struct AdamTable {
    uint64_t total_tiles;
    int32_t count;
    int32_t pad;
    TensorEntry t[CAP];
};

static_assert(sizeof(AdamTable<kCapLarge>) + sizeof(AdamParams) <= 32000,
              "kernel parameters must fit the 32 KB parameter space");

// ----------------------------------------------------------- device math

__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              const RoundKeys &K, uint32_t out[4])
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = static_cast<uint64_t>(kPhiloxM0) * c0;
        const uint64_t p1 = static_cast<uint64_t>(kPhiloxM1) * c2;
        const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ K.k0[r];
        const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ K.k1[r];
        c1 = static_cast<uint32_t>(p1);
        c3 = static_cast<uint32_t>(p0);
        c0 = n0;
        c2 = n2;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

// Words of the counter (q lo, q hi, step, 0).
__device__ __forceinline__ void philox_q(uint64_t q, uint32_t step, const RoundKeys &K, uint32_t out[4])
{
    philox4x32_10(static_cast<uint32_t>(q), static_cast<uint32_t>(q >> 32), step, 0u, K, out);
}

__device__ __forceinline__ bool f32_bits_nan(uint32_t u) { return (u & 0x7FFFFFFFu) > 0x7F800000u; }

// Stochastic rounding: keep the top half of (bits + low 16 random bits).  A
// NaN keeps sign and top payload with the quiet bit forced.
__device__ __forceinline__ uint32_t round_sr(float x, uint32_t r)
{
    const uint32_t u = __float_as_uint(x);
    const uint32_t rounded = (u + (r & 0xFFFFu)) >> 16;
    return f32_bits_nan(u) ? ((u >> 16) | 0x0040u) : rounded;
}

__device__ __forceinline__ uint32_t round_rne(float x)
{
    const uint32_t u = __float_as_uint(x);
    const uint32_t rounded = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    return f32_bits_nan(u) ? ((u >> 16) | 0x0040u) : rounded;
}

// One AdamW element in the fixed binary32 order.
__device__ __forceinline__ float adamw_elem(float p, float g, float &m, float &v, const StepScalars &s)
{
    const float p1 = __fmul_rn(p, s.decay);
    const float m1 = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
    const float v1 = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v1), s.bc2s), s.eps);
    const float pn = __fsub_rn(p1, __fmul_rn(s.step_size, __fdiv_rn(m1, den)));
    m = m1;
    v = v1;
    return pn;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(uint32_t lo, uint32_t hi) { return __byte_perm(lo, hi, 0x5410); }

// Which rounding route each kernel takes (both give identical bits):
// the AdamW kernels use the integer add-and-truncate, measured 1.5 % faster
// there on GB300 (6,562 vs 6,463 GB/s on the 8B set, same run) because they
// are close to issue-bound; the stand-alone rounding op, purely
// memory-bound, uses the hardware conversion.
#ifndef ASR_ADAMW_CVT_RS
#define ASR_ADAMW_CVT_RS 0
#endif
#ifndef ASR_SR_OP_CVT_RS
#define ASR_SR_OP_CVT_RS 1
#endif

// Two stochastically rounded bf16 values packed into one word (lo in bits
// 15:0).  HW: Blackwell's cvt.rs.bf16x2.f32 rounds its first operand into the
// high half with rbits[31:16] and its second into the low half with
// rbits[15:0]; for every non-NaN input it gives exactly the add-and-truncate
// result (checked on GB300 over all 2^32 patterns x all 2^16 random values in
// both lanes).  It turns every NaN into 0x7FFF, so a pair holding a NaN takes
// the integer path, which keeps the NaN rule of round_sr.
template <bool HW>
__device__ __forceinline__ uint32_t sr_pack2(float lo, float hi, uint32_t rlo, uint32_t rhi)
{
    if (HW) {
        uint32_t d;
        asm("cvt.rs.bf16x2.f32 %0, %1, %2, %3;" : "=r"(d) : "f"(hi), "f"(lo), "r"(__byte_perm(rlo, rhi, 0x5410)));
        if (__builtin_expect(isnan(lo) || isnan(hi), 0)) d = pack_bf16(round_sr(lo, rlo), round_sr(hi, rhi));
        return d;
    }
    return pack_bf16(round_sr(lo, rlo), round_sr(hi, rhi));
}

// Selects r[k] = w[s + k] for k < 8 from 12 words, s in 0..3, with static
// register indices only.
__device__ __forceinline__ void shift_words(const uint32_t w[12], uint32_t s, uint32_t r[8])
{
    uint32_t t[10];
#pragma unroll
    for (int k = 0; k < 10; ++k) t[k] = (s & 1u) ? w[k + 1] : w[k];
#pragma unroll
    for (int k = 0; k < 8; ++k) r[k] = (s & 2u) ? t[k + 2] : t[k];
}

// The eight random words of local elements e..e+7 of a tensor whose element 0
// has global index base.  With base % 4 == 0 and e % 8 == 0 the unit covers
// exactly two counters.
template <bool ALIGNED4>
__device__ __forceinline__ void unit_words(uint64_t base, uint64_t e, uint32_t step, const RoundKeys &K,
                                           uint32_t r[8])
{
    const uint64_t i0 = base + e;
    const uint64_t q = i0 >> 2;
    if (ALIGNED4) {
        philox_q(q, step, K, r);
        philox_q(q + 1, step, K, r + 4);
    } else {
        uint32_t w[12];
        philox_q(q, step, K, w);
        philox_q(q + 1, step, K, w + 4);
        philox_q(q + 2, step, K, w + 8);
        shift_words(w, static_cast<uint32_t>(i0 & 3u), r);
    }
}

// ----------------------------------------------------- memory primitives

// Streaming 128-bit accesses: every byte is touched once, so keep it out of
// L1 and mark it evict-first in L2.
__device__ __forceinline__ uint4 ld_stream(const void *p) { return __ldcs(reinterpret_cast<const uint4 *>(p)); }
#ifndef ASR_STORE_CS
#define ASR_STORE_CS 1
#endif
#if ASR_STORE_CS
__device__ __forceinline__ void st_stream(void *p, uint4 v) { __stcs(reinterpret_cast<uint4 *>(p), v); }
#else
__device__ __forceinline__ void st_stream(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }
#endif

// ------------------------------------------------------------ AdamW unit

// Vector unit: eight elements at local offset e, all in range, all pointers
// 16-byte aligned.  Loads are split from compute so a thread keeps several
// units' loads in flight.
template <int PT, int GT>
struct VecUnit {
    uint32_t p[PT == ASR_BF16 ? 4 : 8];
    uint32_t g[GT == ASR_BF16 ? 4 : 8];
    float m[8];
    float v[8];
};

template <int PT, int GT>
__device__ __forceinline__ void vec_load(const TensorEntry &T, uint64_t e, VecUnit<PT, GT> &u)
{
    if (PT == ASR_BF16) {
        const uint4 a = ld_stream(static_cast<const uint16_t *>(T.p) + e);
        u.p[0] = a.x; u.p[1] = a.y; u.p[2] = a.z; u.p[3] = a.w;
    } else {
        const float *pp = static_cast<const float *>(T.p) + e;
        const uint4 a = ld_stream(pp), b = ld_stream(pp + 4);
        u.p[0] = a.x; u.p[1] = a.y; u.p[2] = a.z; u.p[3] = a.w;
        u.p[4] = b.x; u.p[5] = b.y; u.p[6] = b.z; u.p[7] = b.w;
    }
    if (GT == ASR_BF16) {
        const uint4 a = ld_stream(static_cast<const uint16_t *>(T.g) + e);
        u.g[0] = a.x; u.g[1] = a.y; u.g[2] = a.z; u.g[3] = a.w;
    } else {
        const float *gp = static_cast<const float *>(T.g) + e;
        const uint4 a = ld_stream(gp), b = ld_stream(gp + 4);
        u.g[0] = a.x; u.g[1] = a.y; u.g[2] = a.z; u.g[3] = a.w;
        u.g[4] = b.x; u.g[5] = b.y; u.g[6] = b.z; u.g[7] = b.w;
    }
    {
        const uint4 a = ld_stream(T.m + e), b = ld_stream(T.m + e + 4);
        u.m[0] = __uint_as_float(a.x); u.m[1] = __uint_as_float(a.y);
        u.m[2] = __uint_as_float(a.z); u.m[3] = __uint_as_float(a.w);
        u.m[4] = __uint_as_float(b.x); u.m[5] = __uint_as_float(b.y);
        u.m[6] = __uint_as_float(b.z); u.m[7] = __uint_as_float(b.w);
    }
    {
        const uint4 a = ld_stream(T.v + e), b = ld_stream(T.v + e + 4);
        u.v[0] = __uint_as_float(a.x); u.v[1] = __uint_as_float(a.y);
        u.v[2] = __uint_as_float(a.z); u.v[3] = __uint_as_float(a.w);
        u.v[4] = __uint_as_float(b.x); u.v[5] = __uint_as_float(b.y);
        u.v[6] = __uint_as_float(b.z); u.v[7] = __uint_as_float(b.w);
    }
}

template <int PT, int GT>
__device__ __forceinline__ float vec_p(const VecUnit<PT, GT> &u, int k)
{
    if (PT == ASR_BF16) return (k & 1) ? bf16_hi(u.p[k >> 1]) : bf16_lo(u.p[k >> 1]);
    return __uint_as_float(u.p[k]);
}

template <int PT, int GT>
__device__ __forceinline__ float vec_g(const VecUnit<PT, GT> &u, int k)
{
    if (GT == ASR_BF16) return (k & 1) ? bf16_hi(u.g[k >> 1]) : bf16_lo(u.g[k >> 1]);
    return __uint_as_float(u.g[k]);
}

template <int PT, int GT, int RM>
__device__ __forceinline__ void vec_compute_store(const TensorEntry &T, uint64_t e, VecUnit<PT, GT> &u,
                                                  const AdamParams &P)
{
    float pn[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) pn[k] = adamw_elem(vec_p(u, k), vec_g(u, k), u.m[k], u.v[k], P.s);

    if (PT == ASR_BF16) {
        uint32_t w[4];
        if (RM == ASR_ROUND_SR) {
            uint32_t r[8];
            unit_words<true>(T.base, e, P.step, P.keys, r);
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = sr_pack2<ASR_ADAMW_CVT_RS>(pn[2 * k], pn[2 * k + 1], r[2 * k], r[2 * k + 1]);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = pack_bf16(round_rne(pn[2 * k]), round_rne(pn[2 * k + 1]));
        }
        st_stream(static_cast<uint16_t *>(T.p) + e, make_uint4(w[0], w[1], w[2], w[3]));
    } else {
        float *pp = static_cast<float *>(T.p) + e;
        st_stream(pp, make_uint4(__float_as_uint(pn[0]), __float_as_uint(pn[1]), __float_as_uint(pn[2]),
                                 __float_as_uint(pn[3])));
        st_stream(pp + 4, make_uint4(__float_as_uint(pn[4]), __float_as_uint(pn[5]), __float_as_uint(pn[6]),
                                     __float_as_uint(pn[7])));
    }
    st_stream(T.m + e, make_uint4(__float_as_uint(u.m[0]), __float_as_uint(u.m[1]), __float_as_uint(u.m[2]),
                                  __float_as_uint(u.m[3])));
    st_stream(T.m + e + 4, make_uint4(__float_as_uint(u.m[4]), __float_as_uint(u.m[5]),
                                      __float_as_uint(u.m[6]), __float_as_uint(u.m[7])));
    st_stream(T.v + e, make_uint4(__float_as_uint(u.v[0]), __float_as_uint(u.v[1]), __float_as_uint(u.v[2]),
                                  __float_as_uint(u.v[3])));
    st_stream(T.v + e + 4, make_uint4(__float_as_uint(u.v[4]), __float_as_uint(u.v[5]),
                                      __float_as_uint(u.v[6]), __float_as_uint(u.v[7])));
}

// Scalar unit: local elements e..min(e+8, n)-1, any alignment, any base.
template <int PT, int GT, int RM>
__device__ __forceinline__ void scalar_unit(const TensorEntry &T, uint64_t e, const AdamParams &P)
{
    uint32_t r[8];
    if (PT == ASR_BF16 && RM == ASR_ROUND_SR) unit_words<false>(T.base, e, P.step, P.keys, r);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint64_t j = e + k;
        if (j >= T.n) break;
        const float p = PT == ASR_BF16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(T.p)[j]) << 16)
                                       : static_cast<const float *>(T.p)[j];
        const float g = GT == ASR_BF16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(T.g)[j]) << 16)
                                       : static_cast<const float *>(T.g)[j];
        float m = T.m[j], v = T.v[j];
        const float pn = adamw_elem(p, g, m, v, P.s);
        T.m[j] = m;
        T.v[j] = v;
        if (PT == ASR_BF16) {
            const uint32_t h = RM == ASR_ROUND_SR ? round_sr(pn, r[k]) : round_rne(pn);
            static_cast<uint16_t *>(T.p)[j] = static_cast<uint16_t>(h);
        } else {
            static_cast<float *>(T.p)[j] = pn;
        }
    }
}

// Persistent grid-stride kernel over the tiles of every tensor in the table.
// FAST: every tensor has 16-byte-aligned buffers and base % 4 == 0.
template <int PT, int GT, int RM, bool FAST, int CAP>
__global__ void __launch_bounds__(kThreads, ASR_MIN_BLOCKS)
adamw_sr_kernel(const __grid_constant__ AdamTable<CAP> tab, const __grid_constant__ AdamParams P)
{
    int t = 0;
    for (uint64_t tile = blockIdx.x; tile < tab.total_tiles; tile += gridDim.x) {
        while (tile >= tab.t[t].tile_end) ++t;
        const TensorEntry &T = tab.t[t];
        const uint64_t first = t == 0 ? 0 : tab.t[t - 1].tile_end;
        const uint64_t off = (tile - first) * static_cast<uint64_t>(kTile);
        if (FAST && off + kTile <= T.n) {
            VecUnit<PT, GT> u[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k)
                vec_load(T, off + (static_cast<uint64_t>(k) * kThreads + threadIdx.x) * kVec, u[k]);
#pragma unroll
            for (int k = 0; k < kUnroll; ++k)
                vec_compute_store<PT, GT, RM>(T, off + (static_cast<uint64_t>(k) * kThreads + threadIdx.x) * kVec,
                                              u[k], P);
        } else {
#pragma unroll 1
            for (int k = 0; k < kUnroll; ++k) {
                const uint64_t e = off + (static_cast<uint64_t>(k) * kThreads + threadIdx.x) * kVec;
                if (e >= T.n) break;
                if (FAST && e + kVec <= T.n) {
                    VecUnit<PT, GT> one;
                    vec_load(T, e, one);
                    vec_compute_store<PT, GT, RM>(T, e, one, P);
                } else {
                    scalar_unit<PT, GT, RM>(T, e, P);
                }
            }
        }
    }
}

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
#ifndef ASR_TMA_CONSUMER_WARPS
#define ASR_TMA_CONSUMER_WARPS 20
#endif
#ifndef ASR_TMA_SMEM_KB
#define ASR_TMA_SMEM_KB 200
#endif
#ifndef ASR_TMA_EVICT_FIRST
#define ASR_TMA_EVICT_FIRST 1
#endif
#ifndef ASR_TMA_TILE
#define ASR_TMA_TILE 5120
#endif
constexpr int kTmaTile = ASR_TMA_TILE;
constexpr int kTmaConsumerWarps = ASR_TMA_CONSUMER_WARPS;
constexpr int kTmaConsumers = kTmaConsumerWarps * 32;
constexpr int kTmaThreads = kTmaConsumers + 32;        // + one producer warp
constexpr int kTmaUnits = kTmaTile / kVec / kTmaConsumers;   // units per consumer thread per tile
static_assert(kTmaUnits >= 1 && kTmaUnits * kTmaConsumers * kVec == kTmaTile, "tile must split evenly");
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

template <int PT, int GT>
struct TmaStage {
    static constexpr int kPBytes = kTmaTile * (PT == ASR_BF16 ? 2 : 4);
    static constexpr int kGBytes = kTmaTile * (GT == ASR_BF16 ? 2 : 4);
    static constexpr int kMBytes = kTmaTile * 4;
    static constexpr int kBytes = kPBytes + kGBytes + 2 * kMBytes;
    // as many stages as fit in the shared-memory budget, at most ASR_TMA_STAGES
    static constexpr int kFit = ASR_TMA_SMEM_KB * 1024 / kBytes;
    static constexpr int kStages = kFit < ASR_TMA_STAGES ? kFit : ASR_TMA_STAGES;
    static_assert(kStages >= 2, "need at least two stages");
    static constexpr int kSmem = kStages * kBytes + 2 * kStages * 8 + kTmaConsumerWarps * 4;
};

// Locate tile `tile` of the table, advancing the cursor t.
template <int CAP>
__device__ __forceinline__ void find_tile(const AdamTable<CAP> &tab, uint64_t tile, int &t, uint64_t &off,
                                          uint32_t &cnt)
{
    while (tile >= tab.t[t].tile_end) ++t;
    const uint64_t first = t == 0 ? 0 : tab.t[t - 1].tile_end;
    off = (tile - first) * static_cast<uint64_t>(kTmaTile);
    const uint64_t rest = tab.t[t].n - off;
    cnt = rest < static_cast<uint64_t>(kTmaTile) ? static_cast<uint32_t>(rest) : static_cast<uint32_t>(kTmaTile);
}

// All tensors FAST (16-byte-aligned buffers, base % 4 == 0); tile size kTmaTile.
template <int PT, int GT, int RM, int CAP>
__global__ void __launch_bounds__(kTmaThreads, 1)
adamw_sr_tma_kernel(const __grid_constant__ AdamTable<CAP> tab, const __grid_constant__ AdamParams P,
                    uint64_t limit_ns)
{
    using S = TmaStage<PT, GT>;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bars = sbase + S::kStages * S::kBytes;      // full[s] then empty[s]
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (S::kStages + s); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kTmaConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == kTmaConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane != 0) return;
        uint64_t policy;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
        int t = 0;
        uint32_t k = 0;
        for (uint64_t tile = blockIdx.x; tile < tab.total_tiles; tile += gridDim.x, ++k) {
            const int s = static_cast<int>(k % S::kStages);
            const uint32_t use = k / S::kStages;
            if (use > 0 && !mbar_wait(empty(s), (use - 1) & 1u, limit_ns)) break;
            uint64_t off;
            uint32_t cnt;
            find_tile(tab, tile, t, off, cnt);
            const TensorEntry &T = tab.t[t];
            const uint32_t c8 = cnt & ~7u;
            const uint32_t pb = c8 * (PT == ASR_BF16 ? 2u : 4u), gb = c8 * (GT == ASR_BF16 ? 2u : 4u);
            const uint32_t mb = c8 * 4u;
            mbar_arrive_expect_tx(full(s), pb + gb + 2 * mb);
            if (c8) {
                const uint32_t dst = sbase + s * S::kBytes;
                bulk_load(dst, static_cast<const unsigned char *>(T.p) + off * (PT == ASR_BF16 ? 2 : 4), pb,
                          full(s), policy);
                bulk_load(dst + S::kPBytes, static_cast<const unsigned char *>(T.g) + off * (GT == ASR_BF16 ? 2 : 4),
                          gb, full(s), policy);
                bulk_load(dst + S::kPBytes + S::kGBytes, T.m + off, mb, full(s), policy);
                bulk_load(dst + S::kPBytes + S::kGBytes + S::kMBytes, T.v + off, mb, full(s), policy);
            }
        }
        // Every copy this thread issued must land before the CTA may exit:
        // wait (bounded) for the last use of each stage.
        const uint32_t issued = k;
        for (int s = 0; s < S::kStages; ++s) {
            if (static_cast<uint32_t>(s) >= issued) break;
            const uint32_t last_use = (issued - 1 - s) / S::kStages;
            mbar_wait(full(s), last_use & 1u, limit_ns);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ct = threadIdx.x;            // 0 .. kTmaConsumers-1
    const uint32_t dep_slot = bars + 16u * S::kStages + 4u * warp;   // one word per consumer warp
    int t = 0;
    uint32_t k = 0;
    for (uint64_t tile = blockIdx.x; tile < tab.total_tiles; tile += gridDim.x, ++k) {
        const int s = static_cast<int>(k % S::kStages);
        const uint32_t use = k / S::kStages;
        if (!mbar_wait(full(s), use & 1u, limit_ns)) return;
        uint64_t off;
        uint32_t cnt;
        find_tile(tab, tile, t, off, cnt);
        const TensorEntry &T = tab.t[t];
        const uint32_t c8 = cnt & ~7u;
        const unsigned char *st = smem + s * S::kBytes;
        VecUnit<PT, GT> u[kTmaUnits];
#pragma unroll
        for (int j = 0; j < kTmaUnits; ++j) {
            const uint32_t e = (static_cast<uint32_t>(j) * kTmaConsumers + ct) * kVec;
            if (e < c8) {
                if (PT == ASR_BF16) {
                    const uint4 a = *reinterpret_cast<const uint4 *>(st + e * 2);
                    u[j].p[0] = a.x; u[j].p[1] = a.y; u[j].p[2] = a.z; u[j].p[3] = a.w;
                } else {
                    const uint4 a = *reinterpret_cast<const uint4 *>(st + e * 4);
                    const uint4 b = *reinterpret_cast<const uint4 *>(st + e * 4 + 16);
                    u[j].p[0] = a.x; u[j].p[1] = a.y; u[j].p[2] = a.z; u[j].p[3] = a.w;
                    u[j].p[4] = b.x; u[j].p[5] = b.y; u[j].p[6] = b.z; u[j].p[7] = b.w;
                }
                const unsigned char *gs = st + S::kPBytes;
                if (GT == ASR_BF16) {
                    const uint4 a = *reinterpret_cast<const uint4 *>(gs + e * 2);
                    u[j].g[0] = a.x; u[j].g[1] = a.y; u[j].g[2] = a.z; u[j].g[3] = a.w;
                } else {
                    const uint4 a = *reinterpret_cast<const uint4 *>(gs + e * 4);
                    const uint4 b = *reinterpret_cast<const uint4 *>(gs + e * 4 + 16);
                    u[j].g[0] = a.x; u[j].g[1] = a.y; u[j].g[2] = a.z; u[j].g[3] = a.w;
                    u[j].g[4] = b.x; u[j].g[5] = b.y; u[j].g[6] = b.z; u[j].g[7] = b.w;
                }
                const float4 *ms = reinterpret_cast<const float4 *>(st + S::kPBytes + S::kGBytes + e * 4);
                const float4 *vs = reinterpret_cast<const float4 *>(st + S::kPBytes + S::kGBytes + S::kMBytes + e * 4);
                const float4 m0 = ms[0], m1 = ms[1], v0 = vs[0], v1 = vs[1];
                u[j].m[0] = m0.x; u[j].m[1] = m0.y; u[j].m[2] = m0.z; u[j].m[3] = m0.w;
                u[j].m[4] = m1.x; u[j].m[5] = m1.y; u[j].m[6] = m1.z; u[j].m[7] = m1.w;
                u[j].v[0] = v0.x; u[j].v[1] = v0.y; u[j].v[2] = v0.z; u[j].v[3] = v0.w;
                u[j].v[4] = v1.x; u[j].v[5] = v1.y; u[j].v[6] = v1.z; u[j].v[7] = v1.w;
            }
        }
        // Hand the stage back only once this warp's shared-memory loads have
        // returned (the next bulk copy into the stage would otherwise race
        // with a load still queued): every lane folds one register of each
        // 128-bit load into `dep` and stores it; in-order issue holds that
        // store, and so the warp barrier and the release after it, until
        // every folded load is back.
        uint32_t dep = 0;
#pragma unroll
        for (int j = 0; j < kTmaUnits; ++j) {
            const uint32_t e = (static_cast<uint32_t>(j) * kTmaConsumers + ct) * kVec;
            if (e < c8)
                dep ^= u[j].p[0] ^ u[j].g[0] ^ __float_as_uint(u[j].m[0]) ^ __float_as_uint(u[j].m[4]) ^
                       __float_as_uint(u[j].v[0]) ^ __float_as_uint(u[j].v[4]) ^
                       (PT == ASR_BF16 ? 0u : u[j].p[4]) ^ (GT == ASR_BF16 ? 0u : u[j].g[4]);
        }
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(dep_slot), "r"(dep) : "memory");
        __syncwarp();
        if (lane == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(empty(s));
        }
#pragma unroll
        for (int j = 0; j < kTmaUnits; ++j) {
            const uint32_t e = (static_cast<uint32_t>(j) * kTmaConsumers + ct) * kVec;
            if (e < c8) vec_compute_store<PT, GT, RM>(T, off + e, u[j], P);
        }
        // a ragged end of a tensor (< 8 elements) goes through the scalar path
        if (c8 < cnt && ct == (c8 / kVec) % kTmaConsumers) scalar_unit<PT, GT, RM>(T, off + c8, P);
    }
}

// ------------------------------------------------------- SR and Philox ops

struct SrParams {
    const float *x;
    const uint32_t *rbits;
    uint16_t *out;
    uint64_t n;
    uint64_t base;
    uint32_t step;
    RoundKeys keys;
};

// FAST: x/out (and rbits) 16-byte aligned, base % 4 == 0.
template <bool FAST, bool RBITS>
__global__ void __launch_bounds__(kThreads) sr_bf16_kernel(const __grid_constant__ SrParams P)
{
    const uint64_t units = (P.n + kVec - 1) / kVec;
    for (uint64_t unit = blockIdx.x * static_cast<uint64_t>(kThreads) + threadIdx.x; unit < units;
         unit += static_cast<uint64_t>(gridDim.x) * kThreads) {
        const uint64_t e = unit * kVec;
        uint32_t r[8];
        if (FAST && e + kVec <= P.n) {
            const uint4 a = ld_stream(P.x + e), b = ld_stream(P.x + e + 4);
            if (RBITS) {
                const uint4 ra = ld_stream(P.rbits + e), rb = ld_stream(P.rbits + e + 4);
                r[0] = ra.x; r[1] = ra.y; r[2] = ra.z; r[3] = ra.w;
                r[4] = rb.x; r[5] = rb.y; r[6] = rb.z; r[7] = rb.w;
            } else {
                unit_words<true>(P.base, e, P.step, P.keys, r);
            }
            const uint32_t xs[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                w[k] = sr_pack2<ASR_SR_OP_CVT_RS>(__uint_as_float(xs[2 * k]), __uint_as_float(xs[2 * k + 1]), r[2 * k],
                                                  r[2 * k + 1]);
            st_stream(P.out + e, make_uint4(w[0], w[1], w[2], w[3]));
        } else {
            if (!RBITS) unit_words<false>(P.base, e, P.step, P.keys, r);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t j = e + k;
                if (j >= P.n) break;
                const uint32_t rw = RBITS ? P.rbits[j] : r[k];
                P.out[j] = static_cast<uint16_t>(round_sr(P.x[j], rw));
            }
        }
    }
}

struct PhiloxParams {
    uint32_t *out;
    uint64_t n_ctr;
    uint64_t ctr_base;
    uint32_t ctr2, ctr3;
    RoundKeys keys;
};

template <bool ALIGNED16>
__global__ void __launch_bounds__(kThreads) philox_kernel(const __grid_constant__ PhiloxParams P)
{
    for (uint64_t j = blockIdx.x * static_cast<uint64_t>(kThreads) + threadIdx.x; j < P.n_ctr;
         j += static_cast<uint64_t>(gridDim.x) * kThreads) {
        const uint64_t c = P.ctr_base + j;
        uint32_t w[4];
        philox4x32_10(static_cast<uint32_t>(c), static_cast<uint32_t>(c >> 32), P.ctr2, P.ctr3, P.keys, w);
        if (ALIGNED16) {
            st_stream(P.out + 4 * j, make_uint4(w[0], w[1], w[2], w[3]));
        } else {
            P.out[4 * j] = w[0];
            P.out[4 * j + 1] = w[1];
            P.out[4 * j + 2] = w[2];
            P.out[4 * j + 3] = w[3];
        }
    }
}

// ------------------------------------------------------------- host side

thread_local int g_last_cuda_error = 0;

asr_status cuda_fail(cudaError_t e)
{
    g_last_cuda_error = static_cast<int>(e);
    return ASR_ERR_CUDA;
}

RoundKeys make_keys(uint64_t seed)
{
    RoundKeys K;
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        K.k0[r] = k0;
        K.k1[r] = k1;
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    return K;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Persistent grid: SMs x resident CTAs per SM of this kernel, cached per
// (device, kernel).
std::mutex g_grid_mu;
std::unordered_map<uint64_t, int> g_grid_cache;

template <typename K>
asr_status persistent_grid(K kernel, int *grid)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const uint64_t key = (static_cast<uint64_t>(dev) << 48) ^ reinterpret_cast<uintptr_t>(kernel);
    {
        std::lock_guard<std::mutex> lk(g_grid_mu);
        auto it = g_grid_cache.find(key);
        if (it != g_grid_cache.end()) {
            *grid = it->second;
            return ASR_OK;
        }
    }
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    if (per_sm < 1) per_sm = 1;
    *grid = sms * per_sm;
    std::lock_guard<std::mutex> lk(g_grid_mu);
    g_grid_cache[key] = *grid;
    return ASR_OK;
}

asr_status check_launch()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ASR_OK : cuda_fail(e);
}

bool finite_nonneg(double x) { return std::isfinite(x) && x >= 0.0; }

asr_status validate_hparams(const asr_adamw_hparams *hp)
{
    if (!hp) return ASR_ERR_INVALID_VALUE;
    if (hp->rounding != ASR_ROUND_SR && hp->rounding != ASR_ROUND_RNE) return ASR_ERR_UNSUPPORTED_DTYPE;
    if (hp->step == 0) return ASR_ERR_INVALID_VALUE;
    if (!finite_nonneg(hp->lr) || !finite_nonneg(hp->eps) || !finite_nonneg(hp->weight_decay))
        return ASR_ERR_INVALID_VALUE;
    if (!(hp->beta1 >= 0.0 && hp->beta1 < 1.0) || !(hp->beta2 >= 0.0 && hp->beta2 < 1.0))
        return ASR_ERR_INVALID_VALUE;
    return ASR_OK;
}

// Scalars in binary64, each rounded once to binary32.  Host code is compiled
// with contraction off so 1 - lr*wd is two roundings in binary64 as written.
StepScalars make_scalars(const asr_adamw_hparams &hp)
{
    const double t = static_cast<double>(hp.step);
    StepScalars s;
    s.b1 = static_cast<float>(hp.beta1);
    s.b2 = static_cast<float>(hp.beta2);
    s.eps = static_cast<float>(hp.eps);
    s.decay = static_cast<float>(1.0 - hp.lr * hp.weight_decay);
    s.omb1 = static_cast<float>(1.0 - hp.beta1);
    s.omb2 = static_cast<float>(1.0 - hp.beta2);
    s.step_size = static_cast<float>(hp.lr / (1.0 - std::pow(hp.beta1, t)));
    s.bc2s = static_cast<float>(std::sqrt(1.0 - std::pow(hp.beta2, t)));
    return s;
}

asr_status validate_desc(const asr_tensor_desc &d)
{
    if (d.param_dtype != ASR_F32 && d.param_dtype != ASR_BF16) return ASR_ERR_UNSUPPORTED_DTYPE;
    if (d.grad_dtype != ASR_F32 && d.grad_dtype != ASR_BF16) return ASR_ERR_UNSUPPORTED_DTYPE;
    if (d.n == 0) return ASR_OK;
    if (!d.param || !d.grad || !d.exp_avg || !d.exp_avg_sq) return ASR_ERR_INVALID_VALUE;
    if (d.n > (UINT64_MAX >> 4)) return ASR_ERR_INVALID_VALUE;
    if (d.base_index > UINT64_MAX - d.n) return ASR_ERR_INVALID_VALUE;
    // element alignment of each buffer
    const uintptr_t pa = d.param_dtype == ASR_BF16 ? 1 : 3, ga = d.grad_dtype == ASR_BF16 ? 1 : 3;
    if ((reinterpret_cast<uintptr_t>(d.param) & pa) || (reinterpret_cast<uintptr_t>(d.grad) & ga) ||
        (reinterpret_cast<uintptr_t>(d.exp_avg) & 3) || (reinterpret_cast<uintptr_t>(d.exp_avg_sq) & 3))
        return ASR_ERR_INVALID_VALUE;
    return ASR_OK;
}

bool desc_fast(const asr_tensor_desc &d)
{
    return aligned16(d.param) && aligned16(d.grad) && aligned16(d.exp_avg) && aligned16(d.exp_avg_sq) &&
           (d.base_index & 3u) == 0;
}

#ifndef ASR_USE_TMA
#define ASR_USE_TMA 1
#endif

// Dynamic shared memory opt-in and persistent grid of the bulk-copy kernel,
// cached per (device, kernel).
template <typename K>
asr_status tma_grid(K kernel, int smem, int *grid)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const uint64_t key = (static_cast<uint64_t>(dev) << 48) ^ reinterpret_cast<uintptr_t>(kernel) ^ 1u;
    {
        std::lock_guard<std::mutex> lk(g_grid_mu);
        auto it = g_grid_cache.find(key);
        if (it != g_grid_cache.end()) {
            *grid = it->second;
            return ASR_OK;
        }
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail(e);
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kTmaThreads, smem);
    if (e != cudaSuccess) return cuda_fail(e);
    if (per_sm < 1) per_sm = 1;
    *grid = sms * per_sm;
    std::lock_guard<std::mutex> lk(g_grid_mu);
    g_grid_cache[key] = *grid;
    return ASR_OK;
}

template <int PT, int GT, int RM, bool FAST, int CAP>
asr_status launch_group(const asr_tensor_desc *const *descs, int count, const AdamParams &P, cudaStream_t stream)
{
    static_assert(CAP >= 1, "");
    constexpr bool kTma = FAST && ASR_USE_TMA;
    constexpr uint64_t tile = kTma ? kTmaTile : kTile;
    AdamTable<CAP> tab;
    std::memset(&tab, 0, sizeof(tab));
    uint64_t tiles = 0;
    for (int i = 0; i < count; ++i) {
        const asr_tensor_desc &d = *descs[i];
        TensorEntry &T = tab.t[i];
        T.p = d.param;
        T.g = d.grad;
        T.m = d.exp_avg;
        T.v = d.exp_avg_sq;
        T.n = d.n;
        T.base = d.base_index;
        tiles += (d.n + tile - 1) / tile;
        T.tile_end = tiles;
    }
    tab.total_tiles = tiles;
    tab.count = count;
    if (tiles == 0) return ASR_OK;
    int grid = 0;
    asr_status st;
    if (kTma) {
        auto kernel = adamw_sr_tma_kernel<PT, GT, RM, CAP>;
        const int smem = TmaStage<PT, GT>::kSmem;
        st = tma_grid(kernel, smem, &grid);
        if (st != ASR_OK) return st;
        if (static_cast<uint64_t>(grid) > tiles) grid = static_cast<int>(tiles);
        kernel<<<grid, kTmaThreads, smem, stream>>>(tab, P, kWaitLimitNs);
    } else {
        auto kernel = adamw_sr_kernel<PT, GT, RM, FAST, CAP>;
        st = persistent_grid(kernel, &grid);
        if (st != ASR_OK) return st;
        if (static_cast<uint64_t>(grid) > tiles) grid = static_cast<int>(tiles);
        kernel<<<grid, kThreads, 0, stream>>>(tab, P);
    }
    return check_launch();
}

template <int PT, int GT, int RM, bool FAST>
asr_status launch_chunks(const asr_tensor_desc *const *descs, int count, const AdamParams &P, cudaStream_t stream)
{
    if (count == 1) return launch_group<PT, GT, RM, FAST, kCapSmall>(descs, 1, P, stream);
    for (int s = 0; s < count; s += kCapLarge) {
        const int c = count - s < kCapLarge ? count - s : kCapLarge;
        asr_status st = launch_group<PT, GT, RM, FAST, kCapLarge>(descs + s, c, P, stream);
        if (st != ASR_OK) return st;
    }
    return ASR_OK;
}

template <int PT, int GT, int RM>
asr_status dispatch_fast(const asr_tensor_desc *const *descs, int count, bool fast, const AdamParams &P,
                         cudaStream_t stream)
{
    return fast ? launch_chunks<PT, GT, RM, true>(descs, count, P, stream)
                : launch_chunks<PT, GT, RM, false>(descs, count, P, stream);
}

asr_status dispatch(const asr_tensor_desc *const *descs, int count, int pdt, int gdt, int rm, bool fast,
                    const AdamParams &P, cudaStream_t stream)
{
    if (pdt == ASR_BF16) {
        if (gdt == ASR_BF16)
            return rm == ASR_ROUND_SR ? dispatch_fast<ASR_BF16, ASR_BF16, ASR_ROUND_SR>(descs, count, fast, P, stream)
                                      : dispatch_fast<ASR_BF16, ASR_BF16, ASR_ROUND_RNE>(descs, count, fast, P, stream);
        return rm == ASR_ROUND_SR ? dispatch_fast<ASR_BF16, ASR_F32, ASR_ROUND_SR>(descs, count, fast, P, stream)
                                  : dispatch_fast<ASR_BF16, ASR_F32, ASR_ROUND_RNE>(descs, count, fast, P, stream);
    }
    // f32 params are stored as computed: the rounding mode does not apply.
    if (gdt == ASR_BF16) return dispatch_fast<ASR_F32, ASR_BF16, ASR_ROUND_SR>(descs, count, fast, P, stream);
    return dispatch_fast<ASR_F32, ASR_F32, ASR_ROUND_SR>(descs, count, fast, P, stream);
}

asr_status run_adamw(const asr_tensor_desc *table, int32_t n_tensors, const asr_adamw_hparams *hp,
                     cudaStream_t stream)
{
    asr_status st = validate_hparams(hp);
    if (st != ASR_OK) return st;
    if (n_tensors < 0 || (n_tensors > 0 && !table)) return ASR_ERR_INVALID_VALUE;
    for (int32_t i = 0; i < n_tensors; ++i) {
        st = validate_desc(table[i]);
        if (st != ASR_OK) return st;
    }
    AdamParams P;
    P.s = make_scalars(*hp);
    P.keys = make_keys(hp->seed);
    P.step = hp->step;

    // Group by (param dtype, grad dtype, vector eligibility), keeping order.
    // Every element is independent, so the grouping cannot change any bit.
    const int nt = n_tensors;
    const asr_tensor_desc **sel = nullptr;
    const asr_tensor_desc *one[1];
    std::unique_ptr<const asr_tensor_desc *[]> holder;
    if (nt <= 1) {
        sel = one;
    } else {
        holder.reset(new const asr_tensor_desc *[nt]);
        sel = holder.get();
    }
    for (int pdt = 0; pdt < 2; ++pdt)
        for (int gdt = 0; gdt < 2; ++gdt)
            for (int f = 0; f < 2; ++f) {
                int c = 0;
                for (int i = 0; i < nt; ++i) {
                    const asr_tensor_desc &d = table[i];
                    if (d.n == 0 || d.param_dtype != pdt || d.grad_dtype != gdt || desc_fast(d) != (f == 1))
                        continue;
                    sel[c++] = &d;
                }
                if (c == 0) continue;
                st = dispatch(sel, c, pdt, gdt, static_cast<int>(hp->rounding), f == 1, P, stream);
                if (st != ASR_OK) return st;
            }
    return ASR_OK;
}

// ------------------------------------------ allocation-free multi-tensor step
//
// A variant of the bulk-copy pipelined step for callers that must not
// allocate device memory.  Its scratch -- the tensor descriptor table the
// kernel walks -- lives in a file-scope device array owned by the library,
// so one launch per dtype group covers up to kStaticTableMax tensors without
// anyone calling cudaMalloc.  Every device that loads the library holds the
// array until the process exits.  Each call rewrites the part of the array it
// uses, so nothing in it has to start at zero; calls whose kernels overlap on
// the GPU (other streams, other host threads) share the array and race.

constexpr int kStaticTableMax = ASR_STATIC_TABLE_MAX;   // 4096 descriptors x 56 B = 224 KB per device

static __device__ __align__(256) TensorEntry g_static_table[kStaticTableMax];

struct GlobalTable {
    const TensorEntry *t;       // device address inside g_static_table
    uint64_t total_tiles;
};

__device__ __forceinline__ void find_tile(const GlobalTable &tab, uint64_t tile, int &t, uint64_t &off,
                                          uint32_t &cnt)
{
    while (tile >= tab.t[t].tile_end) ++t;
    const uint64_t first = t == 0 ? 0 : tab.t[t - 1].tile_end;
    off = (tile - first) * static_cast<uint64_t>(kTmaTile);
    const uint64_t rest = tab.t[t].n - off;
    cnt = rest < static_cast<uint64_t>(kTmaTile) ? static_cast<uint32_t>(rest) : static_cast<uint32_t>(kTmaTile);
}

// The pipeline of adamw_sr_tma_kernel, with the table read from global memory.
template <int PT, int GT, int RM>
__global__ void __launch_bounds__(kTmaThreads, 1)
adamw_sr_tma_static_kernel(const __grid_constant__ GlobalTable tab, const __grid_constant__ AdamParams P,
                           uint64_t limit_ns)
{
    using S = TmaStage<PT, GT>;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bars = sbase + S::kStages * S::kBytes;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (S::kStages + s); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kTmaConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == kTmaConsumerWarps) {
        if (lane != 0) return;
        uint64_t policy;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
        int t = 0;
        uint32_t k = 0;
        for (uint64_t tile = blockIdx.x; tile < tab.total_tiles; tile += gridDim.x, ++k) {
            const int s = static_cast<int>(k % S::kStages);
            const uint32_t use = k / S::kStages;
            if (use > 0 && !mbar_wait(empty(s), (use - 1) & 1u, limit_ns)) break;
            uint64_t off;
            uint32_t cnt;
            find_tile(tab, tile, t, off, cnt);
            const TensorEntry &T = tab.t[t];
            const uint32_t c8 = cnt & ~7u;
            const uint32_t pb = c8 * (PT == ASR_BF16 ? 2u : 4u), gb = c8 * (GT == ASR_BF16 ? 2u : 4u);
            const uint32_t mb = c8 * 4u;
            mbar_arrive_expect_tx(full(s), pb + gb + 2 * mb);
            if (c8) {
                const uint32_t dst = sbase + s * S::kBytes;
                bulk_load(dst, static_cast<const unsigned char *>(T.p) + off * (PT == ASR_BF16 ? 2 : 4), pb,
                          full(s), policy);
                bulk_load(dst + S::kPBytes, static_cast<const unsigned char *>(T.g) + off * (GT == ASR_BF16 ? 2 : 4),
                          gb, full(s), policy);
                bulk_load(dst + S::kPBytes + S::kGBytes, T.m + off, mb, full(s), policy);
                bulk_load(dst + S::kPBytes + S::kGBytes + S::kMBytes, T.v + off, mb, full(s), policy);
            }
        }
        // every copy issued here must land before the CTA exits
        const uint32_t issued = k;
        for (int s = 0; s < S::kStages; ++s) {
            if (static_cast<uint32_t>(s) >= issued) break;
            const uint32_t last_use = (issued - 1 - s) / S::kStages;
            mbar_wait(full(s), last_use & 1u, limit_ns);
        }
        return;
    }

    const int ct = threadIdx.x;
    const uint32_t dep_slot = bars + 16u * S::kStages + 4u * warp;
    int t = 0;
    uint32_t k = 0;
    for (uint64_t tile = blockIdx.x; tile < tab.total_tiles; tile += gridDim.x, ++k) {
        const int s = static_cast<int>(k % S::kStages);
        const uint32_t use = k / S::kStages;
        if (!mbar_wait(full(s), use & 1u, limit_ns)) return;
        uint64_t off;
        uint32_t cnt;
        find_tile(tab, tile, t, off, cnt);
        const TensorEntry &T = tab.t[t];
        const uint32_t c8 = cnt & ~7u;
        const unsigned char *st = smem + s * S::kBytes;
        VecUnit<PT, GT> u[kTmaUnits];
        uint32_t dep = 0;
#pragma unroll
        for (int j = 0; j < kTmaUnits; ++j) {
            const uint32_t e = (static_cast<uint32_t>(j) * kTmaConsumers + ct) * kVec;
            if (e < c8) {
                if (PT == ASR_BF16) {
                    const uint4 a = *reinterpret_cast<const uint4 *>(st + e * 2);
                    u[j].p[0] = a.x; u[j].p[1] = a.y; u[j].p[2] = a.z; u[j].p[3] = a.w;
                } else {
                    const uint4 a = *reinterpret_cast<const uint4 *>(st + e * 4);
                    const uint4 b = *reinterpret_cast<const uint4 *>(st + e * 4 + 16);
                    u[j].p[0] = a.x; u[j].p[1] = a.y; u[j].p[2] = a.z; u[j].p[3] = a.w;
                    u[j].p[4] = b.x; u[j].p[5] = b.y; u[j].p[6] = b.z; u[j].p[7] = b.w;
                }
                const unsigned char *gs = st + S::kPBytes;
                if (GT == ASR_BF16) {
                    const uint4 a = *reinterpret_cast<const uint4 *>(gs + e * 2);
                    u[j].g[0] = a.x; u[j].g[1] = a.y; u[j].g[2] = a.z; u[j].g[3] = a.w;
                } else {
                    const uint4 a = *reinterpret_cast<const uint4 *>(gs + e * 4);
                    const uint4 b = *reinterpret_cast<const uint4 *>(gs + e * 4 + 16);
                    u[j].g[0] = a.x; u[j].g[1] = a.y; u[j].g[2] = a.z; u[j].g[3] = a.w;
                    u[j].g[4] = b.x; u[j].g[5] = b.y; u[j].g[6] = b.z; u[j].g[7] = b.w;
                }
                const float4 *ms = reinterpret_cast<const float4 *>(st + S::kPBytes + S::kGBytes + e * 4);
                const float4 *vs = reinterpret_cast<const float4 *>(st + S::kPBytes + S::kGBytes + S::kMBytes + e * 4);
                const float4 m0 = ms[0], m1 = ms[1], v0 = vs[0], v1 = vs[1];
                u[j].m[0] = m0.x; u[j].m[1] = m0.y; u[j].m[2] = m0.z; u[j].m[3] = m0.w;
                u[j].m[4] = m1.x; u[j].m[5] = m1.y; u[j].m[6] = m1.z; u[j].m[7] = m1.w;
                u[j].v[0] = v0.x; u[j].v[1] = v0.y; u[j].v[2] = v0.z; u[j].v[3] = v0.w;
                u[j].v[4] = v1.x; u[j].v[5] = v1.y; u[j].v[6] = v1.z; u[j].v[7] = v1.w;
                dep ^= u[j].p[0] ^ u[j].g[0] ^ __float_as_uint(m0.x) ^ __float_as_uint(m1.x) ^
                       __float_as_uint(v0.x) ^ __float_as_uint(v1.x) ^ (PT == ASR_BF16 ? 0u : u[j].p[4]) ^
                       (GT == ASR_BF16 ? 0u : u[j].g[4]);
            }
        }
        // release the stage only after this warp's loads have returned
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(dep_slot), "r"(dep) : "memory");
        __syncwarp();
        if (lane == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(empty(s));
        }
#pragma unroll
        for (int j = 0; j < kTmaUnits; ++j) {
            const uint32_t e = (static_cast<uint32_t>(j) * kTmaConsumers + ct) * kVec;
            if (e < c8) vec_compute_store<PT, GT, RM>(T, off + e, u[j], P);
        }
        if (c8 < cnt && ct == (c8 / kVec) % kTmaConsumers) scalar_unit<PT, GT, RM>(T, off + c8, P);
    }
}

// Per-device set-up of this path, kept in fixed arrays (no allocation): the
// device address of g_static_table -- on the host its name is only a
// stand-in for the symbol, so the address is looked up with
// cudaGetSymbolAddress while the device is current -- and the persistent grid
// of each kernel variant.
constexpr int kMaxDevices = 64;
constexpr int kStaticVariants = 12;        // 6 dtype/rounding combinations x {pipelined, plain}
std::mutex g_static_mu;
TensorEntry *g_static_addr[kMaxDevices];
int g_static_grid[kMaxDevices][kStaticVariants];

asr_status static_device(int *dev_out, TensorEntry **table_out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ASR_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_table);
        if (e != cudaSuccess) return cuda_fail(e);
        g_static_addr[dev] = static_cast<TensorEntry *>(ptr);
    }
    *dev_out = dev;
    *table_out = g_static_addr[dev];
    return ASR_OK;
}

template <typename K>
asr_status static_grid(K kernel, int dev, int slot, int threads, int smem, int *grid)
{
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (g_static_grid[dev][slot] == 0) {
        cudaError_t e = cudaSuccess;
        if (smem > 48 * 1024) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        int sms = 0, per_sm = 0;
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
        if (e != cudaSuccess) return cuda_fail(e);
        g_static_grid[dev][slot] = sms * (per_sm < 1 ? 1 : per_sm);
    }
    *grid = g_static_grid[dev][slot];
    return ASR_OK;
}

constexpr int variant_slot(int pdt, int gdt, int rm) { return pdt == ASR_BF16 ? gdt * 2 + rm : 4 + gdt; }

// Host staging: fixed arrays, guarded by a mutex for the duration of a call.
std::mutex g_stage_mu;
TensorEntry g_stage_table[kStaticTableMax];
AdamTable<kCapLarge> g_stage_plain;

template <int PT, int GT, int RM>
asr_status launch_static_group(int dev, const TensorEntry *dev_table, uint64_t tiles, const AdamParams &P,
                               cudaStream_t stream)
{
    auto kernel = adamw_sr_tma_static_kernel<PT, GT, RM>;
    const int smem = TmaStage<PT, GT>::kSmem;
    int grid = 0;
    asr_status st = static_grid(kernel, dev, variant_slot(PT, GT, RM), kTmaThreads, smem, &grid);
    if (st != ASR_OK) return st;
    if (static_cast<uint64_t>(grid) > tiles) grid = static_cast<int>(tiles);
    GlobalTable tab;
    tab.t = dev_table;
    tab.total_tiles = tiles;
    kernel<<<grid, kTmaThreads, smem, stream>>>(tab, P, kWaitLimitNs);
    return check_launch();
}

// Tensors that are not vector-eligible take the plain kernel, its table in
// the launch parameters (staged in g_stage_plain, kCapLarge per launch).
template <int PT, int GT, int RM>
asr_status launch_static_plain(int dev, const asr_tensor_desc *table, int32_t n_tensors, const AdamParams &P,
                               cudaStream_t stream)
{
    int32_t i = 0;
    int grid = 0;
    while (i < n_tensors) {
        int c = 0;
        uint64_t tiles = 0;
        for (; i < n_tensors && c < kCapLarge; ++i) {
            const asr_tensor_desc &d = table[i];
            if (d.n == 0 || d.param_dtype != PT || d.grad_dtype != GT || desc_fast(d)) continue;
            TensorEntry &T = g_stage_plain.t[c++];
            T.p = d.param;
            T.g = d.grad;
            T.m = d.exp_avg;
            T.v = d.exp_avg_sq;
            T.n = d.n;
            T.base = d.base_index;
            tiles += (d.n + kTile - 1) / kTile;
            T.tile_end = tiles;
        }
        if (c == 0) continue;
        auto kernel = adamw_sr_kernel<PT, GT, RM, false, kCapLarge>;
        if (grid == 0) {
            asr_status st = static_grid(kernel, dev, 6 + variant_slot(PT, GT, RM), kThreads, 0, &grid);
            if (st != ASR_OK) return st;
        }
        g_stage_plain.total_tiles = tiles;
        g_stage_plain.count = c;
        const int g = static_cast<uint64_t>(grid) > tiles ? static_cast<int>(tiles) : grid;
        kernel<<<g, kThreads, 0, stream>>>(g_stage_plain, P);
        asr_status st = check_launch();
        if (st != ASR_OK) return st;
    }
    return ASR_OK;
}

template <int PT, int GT, int RM>
asr_status launch_static_combo(int dev, const TensorEntry *dev_table, uint64_t tiles, bool any_vector,
                               const asr_tensor_desc *table, int32_t n_tensors, const AdamParams &P,
                               cudaStream_t stream)
{
    if (any_vector) {
        asr_status st = launch_static_group<PT, GT, RM>(dev, dev_table, tiles, P, stream);
        if (st != ASR_OK) return st;
    }
    return launch_static_plain<PT, GT, RM>(dev, table, n_tensors, P, stream);
}

asr_status run_adamw_static(const asr_tensor_desc *table, int32_t n_tensors, const asr_adamw_hparams *hp,
                            cudaStream_t stream)
{
    asr_status st = validate_hparams(hp);
    if (st != ASR_OK) return st;
    if (n_tensors < 0 || n_tensors > kStaticTableMax || (n_tensors > 0 && !table)) return ASR_ERR_INVALID_VALUE;
    for (int32_t i = 0; i < n_tensors; ++i) {
        st = validate_desc(table[i]);
        if (st != ASR_OK) return st;
    }
    if (n_tensors == 0) return ASR_OK;
    int dev = 0;
    TensorEntry *dev_table = nullptr;
    st = static_device(&dev, &dev_table);
    if (st != ASR_OK) return st;
    AdamParams P;
    P.s = make_scalars(*hp);
    P.keys = make_keys(hp->seed);
    P.step = hp->step;
    const int rm = static_cast<int>(hp->rounding);

    std::lock_guard<std::mutex> lk(g_stage_mu);
    // Vector-eligible tensors: one contiguous block of the table per dtype
    // group (group index = param dtype * 2 + grad dtype), sent in one copy.
    int used = 0;
    int group_start[4] = {0, 0, 0, 0}, group_count[4] = {0, 0, 0, 0};
    uint64_t group_tiles[4] = {0, 0, 0, 0};
    for (int gi = 0; gi < 4; ++gi) {
        const int pdt = gi / 2, gdt = gi % 2;
        group_start[gi] = used;
        uint64_t tiles = 0;
        for (int32_t i = 0; i < n_tensors; ++i) {
            const asr_tensor_desc &d = table[i];
            if (d.n == 0 || d.param_dtype != pdt || d.grad_dtype != gdt || !desc_fast(d)) continue;
            TensorEntry &T = g_stage_table[used++];
            T.p = d.param;
            T.g = d.grad;
            T.m = d.exp_avg;
            T.v = d.exp_avg_sq;
            T.n = d.n;
            T.base = d.base_index;
            tiles += (d.n + kTmaTile - 1) / kTmaTile;
            T.tile_end = tiles;
        }
        group_count[gi] = used - group_start[gi];
        group_tiles[gi] = tiles;
    }
    if (used > 0) {
        // From pageable host memory: returns once the table is staged for the
        // transfer, which the kernels below follow on the same stream.
        cudaError_t e = cudaMemcpyAsync(dev_table, g_stage_table, sizeof(TensorEntry) * used,
                                        cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    for (int gi = 0; gi < 4; ++gi) {
        const bool any = group_count[gi] > 0;
        const TensorEntry *tb = dev_table + group_start[gi];
        const uint64_t tl = group_tiles[gi];
        if (gi == 3)        // bf16 params, bf16 grads
            st = rm == ASR_ROUND_SR
                ? launch_static_combo<ASR_BF16, ASR_BF16, ASR_ROUND_SR>(dev, tb, tl, any, table, n_tensors, P, stream)
                : launch_static_combo<ASR_BF16, ASR_BF16, ASR_ROUND_RNE>(dev, tb, tl, any, table, n_tensors, P, stream);
        else if (gi == 2)   // bf16 params, f32 grads
            st = rm == ASR_ROUND_SR
                ? launch_static_combo<ASR_BF16, ASR_F32, ASR_ROUND_SR>(dev, tb, tl, any, table, n_tensors, P, stream)
                : launch_static_combo<ASR_BF16, ASR_F32, ASR_ROUND_RNE>(dev, tb, tl, any, table, n_tensors, P, stream);
        else if (gi == 1)   // f32 params, bf16 grads (the rounding mode does not apply)
            st = launch_static_combo<ASR_F32, ASR_BF16, ASR_ROUND_SR>(dev, tb, tl, any, table, n_tensors, P, stream);
        else                // f32 params, f32 grads
            st = launch_static_combo<ASR_F32, ASR_F32, ASR_ROUND_SR>(dev, tb, tl, any, table, n_tensors, P, stream);
        if (st != ASR_OK) return st;
    }
    return ASR_OK;
}

#include "gemm_sr.cuh"

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char *asr_status_string(asr_status status)
{
    switch (status) {
    case ASR_OK: return "ASR_OK: success";
    case ASR_ERR_INVALID_VALUE: return "ASR_ERR_INVALID_VALUE: invalid argument";
    case ASR_ERR_UNSUPPORTED_DTYPE: return "ASR_ERR_UNSUPPORTED_DTYPE: dtype or rounding mode not supported";
    case ASR_ERR_CUDA: return "ASR_ERR_CUDA: the CUDA runtime reported an error";
    }
    return "unknown asr_status";
}

int asr_last_cuda_error(void) { return g_last_cuda_error; }

asr_status asr_selftest_wait_timeout(uint64_t limit_ns, asr_stream_t stream)
{
    if (limit_ns == 0 || limit_ns > kWaitLimitNs) return ASR_ERR_INVALID_VALUE;
    wait_timeout_selftest_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns);
    return check_launch();
}

asr_status asr_take_device_error(uint32_t *bits, asr_stream_t stream)
{
    if (!bits) return ASR_ERR_INVALID_VALUE;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned int h = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&h, g_device_error, sizeof(h), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    *bits = h;
    return ASR_OK;
}

asr_status asr_adamw_prepare(const asr_adamw_hparams *hp, asr_adamw_scalars *out)
{
    asr_status st = validate_hparams(hp);
    if (st != ASR_OK) return st;
    if (!out) return ASR_ERR_INVALID_VALUE;
    const StepScalars s = make_scalars(*hp);
    out->b1 = s.b1;
    out->b2 = s.b2;
    out->eps = s.eps;
    out->decay = s.decay;
    out->omb1 = s.omb1;
    out->omb2 = s.omb2;
    out->step_size = s.step_size;
    out->bc2s = s.bc2s;
    return ASR_OK;
}

asr_status asr_philox4x32(uint32_t *out, uint64_t n_ctr, uint64_t ctr_base, uint32_t ctr2, uint32_t ctr3,
                          uint64_t seed, asr_stream_t stream)
{
    if (n_ctr == 0) return ASR_OK;
    if (!out || n_ctr > (UINT64_MAX >> 4) || (reinterpret_cast<uintptr_t>(out) & 3)) return ASR_ERR_INVALID_VALUE;
    PhiloxParams P;
    P.out = out;
    P.n_ctr = n_ctr;
    P.ctr_base = ctr_base;
    P.ctr2 = ctr2;
    P.ctr3 = ctr3;
    P.keys = make_keys(seed);
    const bool a16 = aligned16(out);
    auto kernel = a16 ? philox_kernel<true> : philox_kernel<false>;
    int grid = 0;
    asr_status st = persistent_grid(kernel, &grid);
    if (st != ASR_OK) return st;
    const uint64_t need = (n_ctr + kThreads - 1) / kThreads;
    if (static_cast<uint64_t>(grid) > need) grid = static_cast<int>(need);
    kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(P);
    return check_launch();
}

asr_status asr_stochastic_round_bf16(const float *x, const uint32_t *rbits, uint16_t *out, uint64_t n,
                                     uint64_t base_index, uint32_t step, uint64_t seed, asr_stream_t stream)
{
    if (n == 0) return ASR_OK;
    if (!x || !out || n > (UINT64_MAX >> 4) || base_index > UINT64_MAX - n) return ASR_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(x) & 3) || (reinterpret_cast<uintptr_t>(out) & 1) ||
        (rbits && (reinterpret_cast<uintptr_t>(rbits) & 3)))
        return ASR_ERR_INVALID_VALUE;
    SrParams P;
    P.x = x;
    P.rbits = rbits;
    P.out = out;
    P.n = n;
    P.base = base_index;
    P.step = step;
    P.keys = make_keys(seed);
    const bool fast = aligned16(x) && aligned16(out) && (!rbits || aligned16(rbits)) && (base_index & 3u) == 0;
    void (*kernel)(const SrParams) = nullptr;
    if (rbits) kernel = fast ? sr_bf16_kernel<true, true> : sr_bf16_kernel<false, true>;
    else kernel = fast ? sr_bf16_kernel<true, false> : sr_bf16_kernel<false, false>;
    int grid = 0;
    asr_status st = persistent_grid(kernel, &grid);
    if (st != ASR_OK) return st;
    const uint64_t need = ((n + kVec - 1) / kVec + kThreads - 1) / kThreads;
    if (static_cast<uint64_t>(grid) > need) grid = static_cast<int>(need);
    kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(P);
    return check_launch();
}

asr_status asr_adamw_sr_step(void *param, int32_t pdt, const void *grad, int32_t gdt, float *exp_avg,
                             float *exp_avg_sq, uint64_t n, uint64_t base_index, const asr_adamw_hparams *hp,
                             asr_stream_t stream)
{
    asr_tensor_desc d;
    d.param = param;
    d.grad = grad;
    d.exp_avg = exp_avg;
    d.exp_avg_sq = exp_avg_sq;
    d.n = n;
    d.base_index = base_index;
    d.param_dtype = pdt;
    d.grad_dtype = gdt;
    return run_adamw(&d, 1, hp, reinterpret_cast<cudaStream_t>(stream));
}

asr_status asr_adamw_sr_multi_tensor(const asr_tensor_desc *table, int32_t n_tensors, const asr_adamw_hparams *hp,
                                     asr_stream_t stream)
{
    return run_adamw(table, n_tensors, hp, reinterpret_cast<cudaStream_t>(stream));
}

asr_status asr_adamw_sr_multi_tensor_static(const asr_tensor_desc *table, int32_t n_tensors,
                                            const asr_adamw_hparams *hp, asr_stream_t stream)
{
    return run_adamw_static(table, n_tensors, hp, reinterpret_cast<cudaStream_t>(stream));
}

asr_status asr_gemm_bf16_sr(const uint16_t *a, const uint16_t *b, uint16_t *c, float *c_f32, uint64_t m, uint64_t n,
                            uint64_t k, uint32_t rounding, uint32_t step, uint64_t seed, asr_stream_t stream)
{
    return gemm::run(a, b, c, c_f32, m, n, k, rounding, step, seed, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
