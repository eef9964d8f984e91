// common.cuh -- configuration, kernel parameter blocks, Philox4x32-10, the
// bf16 roundings, the AdamW element update and the streaming memory primitives
// shared by every kernel of the library.
// Included by asr.cu inside its anonymous namespace (one translation unit).

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
