// rounding_kernels.cuh -- the stand-alone stochastic-rounding and Philox kernels.
// Included by asr.cu inside its anonymous namespace (one translation unit).

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

// FAST: x/out (and rbits) 16-byte aligned.  A4: base % 4 == 0, so each
// 8-element unit's words come from two Philox counters (three otherwise).
template <bool FAST, bool RBITS, bool A4 = true>
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
                unit_words<A4>(P.base, e, P.step, P.keys, r);
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

// Counters per thread and loop iteration in the aligned case, as independent
// chains: a thread's Philox calls are ten dependent rounds of multiplies, so
// two calls in flight per thread keep the integer-multiply pipe busier (the
// op is bound by that pipe and by its 16-byte stores).
#ifndef ASR_PHILOX_CHAINS
#define ASR_PHILOX_CHAINS 3
#endif
constexpr int kPhiloxChains = ASR_PHILOX_CHAINS;

template <bool ALIGNED16>
__global__ void __launch_bounds__(kThreads) philox_kernel(const __grid_constant__ PhiloxParams P)
{
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
    uint64_t j = blockIdx.x * static_cast<uint64_t>(kThreads) + threadIdx.x;
    // kPhiloxChains counters j, j + stride, ... per iteration while all are in range
    for (; ALIGNED16 && j + (kPhiloxChains - 1) * stride < P.n_ctr; j += kPhiloxChains * stride) {
        uint32_t w[kPhiloxChains][4];
#pragma unroll
        for (int q = 0; q < kPhiloxChains; ++q) {
            const uint64_t c = P.ctr_base + j + q * stride;
            philox4x32_10(static_cast<uint32_t>(c), static_cast<uint32_t>(c >> 32), P.ctr2, P.ctr3, P.keys, w[q]);
        }
#pragma unroll
        for (int q = 0; q < kPhiloxChains; ++q)
            st_stream(P.out + 4 * (j + q * stride), make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]));
    }
    for (; j < P.n_ctr; j += stride) {
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
