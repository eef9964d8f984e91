/*
 * asr_oracle.c -- plain, slow, single-threaded C oracle for the fused AdamW step
 * with Philox-keyed stochastic rounding to bf16.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA path is compared
 * against.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header, table or constant generator with the CUDA
 * library and includes none of its files.
 *
 * Build:  gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared
 *         (contraction must stay off: each float operation below is one IEEE
 *         binary32 operation, rounded to nearest-even, evaluated in the order
 *         written; aarch64 GCC would otherwise fuse a*b+c into an FMA).
 *
 * Sources followed (cited by page title and section):
 *   [SR]   "Add stochastic rounding and philox RNG helpers" (FlyDSL PR 907),
 *          section Primitives: add the random bits to the 16 mantissa bits that
 *          bf16 drops, then truncate; probability of rounding up equals the
 *          fractional distance; Inf/NaN pass through.
 *   [RNG]  same page, section Primitives and the review discussion: Philox 4x32,
 *          the generator exposed as cuRAND's Philox4_32_10 and Triton's tl.rand;
 *          Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *          1, 2, 3" (SC'11) for its definition.
 *   [AW]   "adamw-sr", introduction and section Method: decoupled-weight-decay
 *          Adam fused per parameter, bf16 write-back by stochastic rounding,
 *          Philox keyed by (seed, step) and indexed by each element's global
 *          parameter position; section Correctness: shards with base_index equal
 *          the whole update.  Loshchilov and Hutter (2019) for AdamW itself.
 *   [GEMM] "Add stochastic rounding and philox RNG helpers", section Consumer:
 *          the rounding's first user, a bf16 matrix product that may write
 *          its binary32 sums out by stochastic rounding, random bits chosen
 *          per output element from a seed, as an option next to nearest
 *          rounding.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - counter layout: key = (seed lo, seed hi); counter = ((i>>2) lo, (i>>2) hi,
 *     step, 0); element i takes word (i & 3), low 16 bits.
 *   - NaN input to a bf16 rounding: the result keeps sign and the top payload
 *     bits and forces the quiet bit, (u >> 16) | 0x0040, so a NaN stays a NaN
 *     (plain add-and-truncate could turn some NaN payloads into Inf or +-0).
 *   - the per-step scalars are formed in binary64 from the caller's binary64
 *     hyperparameters and each rounded once to binary32.
 *   - the element update order (torch.optim.AdamW's single-tensor order):
 *       p1  = p * decay
 *       m'  = (b1 * m) + (omb1 * g)
 *       v'  = (b2 * v) + (omb2 * (g * g))
 *       den = (sqrt(v') / bc2s) + eps
 *       pn  = p1 - (step_size * (m' / den))
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#include <float.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs binary32 expressions evaluated in binary32 (FLT_EVAL_METHOD == 0)"
#endif

/* ---------------------------------------------------------------- bits ---- */

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* bf16 -> f32 is exact: the bf16 pattern is the top half of the f32 pattern. */
static float bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

static int f32_is_nan_bits(uint32_t u) { return (u & 0x7FFFFFFFu) > 0x7F800000u; }

/* ------------------------------------------------------------- Philox ---- */
/*
 * Philox4x32-10 [RNG].  State (c0,c1,c2,c3), key (k0,k1).  One round takes the
 * two 32x32->64 products M0*c0 and M1*c2 and forms
 *     (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0)).
 * Ten rounds; the key is raised by the Weyl constants between rounds, so the
 * first round uses the key as given.  The output is the final state.
 */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32-bit word that element i draws at a given (seed, step) [AW Method]. */
uint32_t oracle_element_word(uint64_t i, uint32_t step, uint64_t seed)
{
    uint64_t q = i >> 2;
    uint32_t ctr[4] = { (uint32_t)q, (uint32_t)(q >> 32), step, 0u };
    uint32_t key[2] = { (uint32_t)seed, (uint32_t)(seed >> 32) };
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    return w[i & 3];
}

/* n_ctr consecutive counters starting at (ctr_base lo, ctr_base hi, ctr2, ctr3);
 * out receives 4 words per counter, in word order. */
void oracle_philox_fill(uint32_t *out, uint64_t n_ctr, uint64_t ctr_base,
                        uint32_t ctr2, uint32_t ctr3, uint64_t seed)
{
    uint32_t key[2] = { (uint32_t)seed, (uint32_t)(seed >> 32) };
    for (uint64_t j = 0; j < n_ctr; ++j) {
        uint64_t c = ctr_base + j;
        uint32_t ctr[4] = { (uint32_t)c, (uint32_t)(c >> 32), ctr2, ctr3 };
        oracle_philox4x32_10(ctr, key, out + 4 * j);
    }
}

/* ------------------------------------------------------------ rounding ---- */

/* Stochastic rounding f32 -> bf16 [SR]: add the low 16 bits of r to the f32
 * pattern and keep the top 16 bits.  For non-NaN x the sum cannot carry out of
 * 32 bits (the largest non-NaN pattern is 0xFF800000).  NaN: see header. */
uint16_t oracle_sr_bf16(float x, uint32_t r)
{
    uint32_t u = f32_bits(x);
    if (f32_is_nan_bits(u))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t sum = u + (r & 0xFFFFu);
    return (uint16_t)(sum >> 16);
}

/* Round-to-nearest-even f32 -> bf16 (the biased mode SR replaces). */
uint16_t oracle_rne_bf16(float x)
{
    uint32_t u = f32_bits(x);
    if (f32_is_nan_bits(u))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    uint32_t sum = u + 0x7FFFu + keep_lsb;
    return (uint16_t)(sum >> 16);
}

/* Element j of x rounded to nearest, ties to even. */
void oracle_rne_fill(const float *x, uint16_t *out, uint64_t n)
{
    for (uint64_t j = 0; j < n; ++j)
        out[j] = oracle_rne_bf16(x[j]);
}

/* Element j of x (global index base_index + j) rounded stochastically.  If
 * rbits is non-NULL, element j uses rbits[j] instead of the Philox word. */
void oracle_sr_fill(const float *x, const uint32_t *rbits, uint16_t *out, uint64_t n,
                    uint64_t base_index, uint32_t step, uint64_t seed)
{
    for (uint64_t j = 0; j < n; ++j) {
        uint32_t r = rbits ? rbits[j] : oracle_element_word(base_index + j, step, seed);
        out[j] = oracle_sr_bf16(x[j], r);
    }
}

/* ----------------------------------------------------------------- GEMM ---- */

/* [GEMM] C = A . B^T, A (m x k) and B (n x k) row-major bf16 patterns, rows
 * row0 .. row0+m-1 of a product with n columns.  The page fixes no summation
 * order, so the accumulator here is the plain definition: the binary64 sum,
 * in k order, of the bf16 x bf16 products (each exact in binary64), rounded
 * once to binary32.  Element (row0 + i, j) has global index (row0 + i)*n + j
 * and is rounded like every other element of this file: stochastically with
 * its Philox word (rounding 0) or to nearest-even (rounding 1).  acc, if
 * non-NULL, receives the binary32 accumulator. */
void oracle_gemm_bf16(const uint16_t *a, const uint16_t *b, float *acc, uint16_t *out, uint64_t m,
                      uint64_t n, uint64_t k, uint64_t row0, int rounding, uint32_t step, uint64_t seed)
{
    for (uint64_t i = 0; i < m; ++i) {
        for (uint64_t j = 0; j < n; ++j) {
            double s = 0.0;
            for (uint64_t t = 0; t < k; ++t)
                s += (double)bf16_to_f32(a[i * k + t]) * (double)bf16_to_f32(b[j * k + t]);
            const float x = (float)s;
            if (acc)
                acc[i * n + j] = x;
            out[i * n + j] = rounding == 1
                ? oracle_rne_bf16(x)
                : oracle_sr_bf16(x, oracle_element_word((row0 + i) * n + j, step, seed));
        }
    }
}

/* ---------------------------------------------------------------- AdamW ---- */

/* Per-step scalars, in this order:
 *   [0] b1  [1] b2  [2] eps  [3] decay = 1 - lr*wd  [4] omb1 = 1 - beta1
 *   [5] omb2 = 1 - beta2  [6] step_size = lr / (1 - beta1^t)
 *   [7] bc2s = sqrt(1 - beta2^t)
 * each computed in binary64 and rounded once to binary32. */
void oracle_adamw_scalars(double lr, double beta1, double beta2, double eps, double wd,
                          uint32_t step, float out[8])
{
    double t = (double)step;
    out[0] = (float)beta1;
    out[1] = (float)beta2;
    out[2] = (float)eps;
    out[3] = (float)(1.0 - lr * wd);
    out[4] = (float)(1.0 - beta1);
    out[5] = (float)(1.0 - beta2);
    out[6] = (float)(lr / (1.0 - pow(beta1, t)));
    out[7] = (float)sqrt(1.0 - pow(beta2, t));
}

/* dtype codes: 0 = binary32, 1 = bf16.  rounding: 0 = stochastic, 1 = RNE. */
void oracle_adamw_step(void *param, int param_dtype, const void *grad, int grad_dtype,
                       float *exp_avg, float *exp_avg_sq, uint64_t n, uint64_t base_index,
                       double lr, double beta1, double beta2, double eps, double wd,
                       uint32_t step, uint64_t seed, int rounding)
{
    float s[8];
    oracle_adamw_scalars(lr, beta1, beta2, eps, wd, step, s);
    const float b1 = s[0], b2 = s[1], ep = s[2], decay = s[3];
    const float omb1 = s[4], omb2 = s[5], step_size = s[6], bc2s = s[7];

    for (uint64_t j = 0; j < n; ++j) {
        float p = param_dtype == 1 ? bf16_to_f32(((const uint16_t *)param)[j])
                                   : ((const float *)param)[j];
        float g = grad_dtype == 1 ? bf16_to_f32(((const uint16_t *)grad)[j])
                                  : ((const float *)grad)[j];
        float m = exp_avg[j];
        float v = exp_avg_sq[j];

        float p1 = p * decay;                    /* decoupled weight decay   */
        float bm = b1 * m;
        float gm = omb1 * g;
        float m1 = bm + gm;                      /* first moment             */
        float gg = g * g;
        float bv = b2 * v;
        float gv = omb2 * gg;
        float v1 = bv + gv;                      /* second moment            */
        float rt = sqrtf(v1);
        float dq = rt / bc2s;                    /* sqrt(v_hat), bias-corrected */
        float den = dq + ep;
        float ratio = m1 / den;
        float upd = step_size * ratio;           /* lr * m_hat / den         */
        float pn = p1 - upd;

        exp_avg[j] = m1;
        exp_avg_sq[j] = v1;
        if (param_dtype == 1) {
            uint16_t h = rounding == 1
                ? oracle_rne_bf16(pn)
                : oracle_sr_bf16(pn, oracle_element_word(base_index + j, step, seed));
            ((uint16_t *)param)[j] = h;
        } else {
            ((float *)param)[j] = pn;
        }
    }
}

/* a*b + c as two separately rounded binary32 operations; used by a test that
 * checks this file was built with contraction off. */
float oracle_mul_add(float a, float b, float c)
{
    float prod = a * b;
    return prod + c;
}
