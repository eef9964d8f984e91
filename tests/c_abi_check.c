/* A C program that uses the library through include/asr.h alone (device
 * memory from the CUDA runtime, no Python): a multi-tensor AdamW-SR step
 * over three tensors of different dtypes and bases, two steps, and a run of
 * Philox words, each compared byte for byte with the oracle's C functions
 * (oracle/asr_oracle.c) on the same inputs.  Prints C_ABI_OK and exits 0 on
 * success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "asr.h"

/* the oracle's C entry points */
void oracle_adamw_step(void *param, int param_dtype, const void *grad, int grad_dtype, float *exp_avg,
                       float *exp_avg_sq, uint64_t n, uint64_t base_index, double lr, double beta1,
                       double beta2, double eps, double wd, uint32_t step, uint64_t seed, int rounding);
void oracle_philox_fill(uint32_t *out, uint64_t n_ctr, uint64_t ctr_base, uint32_t ctr2, uint32_t ctr3,
                        uint64_t seed);

#define CK(x)                                                                                  \
    do {                                                                                       \
        cudaError_t e_ = (x);                                                                  \
        if (e_ != cudaSuccess) {                                                               \
            printf("%s: %s\n", #x, cudaGetErrorString(e_));                                    \
            return 2;                                                                          \
        }                                                                                      \
    } while (0)

/* seeded inputs: a 64-bit LCG; bf16 patterns are the top halves of binary32
 * values (truncation: any pattern is a valid input) */
static uint64_t g_state = 12345;
static float next_f32(float scale)
{
    g_state = g_state * 6364136223846793005ull + 1442695040888963407ull;
    return ((float)(g_state >> 40) / 16777216.0f - 0.5f) * scale;
}
static uint16_t top_half(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    return (uint16_t)(u >> 16);
}

struct tensor {
    uint64_t n, base;
    int pdt, gdt;
    void *hp, *hg, *hm, *hv;  /* host copies, updated by the oracle */
    void *dp, *dg, *dm, *dv;  /* device buffers, updated by the library */
};

static int make(struct tensor *t, uint64_t n, uint64_t base, int pdt, int gdt)
{
    const size_t ps = pdt == ASR_BF16 ? 2 : 4, gs = gdt == ASR_BF16 ? 2 : 4;
    t->n = n;
    t->base = base;
    t->pdt = pdt;
    t->gdt = gdt;
    t->hp = malloc(n * ps);
    t->hg = malloc(n * gs);
    t->hm = malloc(n * 4);
    t->hv = malloc(n * 4);
    for (uint64_t i = 0; i < n; ++i) {
        const float p = next_f32(0.04f), g = next_f32(0.002f);
        if (pdt == ASR_BF16) ((uint16_t *)t->hp)[i] = top_half(p);
        else ((float *)t->hp)[i] = p;
        if (gdt == ASR_BF16) ((uint16_t *)t->hg)[i] = top_half(g);
        else ((float *)t->hg)[i] = g;
        ((float *)t->hm)[i] = next_f32(2e-4f);
        const float v = next_f32(2e-6f);
        ((float *)t->hv)[i] = v < 0 ? -v : v;
    }
    CK(cudaMalloc(&t->dp, n * ps));
    CK(cudaMalloc(&t->dg, n * gs));
    CK(cudaMalloc(&t->dm, n * 4));
    CK(cudaMalloc(&t->dv, n * 4));
    CK(cudaMemcpy(t->dp, t->hp, n * ps, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(t->dg, t->hg, n * gs, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(t->dm, t->hm, n * 4, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(t->dv, t->hv, n * 4, cudaMemcpyHostToDevice));
    return 0;
}

static int same(const void *dev, const void *host, size_t bytes, const char *what)
{
    void *got = malloc(bytes);
    if (cudaMemcpy(got, dev, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
        printf("copy back failed: %s\n", what);
        return 0;
    }
    const int ok = memcmp(got, host, bytes) == 0;
    if (!ok) printf("differs from the oracle: %s\n", what);
    free(got);
    return ok;
}

int main(void)
{
    CK(cudaSetDevice(0));
    struct tensor t[3];
    if (make(&t[0], 10007, 5, ASR_BF16, ASR_BF16) || make(&t[1], 4099, 10012, ASR_F32, ASR_F32) ||
        make(&t[2], 70001, 14111, ASR_BF16, ASR_F32))
        return 2;
    asr_tensor_desc table[3];
    for (int k = 0; k < 3; ++k) {
        table[k].param = t[k].dp;
        table[k].grad = t[k].dg;
        table[k].exp_avg = (float *)t[k].dm;
        table[k].exp_avg_sq = (float *)t[k].dv;
        table[k].n = t[k].n;
        table[k].base_index = t[k].base;
        table[k].param_dtype = t[k].pdt;
        table[k].grad_dtype = t[k].gdt;
    }
    uint64_t before[ASR_KERNEL_KINDS], after[ASR_KERNEL_KINDS];
    if (asr_kernel_launches(before, ASR_KERNEL_KINDS) != ASR_OK) return 2;
    for (uint32_t step = 1; step <= 2; ++step) {
        asr_adamw_hparams hp;
        memset(&hp, 0, sizeof hp);
        hp.lr = 1e-3;
        hp.beta1 = 0.9;
        hp.beta2 = 0.999;
        hp.eps = 1e-8;
        hp.weight_decay = 0.01;
        hp.step = step;
        hp.rounding = ASR_ROUND_SR;
        hp.seed = 0x123456789ull;
        const asr_status st = asr_adamw_sr_multi_tensor(table, 3, &hp, NULL);
        if (st != ASR_OK) {
            printf("asr_adamw_sr_multi_tensor: %s\n", asr_status_string(st));
            return 1;
        }
        for (int k = 0; k < 3; ++k)
            oracle_adamw_step(t[k].hp, t[k].pdt, t[k].hg, t[k].gdt, (float *)t[k].hm, (float *)t[k].hv, t[k].n,
                              t[k].base, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, step, hp.seed, 0);
    }
    CK(cudaDeviceSynchronize());
    int ok = 1;
    for (int k = 0; k < 3; ++k) {
        ok &= same(t[k].dp, t[k].hp, t[k].n * (t[k].pdt == ASR_BF16 ? 2 : 4), "params");
        ok &= same(t[k].dm, t[k].hm, t[k].n * 4, "exp_avg");
        ok &= same(t[k].dv, t[k].hv, t[k].n * 4, "exp_avg_sq");
    }
    /* Philox words across the 2^32 carry of the counter */
    const uint64_t n_ctr = 5000;
    uint32_t *dw, *want = malloc(4 * n_ctr * 4);
    CK(cudaMalloc((void **)&dw, 4 * n_ctr * 4));
    if (asr_philox4x32(dw, n_ctr, (1ull << 32) - 2500, 3, 0, 99, NULL) != ASR_OK) return 1;
    CK(cudaDeviceSynchronize());
    oracle_philox_fill(want, n_ctr, (1ull << 32) - 2500, 3, 0, 99);
    ok &= same(dw, want, 4 * n_ctr * 4, "Philox words");
    uint32_t bits = 1;
    if (asr_take_device_error(&bits, NULL) != ASR_OK || bits != 0) {
        printf("device error bits %u\n", bits);
        ok = 0;
    }
    if (asr_kernel_launches(after, ASR_KERNEL_KINDS) != ASR_OK) return 2;
    uint64_t launched = 0;
    for (int k = 0; k < ASR_KERNEL_KINDS; ++k) launched += after[k] - before[k];
    if (launched < 3) {
        printf("launch counters moved by %llu\n", (unsigned long long)launched);
        ok = 0;
    }
    if (!ok) return 1;
    printf("C_ABI_OK\n");
    return 0;
}
