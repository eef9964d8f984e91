// Test-only: checks Blackwell's hardware stochastic-rounding conversion
// cvt.rs.bf16x2.f32 against the add-and-truncate definition ("Add stochastic
// rounding and philox RNG helpers", Primitives): for every non-NaN binary32
// pattern x and 16-bit random value r, bf16 = (bits(x) + r) >> 16.  Both
// output lanes are checked: the first operand lands in the high half with
// rbits[31:16], the second in the low half with rbits[15:0].
//
// usage: cvt_rs_sweep R_STRIDE
//   R_STRIDE = 1 sweeps all 65,536 random values (2^48 pairs per lane, about
//   two minutes on GB300); a larger stride takes every R_STRIDE-th value.  In
//   addition, for every x, the two values at the round-up threshold,
//   r = 0x10000 - low16(x) and r = 0xFFFF - low16(x), are always checked.
// Prints the counts; exits 1 on any mismatch.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cuda_runtime.h>

__device__ __forceinline__ uint32_t cvt_rs(float a, float b, uint32_t r)
{
    uint32_t d;
    asm volatile("cvt.rs.bf16x2.f32 %0, %1, %2, %3;" : "=r"(d) : "f"(a), "f"(b), "r"(r));
    return d;
}

__device__ __forceinline__ unsigned long long check(uint32_t u, uint32_t r)
{
    const float x = __uint_as_float(u);
    const uint32_t d = cvt_rs(x, x, (r << 16) | r);
    const uint32_t want = (u + r) >> 16;
    return ((d >> 16) != want) + ((d & 0xFFFFu) != want);
}

__global__ void sweep(uint32_t r_stride, unsigned long long *counts)
{
    unsigned long long bad = 0, tested = 0;
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
    for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < (1ull << 32); i += stride) {
        const uint32_t u = static_cast<uint32_t>(i);
        if ((u & 0x7FFFFFFFu) > 0x7F800000u) continue;      // NaN inputs: the hardware canonicalises them
        for (uint32_t r = 0; r < 65536u; r += r_stride) bad += check(u, r);
        const uint32_t low = u & 0xFFFFu;
        bad += check(u, (0x10000u - low) & 0xFFFFu) + check(u, 0xFFFFu - low);
        tested += 2 * (65536u / r_stride + 2);
    }
    atomicAdd(&counts[0], bad);
    atomicAdd(&counts[1], tested);
}

int main(int argc, char **argv)
{
    const uint32_t r_stride = argc > 1 ? static_cast<uint32_t>(strtoul(argv[1], nullptr, 0)) : 1024u;
    if (r_stride == 0 || r_stride > 65536u) return 2;
    unsigned long long *d_c = nullptr, c[2] = {0, 0};
    if (cudaMalloc(&d_c, sizeof(c)) != cudaSuccess) return 2;
    cudaMemset(d_c, 0, sizeof(c));
    sweep<<<152 * 8, 256>>>(r_stride, d_c);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        printf("cuda error %s\n", cudaGetErrorString(e));
        return 2;
    }
    cudaMemcpy(c, d_c, sizeof(c), cudaMemcpyDeviceToHost);
    cudaFree(d_c);
    printf("cvt.rs.bf16x2.f32 vs add-and-truncate: %llu lane checks, %llu mismatches (r stride %u)\n", c[1], c[0],
           r_stride);
    return c[0] != 0;
}
