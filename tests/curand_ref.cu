// Test-only: cuRAND's Philox4_32_10 device generator, called as a black box,
// as an independent reference for the Philox words.  Element q of the output
// is curand4() of a state initialised with (seed, subsequence = step,
// offset = 4*(q0 + q)).
#include <cstdint>
#include <cuda_runtime.h>
#include <curand_kernel.h>

__global__ void curand_words(uint4 *out, unsigned long long n, unsigned long long q0, unsigned int step,
                             unsigned long long seed)
{
    const unsigned long long q = blockIdx.x * static_cast<unsigned long long>(blockDim.x) + threadIdx.x;
    if (q >= n) return;
    curandStatePhilox4_32_10_t st;
    curand_init(seed, step, 4ull * (q0 + q), &st);
    out[q] = curand4(&st);
}

extern "C" int curand_ref_words(uint32_t *out, unsigned long long n, unsigned long long q0, unsigned int step,
                                unsigned long long seed)
{
    if (n == 0) return 0;
    const unsigned int threads = 256;
    const unsigned long long blocks = (n + threads - 1) / threads;
    curand_words<<<static_cast<unsigned int>(blocks), threads>>>(reinterpret_cast<uint4 *>(out), n, q0, step, seed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return static_cast<int>(e);
    return static_cast<int>(cudaDeviceSynchronize());
}
