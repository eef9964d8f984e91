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
// Design (GB300): the optimizer step is a streaming pass, 22 bytes per
// element for bf16 params/grads with f32 moments, far below the ALU ridge, so
// its kernels are built for HBM bandwidth.  The hot path (adamw_kernels.cuh)
// is a kernel with one resident CTA per SM, in which a producer warp streams
// tiles into a shared-memory ring with bulk copies (pipeline.cuh) while
// consumer warps compute and store; the grid holds one CTA per tile and the
// running CTAs take the tiles of those not yet started (cluster launch
// control), so every SM keeps working until the last tile.  The tensor table
// of a whole model travels by value (__grid_constant__), so one launch covers
// it.  Philox runs in
// registers, one 10-round call per four elements, round keys precomputed on
// the host (common.cuh).  Every float operation is an explicitly rounded IEEE
// binary32 intrinsic in a fixed order, so results are bit-reproducible.  The
// stand-alone rounding and Philox kernels (rounding_kernels.cuh), an
// allocation-free variant of the step (static_table.cuh), the host-buffer
// pipeline around the step (host_pipeline.cuh) and a tensor-core GEMM with a
// stochastic-rounding epilogue (gemm_sr.cuh) share these pieces.
// This file holds the host side: argument checks, launch shapes and the C ABI.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <memory>
#include <mutex>
#include <thread>
#include <unordered_map>
#include <utility>
#include <vector>

#include "asr.h"

namespace {

#include "common.cuh"
#include "pipeline.cuh"
#include "adamw_kernels.cuh"
#include "rounding_kernels.cuh"

// Takes the device error bits: reads and clears the word in one atomic step
// (so no bit set by a kernel still running elsewhere is lost between the two)
// and writes them to dst -- device memory, or page-locked host memory that
// the GPU can write -- or, with dst null, to copy slot `slot` of
// g_error_taken, from which the blocking take copies them to the host.  Each
// blocking take in progress holds its own slot, so concurrent takes from
// several host threads cannot read one another's bits.
constexpr int kTakeSlots = 64;
__device__ unsigned int g_error_taken[kTakeSlots];

__global__ void take_error_kernel(unsigned int *dst, int slot)
{
    const unsigned int bits = atomicExch(&g_device_error, 0u);
    *(dst ? dst : &g_error_taken[slot]) = bits;
}

// ------------------------------------------------------------- host side

thread_local int g_last_cuda_error = 0;

// Copy slots of the blocking error take: a slot is held from its launch to
// the end of its host copy.  With every slot in use (kTakeSlots takes in
// progress at once) the caller yields until one is released.
std::mutex g_take_mu;
uint64_t g_take_busy = 0;
static_assert(kTakeSlots == 64, "one bit of g_take_busy per slot");

int take_slot()
{
    for (;;) {
        {
            std::lock_guard<std::mutex> lk(g_take_mu);
            if (~g_take_busy) {
                const int slot = __builtin_ctzll(~g_take_busy);
                g_take_busy |= 1ull << slot;
                return slot;
            }
        }
        std::this_thread::yield();
    }
}

void release_slot(int slot)
{
    std::lock_guard<std::mutex> lk(g_take_mu);
    g_take_busy &= ~(1ull << slot);
}

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

// Launches per kernel kind (asr_kernel_launches), counted on the host when a
// launch has been queued without error.
std::atomic<uint64_t> g_launches[ASR_KERNEL_KINDS];

asr_status launched(int kind)
{
    const asr_status st = check_launch();
    if (st == ASR_OK) g_launches[kind].fetch_add(1, std::memory_order_relaxed);
    return st;
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

#ifndef ASR_USE_TMA
#define ASR_USE_TMA 1
#endif

// Which kernel updates a tensor.
//   kPlainPath: buffers not all 16-byte aligned -- the register-resident
//     kernel with scalar units;
//   kVecA4: 16-byte-aligned buffers and either a base index that is a
//     multiple of 4 or no random bits needed (f32 params, nearest rounding)
//     -- the pipelined kernel, two Philox counters per 8-element unit, or,
//     for a launch group of at most ASR_SMALL_GROUP_BYTES, the
//     register-resident kernel with 128-bit units;
//   kVecAnyBase: 16-byte-aligned buffers, stochastic rounding of bf16
//     params, base index not a multiple of 4 -- the pipelined kernel drawing
//     three counters per unit.  A model whose parameters are numbered end to
//     end gets such bases after any parameter of odd size.
constexpr int kPlainPath = 0, kVecA4 = 1, kVecAnyBase = 2;

int desc_class(const asr_tensor_desc &d, int rounding)
{
    if (!(aligned16(d.param) && aligned16(d.grad) && aligned16(d.exp_avg) && aligned16(d.exp_avg_sq)))
        return kPlainPath;
    const bool bits = d.param_dtype == ASR_BF16 && rounding == ASR_ROUND_SR;
    if ((d.base_index & 3u) == 0 || !bits) return kVecA4;
    return ASR_USE_TMA ? kVecAnyBase : kPlainPath;
}

// A descriptor whose buffers are not all 16-byte aligned, split where they
// all become aligned: a head of h < 8 elements (the plain kernel) and the
// rest from element h on, its base index advanced by h (a pipelined kernel).
// Such an h exists whenever the four buffers are off alignment by amounts
// that agree -- views of slices that start at the same element offset in
// aligned storage, for instance.  Every element keeps its own global index,
// so the split changes no bit.  Writes 1 or 2 descriptors to out.
int split_unaligned(const asr_tensor_desc &d, int rounding, asr_tensor_desc out[2])
{
    out[0] = d;
    if (d.n == 0 || desc_class(d, rounding) != kPlainPath) return 1;
    const uintptr_t ps = d.param_dtype == ASR_BF16 ? 2 : 4, gs = d.grad_dtype == ASR_BF16 ? 2 : 4;
    for (uint64_t h = 1; h < 8 && h < d.n; ++h) {
        const uintptr_t p = reinterpret_cast<uintptr_t>(d.param) + h * ps;
        const uintptr_t g = reinterpret_cast<uintptr_t>(d.grad) + h * gs;
        const uintptr_t m = reinterpret_cast<uintptr_t>(d.exp_avg + h);
        const uintptr_t v = reinterpret_cast<uintptr_t>(d.exp_avg_sq + h);
        if (((p | g | m | v) & 15u) != 0) continue;
        out[0].n = h;
        out[1] = d;
        out[1].param = reinterpret_cast<void *>(p);
        out[1].grad = reinterpret_cast<const void *>(g);
        out[1].exp_avg = d.exp_avg + h;
        out[1].exp_avg_sq = d.exp_avg_sq + h;
        out[1].n = d.n - h;
        out[1].base_index = d.base_index + h;
        return 2;
    }
    return 1;
}

// Dynamic shared memory opt-in and persistent grid of the bulk-copy kernel,
// cached per (device, kernel).
template <typename K>
asr_status tma_grid(K kernel, int threads, int smem, int *grid)
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
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
    if (e != cudaSuccess) return cuda_fail(e);
    if (per_sm < 1) per_sm = 1;
    *grid = sms * per_sm;
    std::lock_guard<std::mutex> lk(g_grid_mu);
    g_grid_cache[key] = *grid;
    return ASR_OK;
}

// Grid of the pipelined kernel for `tiles` tiles.  Dynamic schedule: one CTA
// per tile (running CTAs take the tiles of CTAs that have not started); fixed
// schedule: the persistent grid, at most one CTA per tile.
asr_status tma_launch_grid(uint64_t tiles, int *grid)
{
#if ASR_TMA_DYNAMIC
    if (tiles > 0x7FFFFFFFull) return ASR_ERR_INVALID_VALUE;     // beyond the grid's x limit
    *grid = static_cast<int>(tiles);
#else
    if (static_cast<uint64_t>(*grid) > tiles) *grid = static_cast<int>(tiles);
#endif
    return ASR_OK;
}

// Launch groups of aligned tensors whose step moves at most this many
// algorithmic bytes take the register-resident kernel: below that the
// pipelined kernel's fixed cost -- barrier set-up, the schedule request, a
// whole stage landing before its consumers start, and tiles so large that
// a small step leaves most SMs idle -- outweighs its streaming.  Measured on
// GB300 with L2 flushed before each step (single tensors, CUDA events), the
// register kernel is 15-40 % faster up to 4 Mi bf16 or 2 Mi f32 params and
// 5-7 % faster at 8 Mi bf16 and 4 Mi f32; the two tie at 16 Mi bf16, and
// from 8 Mi f32 or 32 Mi bf16 params on the pipelined kernel is ahead.
#ifndef ASR_SMALL_GROUP_BYTES
#define ASR_SMALL_GROUP_BYTES (128ull << 20)
#endif

template <int PT, int GT, int RM, int CLS, int CAP>
asr_status launch_group(const asr_tensor_desc *const *descs, int count, const AdamParams &P, cudaStream_t stream)
{
    static_assert(CAP >= 1, "");
    constexpr bool kTma = CLS != kPlainPath && ASR_USE_TMA;
    // algorithmic bytes per element: p read and written, g read, m and v
    // read and written
    constexpr uint64_t kElemBytes = 2 * (PT == ASR_BF16 ? 2 : 4) + (GT == ASR_BF16 ? 2 : 4) + 16;
    uint64_t elems = 0;
    for (int i = 0; i < count; ++i) elems += descs[i]->n;
    // only the class whose units draw two counters each can go either way
    const bool tma = kTma && !(CLS == kVecA4 && elems <= ASR_SMALL_GROUP_BYTES / kElemBytes);
    const uint64_t tile = tma ? static_cast<uint64_t>(TmaShape<PT, GT>::kTile) : static_cast<uint64_t>(kTile);
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
    if constexpr (kTma) {
        if (tma) {
            auto kernel = adamw_sr_tma_kernel<PT, GT, RM, CAP, CLS == kVecA4>;
            const int smem = TmaStage<PT, GT>::kSmem;
            st = tma_grid(kernel, TmaShape<PT, GT>::kThreads, smem, &grid);
            if (st != ASR_OK) return st;
            st = tma_launch_grid(tiles, &grid);
            if (st != ASR_OK) return st;
            kernel<<<grid, TmaShape<PT, GT>::kThreads, smem, stream>>>(tab, P, kWaitLimitNs);
            return launched(CLS == kVecA4 ? ASR_KERNEL_ADAMW_PIPELINED : ASR_KERNEL_ADAMW_PIPELINED_ANY_BASE);
        }
    }
    // the register kernel: vector units for the aligned class, scalar units
    // (any alignment, any base) otherwise
    auto kernel = adamw_sr_kernel<PT, GT, RM, CLS == kVecA4, CAP>;
    st = persistent_grid(kernel, &grid);
    if (st != ASR_OK) return st;
    if (static_cast<uint64_t>(grid) > tiles) grid = static_cast<int>(tiles);
    kernel<<<grid, kThreads, 0, stream>>>(tab, P);
    return launched(CLS == kVecA4 ? ASR_KERNEL_ADAMW_VECTOR : ASR_KERNEL_ADAMW_SCALAR);
}

template <int PT, int GT, int RM, int CLS>
asr_status launch_chunks(const asr_tensor_desc *const *descs, int count, const AdamParams &P, cudaStream_t stream)
{
    if (count == 1) return launch_group<PT, GT, RM, CLS, kCapSmall>(descs, 1, P, stream);
    for (int s = 0; s < count; s += kCapLarge) {
        const int c = count - s < kCapLarge ? count - s : kCapLarge;
        asr_status st = launch_group<PT, GT, RM, CLS, kCapLarge>(descs + s, c, P, stream);
        if (st != ASR_OK) return st;
    }
    return ASR_OK;
}

template <int PT, int GT, int RM>
asr_status dispatch_class(const asr_tensor_desc *const *descs, int count, int cls, const AdamParams &P,
                          cudaStream_t stream)
{
    if (cls == kPlainPath) return launch_chunks<PT, GT, RM, kPlainPath>(descs, count, P, stream);
    if constexpr (PT == ASR_BF16 && RM == ASR_ROUND_SR) {
        if (cls == kVecAnyBase) return launch_chunks<PT, GT, RM, kVecAnyBase>(descs, count, P, stream);
    }
    return launch_chunks<PT, GT, RM, kVecA4>(descs, count, P, stream);
}

asr_status dispatch(const asr_tensor_desc *const *descs, int count, int pdt, int gdt, int rm, int cls,
                    const AdamParams &P, cudaStream_t stream)
{
    if (pdt == ASR_BF16) {
        if (gdt == ASR_BF16)
            return rm == ASR_ROUND_SR ? dispatch_class<ASR_BF16, ASR_BF16, ASR_ROUND_SR>(descs, count, cls, P, stream)
                                      : dispatch_class<ASR_BF16, ASR_BF16, ASR_ROUND_RNE>(descs, count, cls, P, stream);
        return rm == ASR_ROUND_SR ? dispatch_class<ASR_BF16, ASR_F32, ASR_ROUND_SR>(descs, count, cls, P, stream)
                                  : dispatch_class<ASR_BF16, ASR_F32, ASR_ROUND_RNE>(descs, count, cls, P, stream);
    }
    // f32 params are stored as computed: the rounding mode does not apply.
    if (gdt == ASR_BF16) return dispatch_class<ASR_F32, ASR_BF16, ASR_ROUND_SR>(descs, count, cls, P, stream);
    return dispatch_class<ASR_F32, ASR_F32, ASR_ROUND_SR>(descs, count, cls, P, stream);
}

// Launch shapes (and the shared-memory opt-in) of every AdamW kernel, set up
// together on a device's first step, so that any later step -- whichever
// kernels its dtypes, alignment and size pick -- needs no set-up call and
// may be captured into a CUDA graph.
std::atomic<uint64_t> g_adamw_ready{0};

template <int PT, int GT, int RM, int CAP>
asr_status setup_adamw_combo()
{
    int grid = 0;
    asr_status st = persistent_grid(adamw_sr_kernel<PT, GT, RM, false, CAP>, &grid);
    if (st == ASR_OK) st = persistent_grid(adamw_sr_kernel<PT, GT, RM, true, CAP>, &grid);
#if ASR_USE_TMA
    if (st == ASR_OK)
        st = tma_grid(adamw_sr_tma_kernel<PT, GT, RM, CAP, true>, TmaShape<PT, GT>::kThreads,
                      TmaStage<PT, GT>::kSmem, &grid);
    if constexpr (PT == ASR_BF16 && RM == ASR_ROUND_SR) {
        if (st == ASR_OK)
            st = tma_grid(adamw_sr_tma_kernel<PT, GT, RM, CAP, false>, TmaShape<PT, GT>::kThreads,
                          TmaStage<PT, GT>::kSmem, &grid);
    }
#endif
    return st;
}

template <int CAP>
asr_status setup_adamw_cap()
{
    asr_status st = setup_adamw_combo<ASR_BF16, ASR_BF16, ASR_ROUND_SR, CAP>();
    if (st == ASR_OK) st = setup_adamw_combo<ASR_BF16, ASR_BF16, ASR_ROUND_RNE, CAP>();
    if (st == ASR_OK) st = setup_adamw_combo<ASR_BF16, ASR_F32, ASR_ROUND_SR, CAP>();
    if (st == ASR_OK) st = setup_adamw_combo<ASR_BF16, ASR_F32, ASR_ROUND_RNE, CAP>();
    if (st == ASR_OK) st = setup_adamw_combo<ASR_F32, ASR_BF16, ASR_ROUND_SR, CAP>();
    if (st == ASR_OK) st = setup_adamw_combo<ASR_F32, ASR_F32, ASR_ROUND_SR, CAP>();
    return st;
}

asr_status setup_adamw_kernels()
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const uint64_t bit = dev >= 0 && dev < 64 ? 1ull << dev : 0;
    if (bit && (g_adamw_ready.load(std::memory_order_acquire) & bit)) return ASR_OK;
    asr_status st = setup_adamw_cap<kCapSmall>();
    if (st == ASR_OK) st = setup_adamw_cap<kCapLarge>();
    if (st == ASR_OK && bit) g_adamw_ready.fetch_or(bit, std::memory_order_release);
    return st;
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
    bool work = false;
    for (int32_t i = 0; i < n_tensors && !work; ++i) work = table[i].n != 0;
    if (!work) return ASR_OK;                      // nothing to launch, no device touched
    st = setup_adamw_kernels();
    if (st != ASR_OK) return st;
    AdamParams P;
    P.s = make_scalars(*hp);
    P.keys = make_keys(hp->seed);
    P.step = hp->step;

    // Split unaligned tensors at their first common aligned element, then
    // group by (param dtype, grad dtype, kernel class), keeping order.  Every
    // element is independent, so neither step can change any bit.
    const int rm = static_cast<int>(hp->rounding);
    asr_tensor_desc small[8];
    std::unique_ptr<asr_tensor_desc[]> split_holder;
    asr_tensor_desc *split = small;
    if (2 * static_cast<int64_t>(n_tensors) > 8) {
        split_holder.reset(new asr_tensor_desc[2 * static_cast<size_t>(n_tensors)]);
        split = split_holder.get();
    }
    int nt = 0;
    for (int32_t i = 0; i < n_tensors; ++i) nt += split_unaligned(table[i], rm, split + nt);
    // one pass to classify, then a stable counting sort into the 12 groups
    // (param dtype, grad dtype, class), each group in table order
    constexpr int kGroups = 2 * 2 * 3;
    const asr_tensor_desc **sel = nullptr;
    const asr_tensor_desc *one[1];
    int8_t group_small[8];
    std::unique_ptr<const asr_tensor_desc *[]> holder;
    std::unique_ptr<int8_t[]> group_holder;
    int8_t *group = group_small;
    if (nt <= 1) {
        sel = one;
    } else {
        holder.reset(new const asr_tensor_desc *[nt]);
        sel = holder.get();
    }
    if (nt > 8) {
        group_holder.reset(new int8_t[nt]);
        group = group_holder.get();
    }
    int count[kGroups] = {}, start[kGroups];
    for (int i = 0; i < nt; ++i) {
        const asr_tensor_desc &d = split[i];
        group[i] = d.n == 0 ? -1 : static_cast<int8_t>((d.param_dtype * 2 + d.grad_dtype) * 3 + desc_class(d, rm));
        if (group[i] >= 0) ++count[group[i]];
    }
    for (int k = 0, at = 0; k < kGroups; ++k) {
        start[k] = at;
        at += count[k];
    }
    int fill[kGroups];
    std::memcpy(fill, start, sizeof(fill));
    for (int i = 0; i < nt; ++i)
        if (group[i] >= 0) sel[fill[group[i]]++] = &split[i];
    for (int k = 0; k < kGroups; ++k) {
        if (count[k] == 0) continue;
        const int pdt = k / 6, gdt = (k / 3) % 2, cls = k % 3;
        st = dispatch(sel + start[k], count[k], pdt, gdt, rm, cls, P, stream);
        if (st != ASR_OK) return st;
    }
    return ASR_OK;
}

// The launch shapes of every variant of an op, set up together on the op's
// first call on a device, so that a later call may be captured into a CUDA
// graph whichever variant its pointers pick.
template <typename K, size_t N>
asr_status setup_variants(std::atomic<uint64_t> &ready, const K (&kernels)[N])
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const uint64_t bit = dev >= 0 && dev < 64 ? 1ull << dev : 0;
    if (bit && (ready.load(std::memory_order_acquire) & bit)) return ASR_OK;
    for (const K &k : kernels) {
        int grid = 0;
        const asr_status st = persistent_grid(k, &grid);
        if (st != ASR_OK) return st;
    }
    if (bit) ready.fetch_or(bit, std::memory_order_release);
    return ASR_OK;
}

std::atomic<uint64_t> g_philox_ready{0}, g_round_ready{0};

#include "host_pipeline.cuh"
#include "static_table.cuh"
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

asr_status asr_kernel_launches(uint64_t *counts, int32_t n)
{
    if (n < 0 || (n > 0 && !counts)) return ASR_ERR_INVALID_VALUE;
    for (int32_t k = 0; k < n && k < ASR_KERNEL_KINDS; ++k) counts[k] = g_launches[k].load(std::memory_order_relaxed);
    return ASR_OK;
}

asr_status asr_take_device_error(uint32_t *bits, asr_stream_t stream)
{
    if (!bits) return ASR_ERR_INVALID_VALUE;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int slot = take_slot();
    take_error_kernel<<<1, 1, 0, s>>>(nullptr, slot);
    cudaError_t e = cudaGetLastError();
    unsigned int h = 0;
    if (e == cudaSuccess)
        e = cudaMemcpyFromSymbolAsync(&h, g_error_taken, sizeof(h), sizeof(h) * slot, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    release_slot(slot);
    if (e != cudaSuccess) return cuda_fail(e);
    *bits = h;
    return ASR_OK;
}

asr_status asr_take_device_error_async(uint32_t *bits, asr_stream_t stream)
{
    if (!bits || (reinterpret_cast<uintptr_t>(bits) & 3u)) return ASR_ERR_INVALID_VALUE;
    // Only memory the GPU can write: device or managed memory, or page-locked
    // host memory (written through its device-side address).
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, bits);
    if (e != cudaSuccess) return cuda_fail(e);
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged && a.type != cudaMemoryTypeHost)
        return ASR_ERR_INVALID_VALUE;
    if (!a.devicePointer) return ASR_ERR_INVALID_VALUE;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (a.type == cudaMemoryTypeDevice && a.device != dev) return ASR_ERR_INVALID_VALUE;
    take_error_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned int *>(a.devicePointer), 0);
    return check_launch();
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
    void (*const variants[])(const PhiloxParams) = {philox_kernel<true>, philox_kernel<false>};
    asr_status st = setup_variants(g_philox_ready, variants);
    if (st != ASR_OK) return st;
    auto kernel = a16 ? philox_kernel<true> : philox_kernel<false>;
    int grid = 0;
    st = persistent_grid(kernel, &grid);
    if (st != ASR_OK) return st;
    const uint64_t need = (n_ctr + kThreads - 1) / kThreads;
    if (static_cast<uint64_t>(grid) > need) grid = static_cast<int>(need);
    kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(P);
    return launched(ASR_KERNEL_PHILOX);
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
    // vector loads and stores wherever the buffers are 16-byte aligned; a
    // base off a multiple of 4 only costs a third Philox call per unit
    const bool fast = aligned16(x) && aligned16(out) && (!rbits || aligned16(rbits));
    const bool a4 = (base_index & 3u) == 0;
    void (*const variants[])(const SrParams) = {sr_bf16_kernel<true, true>, sr_bf16_kernel<false, true>,
                                                 sr_bf16_kernel<false, false>, sr_bf16_kernel<true, false, true>,
                                                 sr_bf16_kernel<true, false, false>};
    asr_status st = setup_variants(g_round_ready, variants);
    if (st != ASR_OK) return st;
    void (*kernel)(const SrParams) = nullptr;
    if (rbits) kernel = fast ? sr_bf16_kernel<true, true> : sr_bf16_kernel<false, true>;
    else if (!fast) kernel = sr_bf16_kernel<false, false>;
    else kernel = a4 ? sr_bf16_kernel<true, false, true> : sr_bf16_kernel<true, false, false>;
    int grid = 0;
    st = persistent_grid(kernel, &grid);
    if (st != ASR_OK) return st;
    const uint64_t need = ((n + kVec - 1) / kVec + kThreads - 1) / kThreads;
    if (static_cast<uint64_t>(grid) > need) grid = static_cast<int>(need);
    kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(P);
    return launched(ASR_KERNEL_ROUND);
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

asr_status asr_adamw_sr_multi_tensor_host(const asr_host_tensor_desc *table, int32_t n_tensors,
                                          const asr_adamw_hparams *hp, uint64_t chunk_elems, asr_stream_t stream,
                                          asr_stream_t copy_in, asr_stream_t copy_out)
{
    return run_adamw_host(table, n_tensors, hp, chunk_elems, reinterpret_cast<cudaStream_t>(stream),
                          reinterpret_cast<cudaStream_t>(copy_in), reinterpret_cast<cudaStream_t>(copy_out));
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
