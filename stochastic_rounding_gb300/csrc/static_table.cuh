// static_table.cuh -- the allocation-free multi-tensor step (its descriptor
// table in a library-owned static device array) and its host launcher.
// Included by asr.cu inside its anonymous namespace (one translation unit).

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

// The pipelined step with its table read from global memory (g_static_table).
template <int PT, int GT, int RM, bool A4>
__global__ void __launch_bounds__(TmaShape<PT, GT>::kThreads, 1)
adamw_sr_tma_static_kernel(const __grid_constant__ GlobalTable tab, const __grid_constant__ AdamParams P,
                           uint64_t limit_ns)
{
    tma_step<PT, GT, RM, A4>(tab, P, limit_ns);
}

// Per-device set-up of this path, kept in fixed arrays (no allocation): the
// device address of g_static_table -- on the host its name is only a
// stand-in for the symbol, so the address is looked up with
// cudaGetSymbolAddress while the device is current -- and the persistent grid
// of each kernel variant.
constexpr int kMaxDevices = 64;
constexpr int kStaticVariants = 18;        // 6 dtype/rounding combinations x {pipelined with bases that are
                                           // multiples of 4, pipelined with any base, plain}
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

// Host staging: fixed arrays, guarded by a mutex for the duration of a call:
// the descriptors after splitting unaligned tensors (split_unaligned), the
// pipelined kernels' table and the plain kernel's launch table.
std::mutex g_stage_mu;
asr_tensor_desc g_stage_split[2 * kStaticTableMax];
TensorEntry g_stage_table[kStaticTableMax];
AdamTable<kCapLarge> g_stage_plain;

template <int PT, int GT, int RM, bool A4>
asr_status launch_static_group(int dev, const TensorEntry *dev_table, uint64_t tiles, const AdamParams &P,
                               cudaStream_t stream)
{
    auto kernel = adamw_sr_tma_static_kernel<PT, GT, RM, A4>;
    const int smem = TmaStage<PT, GT>::kSmem;
    int grid = 0;
    asr_status st = static_grid(kernel, dev, (A4 ? 0 : 6) + variant_slot(PT, GT, RM), TmaShape<PT, GT>::kThreads,
                                smem, &grid);
    if (st != ASR_OK) return st;
    st = tma_launch_grid(tiles, &grid);
    if (st != ASR_OK) return st;
    GlobalTable tab;
    tab.t = dev_table;
    tab.total_tiles = tiles;
    kernel<<<grid, TmaShape<PT, GT>::kThreads, smem, stream>>>(tab, P, kWaitLimitNs);
    return launched(ASR_KERNEL_ADAMW_STATIC);
}

// Tensors whose buffers are not 16-byte aligned take the plain kernel, its
// table in the launch parameters (staged in g_stage_plain, kCapLarge per
// launch).
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
            if (d.n == 0 || d.param_dtype != PT || d.grad_dtype != GT || desc_class(d, RM) != kPlainPath) continue;
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
            asr_status st = static_grid(kernel, dev, 12 + variant_slot(PT, GT, RM), kThreads, 0, &grid);
            if (st != ASR_OK) return st;
        }
        g_stage_plain.total_tiles = tiles;
        g_stage_plain.count = c;
        const int g = static_cast<uint64_t>(grid) > tiles ? static_cast<int>(tiles) : grid;
        kernel<<<g, kThreads, 0, stream>>>(g_stage_plain, P);
        asr_status st = launched(ASR_KERNEL_ADAMW_STATIC);
        if (st != ASR_OK) return st;
    }
    return ASR_OK;
}

// One dtype/rounding combination: its pipelined blocks of the static array
// (block 0: bases that are multiples of 4, block 1: any base), then its
// tensors with unaligned buffers.
template <int PT, int GT, int RM>
asr_status launch_static_combo(int dev, const TensorEntry *const blocks[2], const uint64_t tiles[2],
                               const int counts[2], const asr_tensor_desc *table, int32_t n_tensors,
                               const AdamParams &P, cudaStream_t stream)
{
    if (counts[0] > 0) {
        asr_status st = launch_static_group<PT, GT, RM, true>(dev, blocks[0], tiles[0], P, stream);
        if (st != ASR_OK) return st;
    }
    if constexpr (PT == ASR_BF16 && RM == ASR_ROUND_SR) {
        if (counts[1] > 0) {
            asr_status st = launch_static_group<PT, GT, RM, false>(dev, blocks[1], tiles[1], P, stream);
            if (st != ASR_OK) return st;
        }
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
    // unaligned tensors split at their first common aligned element; from
    // here on the split descriptors stand for the caller's table
    int32_t n_split = 0;
    for (int32_t i = 0; i < n_tensors; ++i) n_split += split_unaligned(table[i], rm, g_stage_split + n_split);
    table = g_stage_split;
    n_tensors = n_split;
    // Tensors for the pipelined kernel: one contiguous block of the table per
    // (dtype group, base class) -- block index 2 * (param dtype * 2 + grad
    // dtype) + (base class is "any base") -- all sent in one copy.
    int used = 0;
    int block_start[8] = {}, block_count[8] = {};
    uint64_t block_tiles[8] = {};
    for (int b = 0; b < 8; ++b) {
        const int gi = b / 2, pdt = gi / 2, gdt = gi % 2;
        const int cls = b % 2 ? kVecAnyBase : kVecA4;
        block_start[b] = used;
        uint64_t tiles = 0;
        for (int32_t i = 0; i < n_tensors; ++i) {
            const asr_tensor_desc &d = table[i];
            if (d.n == 0 || d.param_dtype != pdt || d.grad_dtype != gdt || desc_class(d, rm) != cls) continue;
            TensorEntry &T = g_stage_table[used++];
            T.p = d.param;
            T.g = d.grad;
            T.m = d.exp_avg;
            T.v = d.exp_avg_sq;
            T.n = d.n;
            T.base = d.base_index;
            tiles += (d.n + tma_tile(pdt, gdt) - 1) / tma_tile(pdt, gdt);
            T.tile_end = tiles;
        }
        block_count[b] = used - block_start[b];
        block_tiles[b] = tiles;
    }
    if (used > 0) {
        // From pageable host memory: returns once the table is staged for the
        // transfer, which the kernels below follow on the same stream.
        cudaError_t e = cudaMemcpyAsync(dev_table, g_stage_table, sizeof(TensorEntry) * used,
                                        cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    for (int gi = 0; gi < 4; ++gi) {
        const TensorEntry *const blocks[2] = {dev_table + block_start[2 * gi], dev_table + block_start[2 * gi + 1]};
        const uint64_t tiles[2] = {block_tiles[2 * gi], block_tiles[2 * gi + 1]};
        const int counts[2] = {block_count[2 * gi], block_count[2 * gi + 1]};
        if (gi == 3)        // bf16 params, bf16 grads
            st = rm == ASR_ROUND_SR
                ? launch_static_combo<ASR_BF16, ASR_BF16, ASR_ROUND_SR>(dev, blocks, tiles, counts, table, n_tensors, P, stream)
                : launch_static_combo<ASR_BF16, ASR_BF16, ASR_ROUND_RNE>(dev, blocks, tiles, counts, table, n_tensors, P, stream);
        else if (gi == 2)   // bf16 params, f32 grads
            st = rm == ASR_ROUND_SR
                ? launch_static_combo<ASR_BF16, ASR_F32, ASR_ROUND_SR>(dev, blocks, tiles, counts, table, n_tensors, P, stream)
                : launch_static_combo<ASR_BF16, ASR_F32, ASR_ROUND_RNE>(dev, blocks, tiles, counts, table, n_tensors, P, stream);
        else if (gi == 1)   // f32 params, bf16 grads (the rounding mode does not apply)
            st = launch_static_combo<ASR_F32, ASR_BF16, ASR_ROUND_SR>(dev, blocks, tiles, counts, table, n_tensors, P, stream);
        else                // f32 params, f32 grads
            st = launch_static_combo<ASR_F32, ASR_F32, ASR_ROUND_SR>(dev, blocks, tiles, counts, table, n_tensors, P, stream);
        if (st != ASR_OK) return st;
    }
    return ASR_OK;
}
