// gemm_sr.cuh -- bf16 GEMM on the 5th-generation tensor cores with a
// stochastic-rounding epilogue.  Included into asr.cu (inside its anonymous
// namespace): it shares the Philox, rounding and mbarrier helpers and the
// device error word with the optimizer kernels.
//
// "Add stochastic rounding and philox RNG helpers" (FlyDSL PR 907), section
// Consumer: the first user of the rounding is a bf16 matrix product that may
// write its binary32 sums out by stochastic rounding, random bits chosen per
// output element from a seed, as an option next to nearest rounding.  Here output
// element (i, j) of the M x N result has global index i*N + j and draws its
// random bits exactly as every other element of this library does: word
// (e & 3) of Philox4x32-10 at counter ((e>>2) lo, (e>>2) hi, step, 0) under
// key (seed lo, seed hi).  So the GEMM's output is
// asr_stochastic_round_bf16(acc, base 0, step, seed) of its own f32
// accumulator acc.
//
// C[M,N] = A[M,K] . B[N,K]^T, all row-major (both operands K-contiguous, as
// nn.Linear keeps its weight).  Two kernels compute it:
//   gemm_bf16_sr_pair_kernel (below, used wherever the GPU can hold CTA
//     pairs -- always on GB300): 256 x 256 tiles on clusters of two SMs with
//     tcgen05.mma.cta_group::2, 128-deep K slices; described at its
//     definition;
//   gemm_bf16_sr_kernel (this one, the fallback): 128 x 256 tiles on one SM.
// Edges, both: the tensor maps read zeros past M, N and K (zeros add nothing
// to the sums), and the epilogue stores only rows < M and columns < N.  The
// one-SM kernel is persistent: one CTA per SM walks the tiles in a grouped
// order (16 M-tiles at a time across N, so the tiles in flight share
// operands in L2):
//   warp 0, lane 0   streams 128 x 64 and 256 x 64 slices of A and B into a
//                    4-stage shared-memory ring (tensor-map bulk copies,
//                    128-byte swizzle), completion counted on mbarriers;
//   warp 1           owns the tensor memory: all 512 columns, two 128 x 256
//                    f32 accumulators; its lane 0 issues tcgen05.mma
//                    (kind::f16, bf16 in, f32 accumulate; four K=16 steps
//                    per slice), commits each slice to its stage's "empty"
//                    barrier and each tile to its accumulator's "full"
//                    barrier, and waits for the epilogue to hand an
//                    accumulator back before reusing it;
//   warps 2..5       read the accumulator rows of their TMEM lane quarter
//                    with tcgen05.ld, round (stochastic or nearest-even),
//                    store bf16 (and, optionally, the f32 accumulator) and
//                    release the accumulator -- while the next tile's
//                    products already go into the other one.
// Every wait is bounded (mbar_wait); on a timeout the error bit is raised,
// the thread skips ahead to the cleanup, and the tensor memory is still
// freed.

namespace gemm {

#ifndef ASR_GEMM_PAIR
#define ASR_GEMM_PAIR 1            // 1: two-SM (CTA pair) kernel where pairs fit; 0: one-SM kernel only
#endif

constexpr int kBM = 128;                   // tile rows (M) = TMEM lanes
constexpr int kBN = 256;                   // tile columns (N) = TMEM columns
constexpr int kBK = 64;                    // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreads = 192;              // 6 warps
constexpr int kEpilogueWarps = 4;
constexpr int kGroupM = 16;                // tile order: 16 M-tiles walked across N, group by group
constexpr uint32_t kStageA = kBM * kBK * 2;     // 16 KB
constexpr uint32_t kStageB = kBN * kBK * 2;     // 32 KB
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr int kAccBufs = 2;                     // two accumulators: the epilogue of one tile
                                                // overlaps the main loop of the next
constexpr uint32_t kTmemCols = kBN * kAccBufs;  // 512 f32 columns = all of the tensor memory
// dynamic shared memory: 1 KB of alignment slack, the stages, the barriers
// (full/empty per stage, full/empty per accumulator) and the TMEM address slot
constexpr int kSmem = 1024 + kStages * kStageBytes + (2 * kStages + 2 * kAccBufs) * 8 + 16;

// Instruction descriptor of tcgen05.mma kind::f16: f32 accumulator
// (bits 4-5 = 1), A and B bf16 (bits 7-9 = 1, bits 10-12 = 1), both
// K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kInstrDesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kBN >> 3) << 17) |
                                (uint32_t(kBM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major operand tile written by the
// tensor map with 128-byte swizzle: rows of 128 bytes, 8-row groups 1024
// bytes apart (stride byte offset), leading byte offset unused (1), version
// 1 (bits 46-47), layout "128-byte swizzle" (2, bits 61-63).  The start
// address advances by 32 bytes per K=16 step inside the swizzle row.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1u << 16) | ((uint64_t)(1024u >> 4) << 32) |
           ((uint64_t)1u << 46) | ((uint64_t)2u << 61);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(kInstrDesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t v[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct GemmParams {
    uint16_t *c;            // M x N bf16
    float *c_f32;           // M x N f32 accumulator copy, or null
    uint32_t m, n, k;
    uint32_t step;
    uint32_t rounding;      // asr_rounding
    uint32_t c_align32;     // c is 32-byte aligned: each lane's 16 outputs go out in one 256-bit store
    // two-SM kernel: the first `wide` work items are 256 x 256 tiles, the
    // next `narrow` are the halves (256 x 128) of the last narrow/2 tiles
    uint32_t wide, narrow;
    RoundKeys keys;
};

// One 256-bit store (sm_100 and later); the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t w[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Epilogue of one warp: accumulator row `row` of the output (this lane's
// TMEM lane, columns from tq), columns n0 .. n0+ncols-1, rounded to bf16
// (stochastic or nearest-even) and stored, with the f32 accumulator if asked
// for.  tcgen05.ld is warp-collective, so every lane loads, and lanes whose
// row lies past M (zeros read past the edge) store nothing.
__device__ __forceinline__ void store_rows(const GemmParams &P, uint32_t tq, uint32_t row, uint32_t n0, int ncols)
{
    for (int c = 0; c < ncols; c += 16) {
        uint32_t v[16];
        tmem_ld16(tq + c, v);
        if (row >= P.m) continue;
        const uint64_t e0 = static_cast<uint64_t>(row) * P.n + n0 + c;   // multiple of 16
        uint32_t w[8];
        if (P.rounding == ASR_ROUND_SR) {
            uint32_t r[16];
            philox_q(e0 >> 2, P.step, P.keys, r);
            philox_q((e0 >> 2) + 1, P.step, P.keys, r + 4);
            philox_q((e0 >> 2) + 2, P.step, P.keys, r + 8);
            philox_q((e0 >> 2) + 3, P.step, P.keys, r + 12);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                w[k] = sr_pack2<true>(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]), r[2 * k],
                                      r[2 * k + 1]);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                w[k] = pack_bf16(round_rne(__uint_as_float(v[2 * k])), round_rne(__uint_as_float(v[2 * k + 1])));
        }
        if (P.c_align32) {
            st_global_v8(P.c + e0, w);              // one full 32-byte sector per lane
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(P.c + e0);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        if (P.c_f32) {
            uint4 *df = reinterpret_cast<uint4 *>(P.c_f32 + e0);
#pragma unroll
            for (int q = 0; q < 4; ++q) df[q] = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
    }
}

// Tile t of the grouped order: groups of `group` M-tiles, walked column by
// column across N (M fastest inside a group).
__device__ __forceinline__ void tile_coords(uint32_t t, uint32_t tiles_m, uint32_t tiles_n, uint32_t &mt,
                                            uint32_t &nt, uint32_t group = kGroupM)
{
    const uint32_t group_size = group * tiles_n;
    const uint32_t first_m = (t / group_size) * group;
    const uint32_t gm = tiles_m - first_m < group ? tiles_m - first_m : group;
    const uint32_t local = t % group_size;
    mt = first_m + local % gm;
    nt = local / gm;
}

// Persistent: each CTA walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...
__global__ void __launch_bounds__(kThreads, 1)
gemm_bf16_sr_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ GemmParams P, uint64_t limit_ns)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;          // 1024-byte aligned for the 128-byte swizzle
    const uint32_t bars = base + kStages * kStageBytes;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (kStages + s); };
    auto acc_full = [&](int b) { return bars + 8u * (2 * kStages + b); };
    auto acc_empty = [&](int b) { return bars + 8u * (2 * kStages + kAccBufs + b); };
    const uint32_t tmem_slot = bars + 8u * (2 * kStages + 2 * kAccBufs);
    const uint32_t *tmem_slot_ptr = reinterpret_cast<const uint32_t *>(smem_raw + (tmem_slot - raw));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tiles_m = (P.m + kBM - 1) / kBM, tiles_n = (P.n + kBN - 1) / kBN;
    const uint32_t tiles = tiles_m * tiles_n;
    const int kblocks = static_cast<int>((P.k + kBK - 1) / kBK);     // a short last slice reads zeros past K

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), kEpilogueWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot_ptr;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------- producer
        uint32_t g = 0;                          // slices issued, over all tiles
        bool ok = true;
        for (uint32_t t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
            uint32_t mt, nt;
            tile_coords(t, tiles_m, tiles_n, mt, nt);
            for (int kb = 0; kb < kblocks; ++kb, ++g) {
                const int s = static_cast<int>(g % kStages);
                const uint32_t use = g / kStages;
                if (use > 0 && !mbar_wait(empty(s), (use - 1) & 1u, limit_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full(s), kStageBytes);
                const uint32_t dst = base + s * kStageBytes;
                tma_load_2d(dst, &map_a, kb * kBK, static_cast<int32_t>(mt * kBM), full(s));
                tma_load_2d(dst + kStageA, &map_b, kb * kBK, static_cast<int32_t>(nt * kBN), full(s));
            }
        }
        // the copies issued here must land before the CTA exits
        for (uint32_t s = 0; s < static_cast<uint32_t>(kStages) && s < g; ++s) {
            const uint32_t last_use = (g - 1 - s) / kStages;
            mbar_wait(full(static_cast<int>(s)), last_use & 1u, limit_ns);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------ MMA issuer
        uint32_t g = 0, i = 0;
        bool ok = true;
        for (uint32_t t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++i) {
            const int b = static_cast<int>(i % kAccBufs);
            const uint32_t ub = i / kAccBufs;
            if (ub > 0 && !mbar_wait(acc_empty(b), (ub - 1) & 1u, limit_ns)) break;   // epilogue done with b
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t d = tmem + static_cast<uint32_t>(b * kBN);
            for (int kb = 0; kb < kblocks; ++kb, ++g) {
                const int s = static_cast<int>(g % kStages);
                const uint32_t use = g / kStages;
                if (!mbar_wait(full(s), use & 1u, limit_ns)) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t sa = base + s * kStageBytes, sb = sa + kStageA;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    mma_bf16(d, smem_desc(sa + kk * 32), smem_desc(sb + kk * 32), (kb | kk) != 0);
                mma_commit(empty(s));           // the stage is free once these MMAs have read it
            }
            mma_commit(acc_full(b));            // fires when every MMA of this tile has completed
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------- epilogue
        const int quarter = warp & 3;                       // TMEM lanes this warp may read
        uint32_t i = 0;
        for (uint32_t t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
            const int b = static_cast<int>(i % kAccBufs);
            const uint32_t ub = i / kAccBufs;
            // tcgen05.ld is warp-collective: the warp agrees on readiness (and
            // reconverges) first; on a timeout it stops
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(acc_full(b), ub & 1u, limit_ns))) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            uint32_t mt, nt;
            tile_coords(t, tiles_m, tiles_n, mt, nt);
            const uint32_t row = mt * kBM + quarter * 32 + lane;
            const uint32_t n0 = nt * kBN;
            const uint32_t tq = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(b * kBN);
            const int ncols = static_cast<int>(P.n - n0) < kBN ? static_cast<int>(P.n - n0) : kBN;
            store_rows(P, tq, row, n0, ncols);
            // this warp is done reading accumulator b
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(b));
        }
    }
    // ------------------------------------------------------------ cleanup
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// ----------------------------------------------------- two-SM (CTA pair) form
//
// The same product with 256 x 256 tiles computed by a cluster of two CTAs on
// neighbouring SMs with tcgen05.mma.cta_group::2: each CTA stages its own 128
// rows of A and its own 128 rows (of N) of B, and one M=256, N=256 MMA
// issued by the pair's first CTA reads all four halves, leaving rows
// 0..127 of the tile in the first CTA's tensor memory and rows 128..255 in
// the second's, all 256 columns each.  Per FLOP every SM stages and reads a
// third less shared memory than with 128 x 256 tiles on one SM.
//   both CTAs, warp 0 lane 0: stream the CTA's halves of A and B, 128 deep
//       in K (two 64-column boxes each), into a 3-stage ring of 64 KB
//       stages; the bytes of both CTAs are counted on the FIRST CTA's
//       "full" barrier (.cta_group::2 bulk tensor copies may signal the
//       peer's barrier), which its producer arms with both CTAs' bytes;
//   both CTAs, warp 1: allocate / free the tensor memory as a pair; in the
//       first CTA its lane 0 issues the MMAs and commits them, multicast to
//       both CTAs: each box of a slice to that box's "empty" barrier (both
//       producers wait on their own), each tile to both "acc_full" barriers;
//   both CTAs, warps 2..5 (2..9, 2..17 for small K): the epilogue of the
//       CTA's 128 rows;
//       each warp hands the accumulator back by arriving on the FIRST CTA's
//       acc_empty barrier (2 x epilogue warps arrivals per tile).
// A slice whose rows lie wholly past M (or N) in the second half of a tile
// is read from row 0 instead: its products land only in rows (columns) the
// epilogue never stores, and no copy starts outside the matrix.
constexpr int kPairBM = 256;                // pair tile rows: 128 per CTA
constexpr int kPairBN = 256;                // pair tile columns: B rows, 128 staged per CTA
#ifndef ASR_GEMM_PDL
#define ASR_GEMM_PDL 1               // programmatic dependent launch: overlap the prologue with the previous kernel
#endif
#ifndef ASR_GEMM_PAIR_BK
#define ASR_GEMM_PAIR_BK 128
#endif
#ifndef ASR_GEMM_PAIR_STAGES
#define ASR_GEMM_PAIR_STAGES (ASR_GEMM_PAIR_BK == 128 ? 3 : 6)
#endif
#ifndef ASR_GEMM_PAIR_GROUP
#define ASR_GEMM_PAIR_GROUP 8
#endif
// Epilogue warps per CTA, a template parameter of the kernel: 4 (one per TMEM
// lane quarter) or 8 (two per quarter, half of the columns each).  The
// stochastic-rounding epilogue costs a Philox call per four outputs; below
// K ~ 1,024 it takes longer than the tile's MMAs and 8 warps hide more of it.
// Same-run TFLOP/s (4 / 8 warps): 8192^2 x 1024: 972-986 / 1,096-1,141;
// 8192^2 x 2048: 1,472-1,501 / 1,408-1,455; 8192^3: 1,716-1,764 / 1,730-1,759.
constexpr int kWideEpilogueMaxK = 1024;
constexpr int kWidestEpilogueMaxK = 512;
template <int EPI>
struct PairShape {
    static_assert(EPI == 4 || EPI == 8 || EPI == 16, "epilogue warps: 4, 8 or 16");
    static constexpr int kThreads = 64 + 32 * EPI;     // producer warp, MMA warp, epilogue
    static constexpr int kSpan = 256 / (EPI / 4);      // columns per epilogue warp
};
constexpr int kPairStages = ASR_GEMM_PAIR_STAGES;   // 64 KB (32 KB) stages: 3 (6) fit beside the barriers
constexpr int kPairGroupM = ASR_GEMM_PAIR_GROUP;    // tile order: 8 pair-tile rows walked across N
constexpr uint32_t kHalfA = 128 * kBK * 2;          // 16 KB per CTA
constexpr uint32_t kHalfB = 128 * kBK * 2;          // 16 KB per CTA
// K per stage: two 64-column boxes per operand, so each wait and commit of
// the MMA thread is spread over eight MMAs (1,024 tensor cycles) instead of
// four -- with 64 the thread's own per-slice cost (the full-barrier wait
// ~75 cycles, four MMA issues ~280, the multicast commit ~125, measured with
// clock64 on GB300) nearly used up the 512 cycles a slice keeps the tensor
// pipe busy, which held it at ~79 %.  Same-run TFLOP/s at 64 / 128:
// 8192^3 1,760-1,784 / 1,862-1,869; 4096^3 1,423-1,427 / 1,543-1,544;
// 8192^2 x 2048 1,504-1,517 / 1,649-1,664; 16384^2 x 8192 1,815-1,819 /
// 1,924-1,926.
constexpr int kPairBK = ASR_GEMM_PAIR_BK;
static_assert(kPairBK == 64 || kPairBK == 128, "K per stage: 64 or 128");
constexpr int kPairBoxes = kPairBK / 64;
constexpr uint32_t kPairStageBytes = kPairBoxes * (kHalfA + kHalfB);   // A boxes, then B boxes
// barriers: full/empty per stage, full/empty per accumulator, the MMA drain
// barriers: full per stage, empty per stage and box, full/empty per
// accumulator, the MMA drain; then the TMEM address slot
constexpr int kPairBars = kPairStages * (1 + kPairBoxes) + 2 * kAccBufs + 1;
constexpr int kPairSmem = 1024 + kPairStages * kPairStageBytes + kPairBars * 8 + 16;
constexpr uint32_t pair_instr_desc(uint32_t n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | (uint32_t(kPairBM >> 4) << 24);
}
constexpr uint32_t kPairInstrDesc = pair_instr_desc(kPairBN);           // M=256, N=256
constexpr uint32_t kPairInstrDescNarrow = pair_instr_desc(kPairBN / 2); // M=256, N=128

// Work item t of the pair schedule: its tile's first row and column and its
// width.  Items below P.wide are whole tiles in the grouped order; item
// P.wide + u is half (u & 1) of whole tile P.wide + u/2.  Splitting the tiles
// of a last, partly filled round in two (when their halves still fit in one
// round) halves that round's length.
__device__ __forceinline__ void pair_item(const GemmParams &P, uint32_t t, uint32_t tiles_m, uint32_t tiles_n,
                                          uint32_t &m0, uint32_t &n0, uint32_t &width)
{
    uint32_t mt, nt;
    if (t < P.wide) {
        tile_coords(t, tiles_m, tiles_n, mt, nt, kPairGroupM);
        n0 = nt * kPairBN;
        width = kPairBN;
    } else {
        const uint32_t u = t - P.wide;
        tile_coords(P.wide + u / 2, tiles_m, tiles_n, mt, nt, kPairGroupM);
        n0 = nt * kPairBN + (u & 1u) * (kPairBN / 2);
        width = kPairBN / 2;
    }
    m0 = mt * kPairBM;
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// An mbarrier wait that also orders what the other CTA of the cluster did
// before arriving (acquire at cluster scope); bounded like mbar_wait.
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// The pair kernel's waits: bounded like mbar_wait (time and poll count), but
// the timer is read only every 64 polls -- its reads sat on the path from a
// barrier's completion to the next MMA or copy (about 1 % at 8192^3).
template <bool CLUSTER>
__device__ __noinline__ bool pair_wait_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    const uint64_t t0 = global_ns();
    for (uint32_t polls = 1;; ++polls) {
        if (CLUSTER ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
        if ((polls & 63u) == 0 && (global_ns() - t0 > limit_ns || polls >= kWaitMaxPolls)) {
            atomicOr(&g_device_error, kErrWaitTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ bool pair_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_test(bar, parity)) return true;
    return pair_wait_slow<false>(bar, parity, limit_ns);
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_test_cluster(bar, parity)) return true;
    return pair_wait_slow<true>(bar, parity, limit_ns);
}

// Arrival of an epilogue warp on the first CTA's accumulator-empty barrier.
// Relaxed: the MMA warp waiting there reuses only the tensor memory, whose
// reads (tcgen05.ld) have completed at the epilogue's tcgen05.wait::ld, so
// nothing has to be released -- a release arrive at cluster scope would
// make the warp wait for its own global stores of the tile to be visible
// (measured as the "membar" stall, 1.3 per issued instruction at K = 512).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y,
                                                 uint32_t cluster_bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar)
        : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on the barrier at this offset in both CTAs of the pair when
// every MMA issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar)
{
    const uint16_t both = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(bar), "h"(both)
        : "memory");
}

// Persistent over pair tiles: cluster c walks tiles c, c + clusters, ...
template <int EPI>
__global__ void __launch_bounds__(PairShape<EPI>::kThreads, 1)
gemm_bf16_sr_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                         const __grid_constant__ CUtensorMap map_b_half, const __grid_constant__ GemmParams P,
                         uint64_t limit_ns)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;          // same offset in both CTAs
    const uint32_t bars = base + kPairStages * kPairStageBytes;
    auto full = [&](int s) { return bars + 8u * s; };
    // a stage is filled as a whole (one "full" barrier) but handed back box
    // by box (one "empty" barrier per 64-column box): the producer can start
    // refilling the first half while the MMAs still read the second
    auto empty = [&](int s, int j) { return bars + 8u * (kPairStages + s * kPairBoxes + j); };
    auto acc_full = [&](int b) { return bars + 8u * (kPairStages * (1 + kPairBoxes) + b); };
    auto acc_empty = [&](int b) { return bars + 8u * (kPairStages * (1 + kPairBoxes) + kAccBufs + b); };
    const uint32_t drained = bars + 8u * (kPairBars - 1);
    const uint32_t tmem_slot = drained + 8u;
    const uint32_t *tmem_slot_ptr = reinterpret_cast<const uint32_t *>(smem_raw + (tmem_slot - raw));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const uint32_t cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
    const uint32_t tiles_m = (P.m + kPairBM - 1) / kPairBM, tiles_n = (P.n + kPairBN - 1) / kPairBN;
    const uint32_t items = P.wide + P.narrow;
    const int kblocks = static_cast<int>((P.k + kPairBK - 1) / kPairBK);   // a short last slice reads zeros past K

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(full(s), 1);
            for (int j = 0; j < kPairBoxes; ++j) mbar_init(empty(s, j), 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), 2 * EPI);
        }
        mbar_init(drained, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }
    // both CTAs' barriers are initialised before either CTA signals the other's
    cluster_sync();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot_ptr;
#if ASR_GEMM_PDL
    // Launched with programmatic stream serialization, this grid may start
    // while the previous kernel on the stream is still finishing: everything
    // above touches only this CTA's shared and tensor memory; global memory
    // (A and B may be that kernel's output, C its input) waits until it has
    // completed.  The next kernel may be launched right away -- it does the
    // same wait before touching memory.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------- producer
        // stage s, its use count's parity, and whether every stage has been
        // used once (only then does a stage have to be waited for)
        uint32_t g = 0, s = 0, phase = 0;
        bool wrapped = false, ok = true;
        const uint32_t full0 = peer_addr(full(0), 0);       // the first CTA's barriers, 8 bytes apart
        for (uint32_t t = cluster; ok && t < items; t += clusters) {
            uint32_t m0, n0, width;
            pair_item(P, t, tiles_m, tiles_n, m0, n0, width);
            const bool half = width != kPairBN;             // each CTA stages 64 rows of B, not 128
            uint32_t ra = m0 + rank * 128, rb = n0 + rank * (width / 2);
            if (ra >= P.m) ra = 0;
            if (rb >= P.n) rb = 0;
            const uint32_t bytes = 2 * kPairBoxes * (kHalfA + (half ? kHalfB / 2 : kHalfB));
            const CUtensorMap *mapb = half ? &map_b_half : &map_b;
            for (int kb = 0; kb < kblocks; ++kb, ++g) {
                const uint32_t bar = full0 + 8u * s;
                const uint32_t dst = base + s * kPairStageBytes;
#pragma unroll
                for (int j = 0; j < kPairBoxes; ++j) {
                    if (wrapped && !pair_wait(empty(s, j), phase ^ 1u, limit_ns)) {
                        ok = false;
                        break;
                    }
                    // box 0 free means the MMAs have passed this stage's last
                    // fill, so the full barrier is armed for the new one
                    if (j == 0 && leader) mbar_arrive_expect_tx(full(s), bytes);
                    const int32_t x = kb * kPairBK + j * 64;
                    tma_load_2d_pair(dst + j * kHalfA, &map_a, x, static_cast<int32_t>(ra), bar);
                    tma_load_2d_pair(dst + kPairBoxes * kHalfA + j * kHalfB, mapb, x, static_cast<int32_t>(rb), bar);
                }
                if (!ok) break;
                if (++s == kPairStages) {
                    s = 0;
                    phase ^= 1u;
                    wrapped = true;
                }
            }
        }
        // the MMAs that read this CTA's stages have completed, and their
        // arrivals on its barriers have landed, before the CTA exits
        for (uint32_t q = 0; q < static_cast<uint32_t>(kPairStages) && q < g; ++q) {
            const uint32_t last_use = (g - 1 - q) / kPairStages;
            for (int j = 0; j < kPairBoxes; ++j) pair_wait(empty(static_cast<int>(q), j), last_use & 1u, limit_ns);
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------------ MMA issuer
        // The tensor pipe runs only as long as this thread keeps it fed: each
        // slice's wait, four MMAs and commit must take less than the slice's
        // 512 MMA cycles, so descriptors advance by constants and the stage
        // and its parity are counters (no division by the stage count).
        uint32_t s = 0, phase = 0, i = 0;
        bool ok = true;
        const uint64_t desc_a0 = smem_desc(base), desc_b0 = smem_desc(base + kPairBoxes * kHalfA);
        constexpr uint64_t kDescStage = kPairStageBytes >> 4;          // a stage in descriptor address units
        for (uint32_t t = cluster; ok && t < items; t += clusters, ++i) {
            const int b = static_cast<int>(i % kAccBufs);
            const uint32_t ub = i / kAccBufs;
            if (ub > 0 && !mbar_wait_cluster(acc_empty(b), (ub - 1) & 1u, limit_ns)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t d = tmem + static_cast<uint32_t>(b * kPairBN);
            const uint32_t idesc = t < P.wide ? kPairInstrDesc : kPairInstrDescNarrow;
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!pair_wait(full(s), phase, limit_ns)) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                // +2 per K=16 step: 32 bytes inside the 128-byte swizzle row;
                // the next 64 columns are the next box
                const uint64_t ad = desc_a0 + s * kDescStage, bd = desc_b0 + s * kDescStage;
#pragma unroll
                for (int j = 0; j < kPairBoxes; ++j) {
                    const uint64_t aj = ad + j * (kHalfA >> 4), bj = bd + j * (kHalfB >> 4);
                    mma_bf16_pair(d, aj, bj, idesc, (kb | j) != 0);
                    mma_bf16_pair(d, aj + 2, bj + 2, idesc, 1u);
                    mma_bf16_pair(d, aj + 4, bj + 4, idesc, 1u);
                    mma_bf16_pair(d, aj + 6, bj + 6, idesc, 1u);
                    mma_commit_pair(empty(s, j));      // this box is free once these MMAs have read it
                }
                if (++s == kPairStages) {
                    s = 0;
                    phase ^= 1u;
                }
            }
            mma_commit_pair(acc_full(b));
        }
        // every MMA issued here has completed before the pair may free its
        // tensor memory or leave (also after a timeout)
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(drained)
                     : "memory");
        pair_wait(drained, 0, limit_ns);
    } else if (warp >= 2) {
        // ------------------------------------------------------- epilogue
        // a warp reads the TMEM lane quarter warp % 4; with 8 warps, two
        // warps share a quarter and take half of the columns each
        const int quarter = warp & 3;
        constexpr int kSpan = PairShape<EPI>::kSpan;
        const int c_lo = ((warp - 2) / 4) * kSpan;
        uint32_t i = 0;
        for (uint32_t t = cluster; t < items; t += clusters, ++i) {
            const int b = static_cast<int>(i % kAccBufs);
            const uint32_t ub = i / kAccBufs;
            if (!__all_sync(0xFFFFFFFFu, pair_wait(acc_full(b), ub & 1u, limit_ns))) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            uint32_t m0, n0, width;
            pair_item(P, t, tiles_m, tiles_n, m0, n0, width);
            const uint32_t row = m0 + rank * 128 + quarter * 32 + lane;
            const uint32_t tq =
                tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(b * kPairBN);
            // the second half of a tile can lie wholly past N: nothing to store
            const int ncols = n0 >= P.n ? 0 : P.n - n0 < width ? static_cast<int>(P.n - n0) : static_cast<int>(width);
            const int c_hi = ncols < c_lo + kSpan ? ncols : c_lo + kSpan;
            if (c_hi > c_lo) store_rows(P, tq + c_lo, row, n0 + c_lo, c_hi - c_lo);
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(peer_addr(acc_empty(b), 0));
        }
    }
    // ------------------------------------------------------------ cleanup
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// Tensor-map encoder from the driver, fetched through the runtime (the
// library does not link libcuda).
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;

asr_status encoder(PFN_cuTensorMapEncodeTiled_v12000 *out)
{
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return cuda_fail(e);
        if (q != cudaDriverEntryPointSuccess || !fn) return cuda_fail(cudaErrorNotSupported);
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return ASR_OK;
}

// Per device, once: opt both kernels in to their dynamic shared memory
// (above the default 48 KB) and find how many CTA pairs of the two-SM kernel
// can be resident at once (pairs sit on neighbouring SMs, so on a GPU with an
// odd number of SMs somewhere fewer than SMs/2 fit).
bool g_gemm_ready[kMaxDevices];
int g_gemm_sms[kMaxDevices];
int g_gemm_pairs[kMaxDevices][3];

template <int EPI>
cudaError_t pair_setup(int n_sms, int *n_pairs)
{
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_sr_pair_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kPairSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(n_sms & ~1), 1, 1);
    cfg.blockDim = dim3(PairShape<EPI>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = kPairSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n_pairs, gemm_bf16_sr_pair_kernel<EPI>, &cfg);
}

// pairs[0], [1], [2]: resident pairs of the kernel with 4, 8, 16 epilogue warps
asr_status device_setup(int *sms, int pairs[3])
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ASR_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (!g_gemm_ready[dev]) {
        e = cudaFuncSetAttribute(gemm_bf16_sr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        int n_sms = 0, p4 = 0, p8 = 0, p16 = 0;
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = pair_setup<4>(n_sms, &p4);
        if (e == cudaSuccess) e = pair_setup<8>(n_sms, &p8);
        if (e == cudaSuccess) e = pair_setup<16>(n_sms, &p16);
        if (e != cudaSuccess) return cuda_fail(e);
        g_gemm_sms[dev] = n_sms;
        g_gemm_pairs[dev][0] = p4;
        g_gemm_pairs[dev][1] = p8;
        g_gemm_pairs[dev][2] = p16;
        g_gemm_ready[dev] = true;
    }
    *sms = g_gemm_sms[dev];
    pairs[0] = g_gemm_pairs[dev][0];
    pairs[1] = g_gemm_pairs[dev][1];
    pairs[2] = g_gemm_pairs[dev][2];
    return ASR_OK;
}

// The pair schedule for `tiles` whole tiles on up to `pairs` resident pairs:
// whole tiles round by round; if the last round is at most half full, its
// tiles go as halves (twice the items, each half as long), so the round
// takes half the time.  Returns the number of clusters to launch.
unsigned pair_schedule(uint64_t tiles, uint64_t pairs, GemmParams &P)
{
    uint64_t rest = tiles % pairs;                   // tiles of the last, partly filled round
    if (tiles < pairs) rest = tiles;
    const bool split = rest > 0 && 2 * rest <= pairs;
    P.wide = static_cast<uint32_t>(tiles - (split ? rest : 0));
    P.narrow = static_cast<uint32_t>(split ? 2 * rest : 0);
    const uint64_t items = P.wide + static_cast<uint64_t>(P.narrow);
    return static_cast<unsigned>(items < pairs ? items : pairs);
}

template <int EPI>
asr_status launch_pair(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mb_half, GemmParams &P,
                       uint64_t tiles, int pairs, cudaStream_t stream)
{
    const unsigned clusters = pair_schedule(tiles, static_cast<uint64_t>(pairs), P);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(PairShape<EPI>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = kPairSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = ASR_GEMM_PDL ? 2 : 1;
    const uint64_t limit = kWaitLimitNs;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_bf16_sr_pair_kernel<EPI>, ma, mb, mb_half, P, limit);
    if (e != cudaSuccess) return cuda_fail(e);
    return launched(ASR_KERNEL_GEMM);
}

// Row-major rows x k bf16 matrix, boxes of box_rows x 64 with 128-byte swizzle.
asr_status make_map(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t k, uint32_t box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    asr_status st = encoder(&enc);
    if (st != ASR_OK) return st;
    const cuuint64_t dims[2] = {k, rows};
    const cuuint64_t strides[1] = {k * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ASR_OK : ASR_ERR_INVALID_VALUE;
}

asr_status run(const uint16_t *a, const uint16_t *b, uint16_t *c, float *c_f32, uint64_t m, uint64_t n,
               uint64_t k, uint32_t rounding, uint32_t step, uint64_t seed, cudaStream_t stream)
{
    if (rounding != ASR_ROUND_SR && rounding != ASR_ROUND_RNE) return ASR_ERR_UNSUPPORTED_DTYPE;
    if (m == 0 || n == 0) return ASR_OK;
    if (!a || !b || !c) return ASR_ERR_INVALID_VALUE;
    if (n % 16 || k == 0 || k % 8) return ASR_ERR_INVALID_VALUE;
    if (m > (1u << 24) || n > (1u << 24) || k > (1u << 24)) return ASR_ERR_INVALID_VALUE;
    // the tile index is 32-bit: checked here, before any CUDA call, on the
    // larger two-SM tiles (the one-SM fallback's own count is checked later)
    if (((m + 255) / 256) * ((n + 255) / 256) >= (1ull << 31)) return ASR_ERR_INVALID_VALUE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(c) || (c_f32 && !aligned16(c_f32)))
        return ASR_ERR_INVALID_VALUE;
    int sms = 0, pairs[3] = {0, 0, 0};
    asr_status st = device_setup(&sms, pairs);
    if (st != ASR_OK) return st;
    GemmParams P;
    P.c = c;
    P.c_f32 = c_f32;
    P.m = static_cast<uint32_t>(m);
    P.n = static_cast<uint32_t>(n);
    P.k = static_cast<uint32_t>(k);
    P.step = step;
    P.rounding = rounding;
    // rows are 32-byte multiples apart (n % 16 == 0), so every lane's
    // 16-column piece is 32-byte aligned when c is
    P.c_align32 = (reinterpret_cast<uintptr_t>(c) & 31u) == 0 ? 1u : 0u;
    P.wide = 0;
    P.narrow = 0;
    P.keys = make_keys(seed);
    CUtensorMap ma, mb;
#if ASR_GEMM_PAIR
    int shape = k <= static_cast<uint64_t>(kWidestEpilogueMaxK) ? 2
                : k <= static_cast<uint64_t>(kWideEpilogueMaxK) ? 1 : 0;
    // When every tile fits in one round of resident pairs, no tile's
    // epilogue overlaps another's MMAs: the widest epilogue then shortens
    // the step at any K (SR at 2048^3: 886 against 767 TFLOP/s).
    const uint64_t pair_tiles = ((m + kPairBM - 1) / kPairBM) * ((n + kPairBN - 1) / kPairBN);
    if (pairs[2] > 0 && pair_tiles <= static_cast<uint64_t>(pairs[2])) shape = 2;
    if (pairs[shape] > 0) {
        // two-SM form: both operands in 128-row boxes (one half per CTA)
        CUtensorMap mb_half;
        st = make_map(&ma, a, m, k, 128);
        if (st == ASR_OK) st = make_map(&mb, b, n, k, 128);
        if (st == ASR_OK) st = make_map(&mb_half, b, n, k, 64);     // B halves of split tiles
        if (st != ASR_OK) return st;
        const uint64_t tiles = ((m + kPairBM - 1) / kPairBM) * ((n + kPairBN - 1) / kPairBN);
        if (tiles >= (1ull << 31)) return ASR_ERR_INVALID_VALUE;
        if (shape == 2) return launch_pair<16>(ma, mb, mb_half, P, tiles, pairs[2], stream);
        if (shape == 1) return launch_pair<8>(ma, mb, mb_half, P, tiles, pairs[1], stream);
        return launch_pair<4>(ma, mb, mb_half, P, tiles, pairs[0], stream);
    }
#endif
    st = make_map(&ma, a, m, k, kBM);
    if (st == ASR_OK) st = make_map(&mb, b, n, k, kBN);
    if (st != ASR_OK) return st;
    const uint64_t tiles = ((m + kBM - 1) / kBM) * ((n + kBN - 1) / kBN);
    if (tiles >= (1ull << 31)) return ASR_ERR_INVALID_VALUE;
    const unsigned grid = static_cast<unsigned>(tiles < static_cast<uint64_t>(sms) ? tiles : sms);
    gemm_bf16_sr_kernel<<<grid, kThreads, kSmem, stream>>>(ma, mb, P, kWaitLimitNs);
    return launched(ASR_KERNEL_GEMM);
}

}  // namespace gemm
