// adamw_kernels.cuh -- the fused AdamW-SR kernels: the register-resident kernel
// (any alignment) and the bulk-copy pipelined kernel (the hot path).
// Included by asr.cu inside its anonymous namespace (one translation unit).

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

// A4: the tensor's base index is a multiple of 4, so the unit's eight random
// words come from two Philox counters; otherwise from three (unit_words).
template <int PT, int GT, int RM, bool A4 = true>
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
            unit_words<A4>(T.base, e, P.step, P.keys, r);
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

template <int PT, int GT>
struct TmaStage {
    static constexpr int kTile = TmaShape<PT, GT>::kTile;
    static constexpr int kPBytes = kTile * (PT == ASR_BF16 ? 2 : 4);
    static constexpr int kGBytes = kTile * (GT == ASR_BF16 ? 2 : 4);
    static constexpr int kMBytes = kTile * 4;
    static constexpr int kBytes = kPBytes + kGBytes + 2 * kMBytes;
    // as many stages as fit in the shared-memory budget, at most ASR_TMA_STAGES
    static constexpr int kFit = ASR_TMA_SMEM_KB * 1024 / kBytes;
    static constexpr int kStages = kFit < ASR_TMA_STAGES ? kFit : ASR_TMA_STAGES;
    static_assert(kStages >= 2, "need at least two stages");
    static_assert(kBytes % 16 == 0, "stage size keeps 16-byte alignment");
    // after the stages: full[] and empty[] barriers and the tile index of each
    // stage (8 B each), the schedule barrier (8 B), the 16-byte schedule
    // answer (16-byte aligned), one dependency word per consumer warp
    static constexpr int kBarOff = kStages * kBytes;
    static constexpr int kTileSlotOff = kBarOff + 16 * kStages;
    static constexpr int kClcBarOff = kTileSlotOff + 8 * kStages;
    static constexpr int kClcBufOff = (kClcBarOff + 8 + 15) / 16 * 16;
    static constexpr int kDepOff = kClcBufOff + 16;
    static constexpr int kSmem = kDepOff + TmaShape<PT, GT>::kWarps * 4;
};

// Tile schedule of the pipelined kernel: dynamic (cluster launch control, a
// grid of one CTA per tile) unless built with ASR_TMA_DYNAMIC=0 (a persistent
// grid walking the tiles with a fixed stride).
#ifndef ASR_TMA_DYNAMIC
#define ASR_TMA_DYNAMIC 1
#endif
constexpr uint64_t kNoTile = ~0ull;

// Locate tile `tile` (of tile_elems elements) of a descriptor table, advancing
// the cursor t.  Tab is AdamTable<CAP> (descriptors in the launch parameters)
// or any type with the same `t[]` and `total_tiles` members.
template <typename Tab>
__device__ __forceinline__ void find_tile(const Tab &tab, uint64_t tile, uint32_t tile_elems, int &t,
                                          uint64_t &off, uint32_t &cnt)
{
    if (t > 0 && tile < tab.t[t - 1].tile_end) t = 0;     // tiles normally come in rising order
    while (tile >= tab.t[t].tile_end) ++t;
    const uint64_t first = t == 0 ? 0 : tab.t[t - 1].tile_end;
    off = (tile - first) * static_cast<uint64_t>(tile_elems);
    const uint64_t rest = tab.t[t].n - off;
    cnt = rest < static_cast<uint64_t>(tile_elems) ? static_cast<uint32_t>(rest) : tile_elems;
}

// The body of the pipelined step, shared by the kernels that differ only in
// where their descriptor table lives.  Every tensor has 16-byte-aligned
// buffers, and with A4 a base index that is a multiple of 4 (without A4 the
// bases may be anything: each unit then draws three Philox counters instead
// of two); tile and block shape TmaShape<PT, GT>.
//
// The producer decides which tile each stage holds and writes the tile's
// index into the stage's slot before the stage's barrier completes; the
// consumers read it after their wait (the barrier orders the two), and a
// slot holding kNoTile ends their loop.
template <int PT, int GT, int RM, bool A4, typename Tab>
__device__ __forceinline__ void tma_step(const Tab &tab, const AdamParams &P, uint64_t limit_ns)
{
    using S = TmaStage<PT, GT>;
    using SH = TmaShape<PT, GT>;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = smem_addr(smem);
    auto full = [&](int s) { return sbase + S::kBarOff + 8u * s; };
    auto empty = [&](int s) { return sbase + S::kBarOff + 8u * (S::kStages + s); };
    auto slot = [&](int s) { return sbase + S::kTileSlotOff + 8u * s; };
    const uint32_t clc_bar = sbase + S::kClcBarOff, clc_buf = sbase + S::kClcBufOff;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), SH::kWarps);
        }
        mbar_init(clc_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == SH::kWarps) {
        // ------------------------------------------------------ producer
        if (lane != 0) return;
        uint64_t policy;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
        int t = 0;
        uint32_t k = 0;
        uint64_t tile = blockIdx.x;           // a CTA's first tile is its own
#if ASR_TMA_DYNAMIC
        // one request for the next tile is always in flight, so its answer is
        // there by the time a stage frees up
        uint32_t clc_phase = 0;
        bool asking = true;
        mbar_arrive_expect_tx(clc_bar, 16);
        clc_try_cancel(clc_buf, clc_bar);
#endif
        for (;; ++k) {
            const int s = static_cast<int>(k % S::kStages);
            const uint32_t use = k / S::kStages;
            if (use > 0 && !mbar_wait(empty(s), (use - 1) & 1u, limit_ns)) break;
            if (tile >= tab.total_tiles) {
                st_shared_u64(slot(s), kNoTile);
                mbar_arrive(full(s));
                ++k;
                break;
            }
            uint64_t off;
            uint32_t cnt;
            find_tile(tab, tile, S::kTile, t, off, cnt);
            const TensorEntry &T = tab.t[t];
            const uint32_t c8 = cnt & ~7u;
            const uint32_t pb = c8 * (PT == ASR_BF16 ? 2u : 4u), gb = c8 * (GT == ASR_BF16 ? 2u : 4u);
            const uint32_t mb = c8 * 4u;
            st_shared_u64(slot(s), tile);
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
#if ASR_TMA_DYNAMIC
            // the next tile: the one whose launch the pending request cancelled;
            // none once a request finds no CTA left (and no request is made
            // after that)
            tile = kNoTile;
            if (asking) {
                asking = false;
                if (mbar_wait(clc_bar, clc_phase, limit_ns)) {
                    clc_phase ^= 1u;
                    uint32_t x;
                    if (clc_answer(clc_buf, x)) {
                        tile = x;
                        asking = true;
                        mbar_arrive_expect_tx(clc_bar, 16);
                        clc_try_cancel(clc_buf, clc_bar);
                    }
                }
            }
#else
            tile += gridDim.x;
#endif
        }
        // Every copy this thread issued must land before the CTA may exit:
        // wait (bounded) for the last use of each stage; likewise for a
        // schedule request still in flight (only after a failed wait).
        const uint32_t issued = k;
        for (int s = 0; s < S::kStages; ++s) {
            if (static_cast<uint32_t>(s) >= issued) break;
            const uint32_t last_use = (issued - 1 - s) / S::kStages;
            mbar_wait(full(s), last_use & 1u, limit_ns);
        }
#if ASR_TMA_DYNAMIC
        if (asking) mbar_wait(clc_bar, clc_phase, limit_ns);
#endif
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ct = threadIdx.x;            // 0 .. SH::kConsumers-1
    const uint32_t dep_slot = sbase + S::kDepOff + 4u * warp;   // one word per consumer warp
    int t = 0;
    for (uint32_t k = 0;; ++k) {
        const int s = static_cast<int>(k % S::kStages);
        const uint32_t use = k / S::kStages;
        if (!mbar_wait(full(s), use & 1u, limit_ns)) return;
        const uint64_t tile = ld_shared_u64(slot(s));
        if (tile == kNoTile) return;
        uint64_t off;
        uint32_t cnt;
        find_tile(tab, tile, S::kTile, t, off, cnt);
        const TensorEntry &T = tab.t[t];
        const uint32_t c8 = cnt & ~7u;
        const unsigned char *st = smem + s * S::kBytes;
        VecUnit<PT, GT> u[SH::kUnits];
#pragma unroll
        for (int j = 0; j < SH::kUnits; ++j) {
            const uint32_t e = (static_cast<uint32_t>(j) * SH::kConsumers + ct) * kVec;
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
        for (int j = 0; j < SH::kUnits; ++j) {
            const uint32_t e = (static_cast<uint32_t>(j) * SH::kConsumers + ct) * kVec;
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
        for (int j = 0; j < SH::kUnits; ++j) {
            const uint32_t e = (static_cast<uint32_t>(j) * SH::kConsumers + ct) * kVec;
            if (e < c8) vec_compute_store<PT, GT, RM, A4>(T, off + e, u[j], P);
        }
        // a ragged end of a tensor (< 8 elements) goes through the scalar path
        if (c8 < cnt && ct == (c8 / kVec) % SH::kConsumers) scalar_unit<PT, GT, RM>(T, off + c8, P);
    }
}

// Descriptor table in the launch parameters (up to CAP tensors).
template <int PT, int GT, int RM, int CAP, bool A4>
__global__ void __launch_bounds__(TmaShape<PT, GT>::kThreads, 1)
adamw_sr_tma_kernel(const __grid_constant__ AdamTable<CAP> tab, const __grid_constant__ AdamParams P,
                    uint64_t limit_ns)
{
    tma_step<PT, GT, RM, A4>(tab, P, limit_ns);
}
