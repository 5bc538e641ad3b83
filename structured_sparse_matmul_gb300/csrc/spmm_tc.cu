// V:N:M SpMM on Blackwell's 2:4 sparse tensor cores (tcgen05.mma.sp).
//
// VENOM: A Vectorized N:M Format for Unleashing the Power of Sparse Tensor
// Cores, section 4 (Figure 4): the V:N:M matrix is run on 2:4 sparse tensor
// cores as an R x (K/M*4) operand, each block's column-loc selecting 4 of
// its M rows of B; section 4.1 (Figures 5-8): a thread-block tile spans V
// rows (BSr = V), column-loc is fetched ahead of the B rows it selects, and
// the output tile is written back with wide, coalesced stores.
//
// GB300 design: persistent CTAs (at most one per SM and TMEM share), each
// taking tiles b, b + grid, ... of C (tile_m x tile_n over a range of the
// condensed K; tile_m = 128, or 64 when V = 64 and column-loc differs per
// 64-row block); n varies fastest, so the CTAs running at one time share A
// rows in L2. Per 128-column stage of the condensed K (4 MMA k-steps):
//   warp 0    TMA producer. Per stage: one tiled load of the A values
//             (tile_m rows x 64 values, 128B swizzle; MMA k-step s reads bytes
//             32s..32s+31 of each row) and one of the m-indices (tile_m rows x
//             16 bytes), on their own barrier, and, when M == 4 (column-loc is
//             the identity), the B rows as plain tiled loads on a second one.
//             TMA instructions cost the SM's copy engine ~100 cycles each
//             however small, so a stage issues as few as possible.
//   warps 10+ (M > 4) the B gather: per stage these warps copy the 128
//             selected B rows (4 per block, tile_n columns each) with 16-byte
//             cp.async, coalesced along each row, straight into the
//             128B-swizzled operand layout (zero-filled past N); the
//             column-loc words that select the rows are loaded four stages
//             ahead; each thread's copies arrive on the stage's barrier by
//             themselves when they land (cp.async.mbarrier.arrive), so every
//             pipeline stage can be in flight; the MMA thread fences the
//             generic-proxy writes into the async proxy after acquiring the
//             barrier.
//   warps 2-5 per stage, as soon as A and the m-indices landed (B may still
//             be in flight): read their rows' m-index words from shared memory,
//             pair them the way the sparse MMA reads them (rows i and i+8 of
//             each 16-row group share their 16-bit halves between TMEM lanes
//             i and i+8) and write them to TMEM (tcgen05.st), each MMA's word
//             in its own 8-column-aligned slot.
//   warp 1    TMEM owner and MMA issuer (one thread): 4 sparse MMAs of
//             M=tile_m, N=tile_n, K=32 per stage into an fp32 accumulator in
//             TMEM; tcgen05.commit releases the stage, and the tile's
//             accumulator to the epilogue. Two accumulators alternate between
//             tiles when TMEM holds them (tile_n <= 192).
//   warps 6-9 epilogue: TMEM -> registers (tcgen05.ld) -> fp16 (RNE) or
//             fp32 -> global, each thread writing whole 32-byte sectors of
//             its row (fp32 partials to the workspace under split-K), while
//             the other warps already run the next tile; then they release
//             the accumulator (with a single accumulator and 64-row tiles
//             the m-index warps drain half of its columns). With M=128 row r
//             of the tile lives in TMEM lane r; with M=64 in lane
//             32*(r/16) + r%16 (lanes 16..31 of each quarter stay unused).
// Every mbarrier wait is bounded: on time-out the CTA records
// VNM_ERR_TIMEOUT, drains what it already issued, frees TMEM and returns.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "vnm_internal.h"
#include "vnm_ptx.cuh"

namespace vnm {
namespace {

constexpr int kTcWarpsFixed = 10;  // warps 0-9; gathering CTAs add gather warps after them
constexpr int kEpiWarp0 = 6;       // warps 6-9: epilogue
constexpr int kKTile = 128;        // condensed K per stage = 4 MMAs of K = 32
constexpr int kValsPerKTile = 64;  // stored values per row per stage (128 bytes)
constexpr int kMetaSlotCols = 8;   // TMEM columns between consecutive MMAs' m-index words
constexpr int kMetaStageCols = 4 * kMetaSlotCols;
// Sleep between polls of a barrier, per role (ns): the MMA thread polls
// flat out; the others park so that ~20 waiting warps do not take the issue
// slots of the ones doing work. The epilogue waits a whole tile.
constexpr uint32_t kSleepProducer = 32;
constexpr uint32_t kSleepMeta = 64;
constexpr uint32_t kSleepGather = 64;
constexpr uint32_t kSleepEpilogue = 256;
// m-index word of a row that lies beyond R: slots (0, 1) in all 8 groups
constexpr uint32_t kPadMeta = 0x44444444u;

struct TcArgs {
    const uint32_t* colidx;  // [R/V][nblk] words of 4 column bytes
    const uint16_t* B;       // K x N fp16 (ld_b), read by the gather warps
    int64_t ld_b;
    void* C;
    int64_t ld_c;
    float* partial;          // [splits][R][N] fp32, or null
    int64_t R, N;
    int V, M;
    int64_t nblk;
    int num_kt;              // condensed K / kKTile
    int kt_per_split;
    int n_tiles, m_tiles;    // tile grid: tile t -> (n = t % n_tiles, m = t / n_tiles % m_tiles, split)
    int total_tiles;
    int c_f32;
    int vec_store;           // C row starts 16-byte aligned
    int skip_stage;          // tests of the bounded waits: CTA 0 never issues this stage's loads (-1: none)
    int* status;
};

__host__ __device__ constexpr int pow2_at_least(int x) {
    int p = 32;
    while (p < x) p *= 2;
    return p;
}

template <int TM, int BN, bool NARROW>
struct TcCfg {
    static constexpr int kAtoms = (BN + 63) / 64;            // 64-column swizzle atoms of B
    static constexpr int kABytes = TM * 128;                 // TM rows x 64 values, 128B swizzle
    // per atom: 128 rows x 128 B; narrow: 128 rows x BN x 2 B
    static constexpr int kBBytes = NARROW ? kKTile * BN * 2 : kAtoms * kKTile * 128;
    static constexpr int kEBytes = TM * 16;                  // 4 m-index words per row
    static constexpr int kStageBytes = kABytes + kBBytes + kEBytes;
    static constexpr int kStages = tc_stages_for(TM, BN, NARROW);
    // two accumulators (the epilogue of one tile overlaps the next tile's
    // main loop) when they fit TMEM beside the m-index slots
    static constexpr int kAccBufs = 2 * BN + kStages * kMetaStageCols <= 512 ? 2 : 1;
    static constexpr int kTmemCols = pow2_at_least(kAccBufs * BN + kStages * kMetaStageCols);
    static constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
    static_assert(kStages >= 2, "pipeline depth");
    static_assert(BN + kStages * kMetaStageCols <= 512, "TMEM budget");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(TM == 64 || TM == 128, "MMA M");
};

// Gather threads of a gathering CTA: the gathered B tile needs many 16-byte
// copies in flight per SM (one CTA per SM): 16 warps (measured 1-5 % faster
// than 8 for 128-row tiles too); never more threads than 16-byte chunks per
// stage (kKTile * BN / 8).
__host__ __device__ constexpr int gather_threads(int tm, int bn) {
    // 192 columns are 24 chunks a row: a multiple of 24 threads, 8 rows each
    return (void)tm, bn == 192 ? 384 : 512 < kKTile * bn / 8 ? 512 : kKTile * bn / 8;
}

template <int TM, int BN, bool GATHER>
__host__ __device__ constexpr int tc_threads() {
    return kTcWarpsFixed * 32 + (GATHER ? gather_threads(TM, BN) : 0);
}

// TMEM lane quarter q (warp % 4), lane l -> row of the tile (or -1).
template <int TM>
__device__ __forceinline__ int tile_row_of_lane(int q, int l) {
    if (TM == 128) return 32 * q + l;
    return l < 16 ? 16 * q + l : -1;
}

struct TileGeom {
    int64_t m0, n0;  // first row and column of the C tile
    int split;       // K split
    int kt0, nkt;    // first stage (of kKTile condensed columns) and stage count
};

__device__ __forceinline__ TileGeom tile_geom(const TcArgs& p, int t, int tm, int bn) {
    TileGeom g;
    const int n_idx = t % p.n_tiles;
    const int rest = t / p.n_tiles;
    const int m_idx = rest % p.m_tiles;
    g.split = rest / p.m_tiles;
    g.m0 = static_cast<int64_t>(m_idx) * tm;
    g.n0 = static_cast<int64_t>(n_idx) * bn;
    g.kt0 = g.split * p.kt_per_split;
    g.nkt = min(p.num_kt, g.kt0 + p.kt_per_split) - g.kt0;
    return g;
}

// Columns [c0, c1) of this warp's lanes of an accumulator (TMEM address
// `tacc`: the buffer's column 0 in this warp's lane quarter) -> registers ->
// C (fp16, RNE, or fp32) or the split-K partials; `row` is this thread's row
// of C (>= R: none). Each thread writes whole 32-byte sectors of its row.
template <int BN>
__device__ __forceinline__ void drain_columns(const TcArgs& p, const TileGeom& g, uint32_t tacc, int64_t row, int c0,
                                              int c1) {
    // one 16-column chunk of this thread's row: fp32 partials, fp32 or fp16 C
    auto store16 = [&](const uint32_t (&v)[16], int c) {
        const int64_t col = g.n0 + c;
        if (row >= p.R || col >= p.N) return;
        const bool full = col + 16 <= p.N;
        if (p.partial != nullptr) {
            float* dst = p.partial + (static_cast<int64_t>(g.split) * p.R + row) * p.N + col;
            if (full && (p.N % 4) == 0) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    reinterpret_cast<uint4*>(dst)[u] = make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            } else {
                for (int u = 0; u < 16 && col + u < p.N; ++u) dst[u] = __uint_as_float(v[u]);
            }
        } else if (p.c_f32) {
            float* dst = static_cast<float*>(p.C) + row * p.ld_c + col;
            if (full && p.vec_store) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    reinterpret_cast<uint4*>(dst)[u] = make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            } else {
                for (int u = 0; u < 16 && col + u < p.N; ++u) dst[u] = __uint_as_float(v[u]);
            }
        } else {
            __half* dst = static_cast<__half*>(p.C) + row * p.ld_c + col;
            uint32_t h[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const __half2 t2 = __floats2half2_rn(__uint_as_float(v[2 * u]), __uint_as_float(v[2 * u + 1]));
                h[u] = *reinterpret_cast<const uint32_t*>(&t2);
            }
            if (full && p.vec_store) {
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(h[0], h[1], h[2], h[3]);
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(h[4], h[5], h[6], h[7]);
            } else {
                for (int u = 0; u < 16 && col + u < p.N; ++u)
                    dst[u] = __float2half_rn(__uint_as_float(v[u]));
            }
        }
    };
    // two TMEM loads in flight per wait
    constexpr int kEpiStep = BN >= 32 ? 32 : 16;
#pragma unroll 1
    for (int c = c0; c < c1; c += kEpiStep) {
        uint32_t v0[16], v1[16];
        tmem_ld_32x32b_x16(tacc + c, v0);
        if (kEpiStep == 32) tmem_ld_32x32b_x16(tacc + c + 16, v1);
        tmem_wait_ld();
        store16(v0, c);
        if (kEpiStep == 32) store16(v1, c + 16);
    }
}

// Persistent: CTA b takes tiles b, b + gridDim.x, ... (all roles walk the
// same sequence, so their stage and accumulator counters agree).
template <int TM, int BN, bool GATHER>
__global__ void __launch_bounds__(tc_threads<TM, BN, GATHER>(), 1)
    spmm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_e,
                   const __grid_constant__ CUtensorMap tm_b, const TcArgs p) {
    using Cfg = TcCfg<TM, BN, tc_narrow_b(BN, GATHER)>;
    constexpr int STAGES = Cfg::kStages;
    constexpr int ACC = Cfg::kAccBufs;
    constexpr int kGatherThreads = gather_threads(TM, BN);
    // With a single accumulator the next tile's MMAs wait for the whole
    // drain, so for 64-row tiles (16 rows per warp: the drain is bound by
    // TMEM load latency, not by the stores) the m-index warps, idle then,
    // drain the upper half of the columns while the epilogue warps drain the
    // lower half. (128-row tiles measured slower this way: their drain is
    // bound by the stores, and the next tile's m-indices wait.)
    constexpr bool kSplitEpi = ACC == 1 && BN >= 64 && TM == 64;
    constexpr int kEpiCols = kSplitEpi ? BN / 2 : BN;  // columns [0, kEpiCols) drained by the epilogue warps
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t ae_bar[STAGES];     // A values and m-indices landed (TMA)
    __shared__ __align__(8) uint64_t b_bar[STAGES];      // B rows landed (TMA, or every gather thread)
    __shared__ __align__(8) uint64_t meta_bar[STAGES];   // m-indices written to TMEM (4 warps)
    __shared__ __align__(8) uint64_t empty_bar[STAGES];  // MMAs done with the stage
    __shared__ __align__(8) uint64_t accf_bar[ACC];      // accumulator complete (MMA commit)
    __shared__ __align__(8) uint64_t acce_bar[ACC];      // accumulator read out (4 epilogue warps)
    __shared__ __align__(8) uint64_t done_bar;           // every MMA of this CTA complete
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    // B stages first: a B descriptor read stays inside this CTA's allocation
    // even if its two strides were interpreted the other way round.
    const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sB0 = smem_base;
    const uint32_t sA0 = sB0 + STAGES * Cfg::kBBytes;
    const uint32_t sE0 = sA0 + STAGES * Cfg::kABytes;
    const uint8_t* sE_generic = smem_raw + (sE0 - smem_u32(smem_raw));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&ae_bar[s]), 1);
            mbar_init(smem_u32(&b_bar[s]), GATHER ? kGatherThreads : 1);
            mbar_init(smem_u32(&meta_bar[s]), 4);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < ACC; ++b) {
            mbar_init(smem_u32(&accf_bar[b]), 1);
            mbar_init(smem_u32(&acce_bar[b]), kSplitEpi ? 8 : 4);
        }
        mbar_init(smem_u32(&done_bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_e);
        tma_prefetch_desc(&tm_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_acc = tmem_slot;           // columns [0, ACC*BN): fp32 accumulators
    const uint32_t tmem_e = tmem_slot + ACC * BN;  // then STAGES*32 columns of m-index words
    volatile int* abort = &abort_flag;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        int last_it[STAGES];
#pragma unroll
        for (int s = 0; s < STAGES; ++s) last_it[s] = -1;
        int it = 0;
        bool run = true;
        for (int t = static_cast<int>(blockIdx.x); run && t < p.total_tiles; t += static_cast<int>(gridDim.x)) {
            const TileGeom g = tile_geom(p, t, TM, BN);
            for (int k = 0; k < g.nkt; ++k, ++it) {
                const int slot = it % STAGES;
                const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
                const bool ok = mbar_wait_warp(smem_u32(&empty_bar[slot]), ph ^ 1u, abort, kSleepProducer);
                if (!ok) {
                    run = false;
                    break;
                }
                const int kt = g.kt0 + k;
                const uint32_t aeb = smem_u32(&ae_bar[slot]);
                const uint32_t sA = sA0 + slot * Cfg::kABytes;
                const uint32_t sB = sB0 + slot * Cfg::kBBytes;
                const uint32_t sE = sE0 + slot * Cfg::kEBytes;
                if (lane == 0 && blockIdx.x == 0 && it == p.skip_stage) {
                    // test hook: this stage's loads stay unissued, so the waits on it run out
                } else if (lane == 0) {
                    // one box each for the stage's A values (64 per row) and m-index words
                    mbar_arrive_expect_tx(aeb, Cfg::kABytes + Cfg::kEBytes);
                    tma_load_2d(sA, &tm_a, kt * kValsPerKTile, static_cast<int32_t>(g.m0), aeb);
                    tma_load_2d(sE, &tm_e, kt * 4, static_cast<int32_t>(g.m0), aeb);
                    if (!GATHER) {
                        const uint32_t bb = smem_u32(&b_bar[slot]);
                        mbar_arrive_expect_tx(bb, Cfg::kBBytes);
                        if (tc_narrow_b(BN, GATHER)) {
                            tma_load_2d(sB, &tm_b, static_cast<int32_t>(g.n0), kt * kKTile, bb);
                        } else {
#pragma unroll
                            for (int a = 0; a < Cfg::kAtoms; ++a)
                                tma_load_2d(sB + a * kKTile * 128, &tm_b, static_cast<int32_t>(g.n0 + 64 * a),
                                            kt * kKTile, bb);
                        }
                    }
                    last_it[slot] = it;
                }
            }
        }
        if (lane == 0 && *abort) {
            // let every copy already issued land before the CTA exits
            for (int s = 0; s < STAGES; ++s) {
                if (last_it[s] < 0) continue;
                const uint32_t par = static_cast<uint32_t>(last_it[s] / STAGES) & 1u;
                mbar_drain(smem_u32(&ae_bar[s]), par);
                if (!GATHER) mbar_drain(smem_u32(&b_bar[s]), par);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc_f16_f32(TM, BN, /*sparse=*/true, /*a_mn=*/false, /*b_mn=*/true);
            int it = 0, ti = 0;
            bool run = true;
            for (int t = static_cast<int>(blockIdx.x); run && t < p.total_tiles; t += static_cast<int>(gridDim.x), ++ti) {
                const TileGeom g = tile_geom(p, t, TM, BN);
                const int buf = ti % ACC;
                const uint32_t use = static_cast<uint32_t>(ti / ACC) & 1u;
                // the epilogue must have read this accumulator out (first use passes)
                if (!mbar_wait(smem_u32(&acce_bar[buf]), use ^ 1u, abort)) break;
                tc_fence_after_sync();
                const uint32_t d = tmem_acc + buf * BN;
                for (int k = 0; k < g.nkt; ++k, ++it) {
                    const int slot = it % STAGES;
                    const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
                    // the m-index warps arrive only after the stage's A values and m-indices landed
                    if (!mbar_wait(smem_u32(&meta_bar[slot]), ph, abort) ||
                        !mbar_wait(smem_u32(&b_bar[slot]), ph, abort)) {
                        run = false;
                        break;
                    }
                    if (GATHER) fence_proxy_async_smem();  // gathered B rows were written by cp.async
                    tc_fence_after_sync();
                    const uint32_t sA = sA0 + slot * Cfg::kABytes;
                    const uint32_t sB = sB0 + slot * Cfg::kBBytes;
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        // A: K-major, 128B swizzle, 128-byte rows (64 values), 8-row groups 1024 bytes
                        // apart; MMA k-step s takes bytes 32s .. 32s+31 of every row
                        const uint64_t ad = make_smem_desc(sA + s * 32, 16, 1024, kLayoutSw128);
                        // B: N-major, 128B swizzle; 64-column atoms kKTile*128 bytes apart (leading
                        // dimension), 8-row groups of K 1024 bytes apart (stride dimension)
                        // narrow: BN * 2-byte rows, 32B/64B swizzle, 8-row groups 16 * BN bytes apart
                        const uint64_t bd =
                            tc_narrow_b(BN, GATHER)
                                ? make_smem_desc(sB + s * 32 * (BN * 2), 16, 16 * BN, BN == 16 ? kLayoutSw32 : kLayoutSw64)
                                : make_smem_desc(sB + s * 32 * 128, Cfg::kAtoms > 1 ? kKTile * 128 : 1024, 1024,
                                                 kLayoutSw128);
                        const uint32_t te = tmem_e + slot * kMetaStageCols + s * kMetaSlotCols;
                        tc_mma_sp_f16(d, ad, bd, te, idesc, (k > 0 || s > 0) ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&empty_bar[slot]));
                }
                if (run) tc_commit(smem_u32(&accf_bar[buf]));
            }
            // every MMA issued must finish before TMEM is released
            tc_commit(smem_u32(&done_bar));
            mbar_drain(smem_u32(&done_bar), 0);
        }
        __syncwarp();
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------ m-indices -> TMEM (warps 2-5)
        const int q = warp & 3;  // this warp may access TMEM lanes 32q .. 32q+31
        const int trow = tile_row_of_lane<TM>(q, lane);
        const int srow = trow >= 0 ? trow : tile_row_of_lane<TM>(q, lane & 15);  // an in-tile row to read
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        int it = 0;
        bool run = true;
        // upper half of tile ti's accumulator (single buffer: use ti & 1), when the split applies
        auto drain_upper = [&](const TileGeom& g, int ti) -> bool {
            const bool ok = mbar_wait_warp(smem_u32(&accf_bar[0]), static_cast<uint32_t>(ti) & 1u, abort, kSleepMeta) &&
                            !*abort;
            if (!ok) return false;
            tc_fence_after_sync();
            drain_columns<BN>(p, g, tmem_acc + lane_addr, trow >= 0 ? g.m0 + trow : p.R, kEpiCols, BN);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acce_bar[0]));
            return true;
        };
        TileGeom prev;
        int ti = 0;
        for (int t = static_cast<int>(blockIdx.x); run && t < p.total_tiles; t += static_cast<int>(gridDim.x), ++ti) {
            const TileGeom g = tile_geom(p, t, TM, BN);
            if (kSplitEpi && ti > 0 && !drain_upper(prev, ti - 1)) {
                run = false;
                break;
            }
            prev = g;
            const bool pad = trow < 0 || g.m0 + trow >= p.R;  // lanes with no row act as padding
            for (int k = 0; k < g.nkt; ++k, ++it) {
                const int slot = it % STAGES;
                const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
                const bool ok = mbar_wait_warp(smem_u32(&ae_bar[slot]), ph, abort, kSleepMeta);
                if (!ok) {
                    run = false;
                    break;
                }
                uint4 w = *reinterpret_cast<const uint4*>(sE_generic + slot * Cfg::kEBytes + srow * 16);
                if (pad) w = make_uint4(kPadMeta, kPadMeta, kPadMeta, kPadMeta);
                // lane i (i % 16 < 8) pairs its low halves with lane i+8's low halves, lane i+8
                // its high halves with lane i's: each lane sends the four halves its partner
                // needs, packed in two words
                const bool hi = (lane & 8) != 0;
                const uint32_t send01 = hi ? ((w.x & 0xFFFFu) | (w.y << 16)) : ((w.x >> 16) | (w.y & 0xFFFF0000u));
                const uint32_t send23 = hi ? ((w.z & 0xFFFFu) | (w.w << 16)) : ((w.z >> 16) | (w.w & 0xFFFF0000u));
                const uint32_t got01 = __shfl_xor_sync(0xFFFFFFFFu, send01, 8);
                const uint32_t got23 = __shfl_xor_sync(0xFFFFFFFFu, send23, 8);
                const uint32_t own[4] = {w.x, w.y, w.z, w.w};
                const uint32_t got[4] = {got01 & 0xFFFFu, got01 >> 16, got23 & 0xFFFFu, got23 >> 16};
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    // low lane: [own low | partner low]; high lane: [partner high | own high]
                    const uint32_t word = hi ? (got[s] | (own[s] & 0xFFFF0000u)) : ((own[s] & 0xFFFFu) | (got[s] << 16));
                    tmem_st_32x32b_x1(tmem_e + slot * kMetaStageCols + s * kMetaSlotCols + lane_addr, word);
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&meta_bar[slot]));
            }
        }
        if (kSplitEpi && run && ti > 0) drain_upper(prev, ti - 1);
    } else if (warp < kTcWarpsFixed) {
        // ------------------------------------------------ epilogue (warps 6-9)
        const int q = warp & 3;
        const int trow = tile_row_of_lane<TM>(q, lane);
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        int ti = 0;
        for (int t = static_cast<int>(blockIdx.x); t < p.total_tiles; t += static_cast<int>(gridDim.x), ++ti) {
            const TileGeom g = tile_geom(p, t, TM, BN);
            const int buf = ti % ACC;
            const uint32_t use = static_cast<uint32_t>(ti / ACC) & 1u;
            const bool ok = mbar_wait_warp(smem_u32(&accf_bar[buf]), use, abort, kSleepEpilogue) && !*abort;
            if (!ok) break;
            tc_fence_after_sync();
            const int64_t row = trow >= 0 ? g.m0 + trow : p.R;
            drain_columns<BN>(p, g, tmem_acc + buf * BN + lane_addr, row, 0, kEpiCols);
            // this warp's lanes of the accumulator are in registers: release it
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acce_bar[buf]));
        }
    } else if (GATHER) {
        // ------------------------------------------------ B gather (cp.async), warps 10+
        constexpr int kChunksPerRow = BN / 8;                       // 16-byte chunks of a gathered row
        constexpr int kChunks = kKTile * kChunksPerRow;             // per stage
        static_assert(kChunks % kGatherThreads == 0, "gather split");
        const int gt = threadIdx.x - kTcWarpsFixed * 32;
        // Fixed thread -> (chunk, row) map: thread gt copies chunk c of the
        // kPasses consecutive rows q = q0 * kPasses + u (whole blocks of 4
        // rows when kPasses >= 4, so one column-loc word serves 4 rows);
        // consecutive threads cover consecutive 16-byte chunks of a row
        // (coalesced reads).
        constexpr int kPasses = kChunks / kGatherThreads;
        constexpr int kWords = kPasses >= 4 ? kPasses / 4 : 1;  // column-loc words a thread uses per stage
        const int c = gt % kChunksPerRow;
        const int q0 = gt / kChunksPerRow;
        const uint32_t dst_atom = (c >> 3) * (kKTile * 128);  // 64-column atom of chunk c
        const int cx = c & 7;                                  // chunk within the atom's 128-byte row
        // Stage iterator over this CTA's (tile, stage) sequence.
        struct StageIt {
            int t, k;
            TileGeom g;
            bool valid;
        };
        auto it_start = [&](StageIt& x) {
            x.t = static_cast<int>(blockIdx.x);
            x.k = 0;
            x.valid = x.t < p.total_tiles;
            if (x.valid) x.g = tile_geom(p, x.t, TM, BN);
        };
        auto it_next = [&](StageIt& x) {
            if (++x.k == x.g.nkt) {
                x.k = 0;
                x.t += static_cast<int>(gridDim.x);
                x.valid = x.t < p.total_tiles;
                if (x.valid) x.g = tile_geom(p, x.t, TM, BN);
            }
        };
        // Lane l holds column-loc word l (block l of the stage) of the stages
        // kPrefetch ahead: one coalesced 128-byte load per warp and stage, in
        // flight for kPrefetch stages (a register ring, unrolled).
        constexpr int kPrefetch = 4;
        auto load_word = [&](const StageIt& x) -> uint32_t {
            uint32_t w = 0u;
            if (x.valid)
                w = __ldg(p.colidx + (x.g.m0 / p.V) * p.nblk + static_cast<int64_t>(x.g.kt0 + x.k) * 32 + lane);
            return w;
        };
        StageIt cur, ahead;
        it_start(cur);
        ahead = cur;
        uint32_t ring[kPrefetch];
#pragma unroll
        for (int j = 0; j < kPrefetch; ++j) {
            ring[j] = load_word(ahead);
            if (ahead.valid) it_next(ahead);
        }
        int it = 0;
        bool stop = !cur.valid;
        while (!stop) {
#pragma unroll
            for (int j = 0; j < kPrefetch; ++j) {
                const uint32_t word = ring[j];  // this stage's words (loaded kPrefetch stages ago)
                ring[j] = load_word(ahead);
                if (ahead.valid) it_next(ahead);

                const int slot = it % STAGES;
                const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
                const bool ok = mbar_wait_warp(smem_u32(&empty_bar[slot]), ph ^ 1u, abort, kSleepGather);
                if (!ok) {
                    stop = true;
                    break;
                }
                const TileGeom& g = cur.g;
                const int64_t col = g.n0 + 8 * c;
                const int64_t left = p.N - col;
                const uint32_t bytes = left >= 8 ? 16u : (left > 0 ? static_cast<uint32_t>(2 * left) : 0u);
                const uint16_t* bcol = p.B + (bytes ? col : 0);
                const uint32_t sB = sB0 + slot * Cfg::kBBytes + dst_atom;
                const int64_t kbase = static_cast<int64_t>(g.kt0 + cur.k) * 32 * p.M;
                constexpr int kRowsPerWord = kPasses >= 4 ? 4 : kPasses;
#pragma unroll 2
                for (int wi = 0; wi < kWords; ++wi) {
                    // the column-loc word of the block holding rows q0*kPasses + 4*wi ..
                    const uint32_t sel = __shfl_sync(0xFFFFFFFFu, word, ((q0 * kPasses) >> 2) + wi);
#pragma unroll
                    for (int r = 0; r < kRowsPerWord; ++r) {
                        const int qq = q0 * kPasses + wi * 4 + r;  // row of the gathered tile: block qq/4, slot qq%4
                        // column-loc byte, clamped so that a corrupt array cannot address past K
                        const uint32_t cb = min((sel >> (8 * (qq & 3))) & 0xFFu, static_cast<uint32_t>(p.M - 1));
                        const int64_t kr = kbase + (qq >> 2) * p.M + static_cast<int64_t>(cb);
                        // 128B swizzle: chunk cx of row qq sits at chunk cx ^ (qq % 8)
                        cp_async_16(sB + qq * 128 + ((cx ^ (qq & 7)) << 4), bcol + kr * p.ld_b, bytes);
                    }
                }
                cp_async_arrive_noinc(smem_u32(&b_bar[slot]));
                ++it;
                it_next(cur);
                if (!cur.valid) {
                    stop = true;
                    break;
                }
            }
        }
        cp_async_wait_all();  // nothing may still be landing when the CTA exits
    }

    // ---------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) record_error(p.status, VNM_ERR_TIMEOUT, 10);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_acc, Cfg::kTmemCols);
    }
}

// Co-resident CTAs per SM of one kernel instance on one device (0: not yet
// known). The kernel's shared-memory attribute is set on the first launch
// of the instance on each device.
constexpr int kMaxDevices = 64;

template <int TM, int BN, bool GATHER>
cudaError_t launch_variant(const TcLaunch& L, const TcArgs& p, cudaStream_t stream) {
    using Cfg = TcCfg<TM, BN, tc_narrow_b(BN, GATHER)>;
    auto kern = spmm_tc_kernel<TM, BN, GATHER>;
    constexpr int threads = tc_threads<TM, BN, GATHER>();
    static std::atomic<int> per_sm_cache[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int per_sm = per_sm_cache[dev].load(std::memory_order_relaxed);
    if (per_sm == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
        if (e != cudaSuccess) return e;
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, Cfg::kSmemBytes);
        if (e != cudaSuccess) return e;
        // co-resident CTAs must find their TMEM columns free
        per_sm = std::max(1, std::min(occ, 512 / Cfg::kTmemCols));
        per_sm_cache[dev].store(per_sm, std::memory_order_relaxed);
    }
    const int64_t units = std::min<int64_t>(p.total_tiles, static_cast<int64_t>(L.sm_count) * per_sm);
    kern<<<static_cast<unsigned>(units), threads, Cfg::kSmemBytes, stream>>>(L.tm_a, L.tm_e, L.tm_b, p);
    return cudaGetLastError();
}

template <int TM, bool GATHER>
cudaError_t dispatch_bn(const TcLaunch& L, const TcArgs& p, cudaStream_t stream) {
    switch (L.tile_n) {
        case 16: return launch_variant<TM, 16, GATHER>(L, p, stream);
        case 32: return launch_variant<TM, 32, GATHER>(L, p, stream);
        case 64: return launch_variant<TM, 64, GATHER>(L, p, stream);
        case 128: return launch_variant<TM, 128, GATHER>(L, p, stream);
        case 192: return launch_variant<TM, 192, GATHER>(L, p, stream);
        case 256: return launch_variant<TM, 256, GATHER>(L, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int tc_default_stages(int tile_m, int tile_n, bool gather) {
    if (tile_m != 64 && tile_m != 128) return 0;
    if (tile_n != 16 && tile_n != 32 && tile_n != 64 && tile_n != 128 && tile_n != 192 && tile_n != 256) return 0;
    return tc_stages_for(tile_m, tile_n, tc_narrow_b(tile_n, gather));
}

cudaError_t launch_spmm_tc(const vnm_matrix_s& A, const TcLaunch& L, const void* B, int64_t ld_b, int64_t N, void* C,
                           int64_t ld_c, bool c_f32, float* partial, cudaStream_t stream) {
    if (tc_default_stages(L.tile_m, L.tile_n, L.gather) == 0 ||
        L.stages != tc_default_stages(L.tile_m, L.tile_n, L.gather))
        return cudaErrorInvalidValue;
    TcArgs p;
    p.colidx = static_cast<const uint32_t*>(A.colidx);
    p.B = static_cast<const uint16_t*>(B);
    p.ld_b = ld_b;
    p.C = C;
    p.ld_c = ld_c;
    p.R = A.R;
    p.N = N;
    p.V = A.V;
    p.M = A.M;
    p.nblk = A.K / A.M;
    p.num_kt = static_cast<int>(p.nblk / 32);
    const int splits_req = max(1, min(L.splits, p.num_kt));
    p.kt_per_split = (p.num_kt + splits_req - 1) / splits_req;
    const int splits = (p.num_kt + p.kt_per_split - 1) / p.kt_per_split;
    p.partial = splits > 1 ? partial : nullptr;
    p.c_f32 = c_f32 ? 1 : 0;
    const int64_t esz = c_f32 ? 4 : 2;
    p.vec_store = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && ((ld_c * esz) % 16 == 0);
    p.status = A.status;
    p.skip_stage = L.skip_stage;
    if (splits > 1 && partial == nullptr) return cudaErrorInvalidValue;
    p.n_tiles = static_cast<int>((N + L.tile_n - 1) / L.tile_n);
    p.m_tiles = static_cast<int>((A.R + L.tile_m - 1) / L.tile_m);
    const int64_t total = static_cast<int64_t>(p.n_tiles) * p.m_tiles * splits;
    if (total > INT32_MAX) return cudaErrorInvalidValue;
    p.total_tiles = static_cast<int>(total);
    cudaError_t e;
    if (L.tile_m == 128)
        e = L.gather ? dispatch_bn<128, true>(L, p, stream) : dispatch_bn<128, false>(L, p, stream);
    else
        e = L.gather ? dispatch_bn<64, true>(L, p, stream) : dispatch_bn<64, false>(L, p, stream);
    if (e != cudaSuccess) return e;
    if (splits > 1) return launch_splitk_reduce(partial, splits, A.R, N, C, ld_c, c_f32, stream);
    return cudaSuccess;
}

}  // namespace vnm
