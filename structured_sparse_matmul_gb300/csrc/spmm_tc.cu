// V:N:M SpMM on Blackwell's 2:4 sparse tensor cores (tcgen05.mma.sp).
//
// VENOM: A Vectorized N:M Format for Unleashing the Power of Sparse Tensor
// Cores, section 4 (Figure 4): the V:N:M matrix is run on 2:4 sparse tensor
// cores as an R x (K/M*4) operand, each block's column-loc selecting 4 of
// its M rows of B; section 4.1 (Figures 5-8): a thread-block tile spans V
// rows (BSr = V), column-loc is fetched ahead of the B rows it selects, and
// the output tile is written back with wide, coalesced stores.
//
// GB300 design: persistent CTAs (one or two per SM by shared memory and
// TMEM), each taking tiles b, b + grid, ... of C (tile_m x tile_n over a
// range of the MMAs' K; tile_m = 128, or 64 when V = 64 and column-loc
// differs per 64-row block). Tiles are ordered in groups of group_m row
// tiles: within a group the row tile varies fastest, so the CTAs running at
// one time cover many row tiles of one or two column slices of B, reusing
// each slice of B from L2, and a group's A rows (sized to stay in L2) are
// reused over all the column slices. A stage is 128 columns of the MMAs' K
// (4 MMA k-steps): a B ring of stages (the 128 rows of B the stage needs,
// tile_n wide) and a shallower A ring (tile_m rows x 64 stored values,
// 128B swizzle) feed the MMAs; the m-indices go to TMEM. Three ways to form
// the operands (TcMode):
//   kTcTiled  (M == 4): A values by TMA, B in TMA tiles.
//   kTcGather (M > 4): A values by TMA; the MMAs run over the condensed K,
//             B's 4 selected rows of every block copied in by gather warps.
//   kTcLift   (M == 8): the MMAs run over the whole K, B in TMA tiles; a
//             row keeps 2 values of 8 columns, never more than 2 of a group
//             of 4, so warps re-encode each block as 2:4 over its columns
//             and write A to shared memory themselves.
// Warp roles:
//   warp 0    A producer: one tiled TMA load per A stage (idle for kTcLift).
//   warp 1    TMEM owner and MMA issuer (one thread): per stage one
//             combined wait, 4 sparse MMAs of M = tile_m, N = tile_n, K = 32
//             into an fp32 accumulator in TMEM, and one commit that frees
//             the stage's B slot, A slot and m-index slot; a commit per tile
//             hands the accumulator to the epilogue. Two accumulators
//             alternate when TMEM holds them beside the m-index slots.
//   warps 2-5 m-index warps, one lane per row: each loads its row's four
//             m-index words of a stage from global memory a few stages
//             ahead, pairs them the way the sparse MMA reads them (rows i
//             and i+8 of each 16-row group share 16-bit halves between TMEM
//             lanes i and i+8) and writes them to the stage's TMEM slot (each
//             MMA's word 8-column aligned). With kTcLift they, and two more
//             groups of four warps (11+), re-encode A instead (see there).
//   warps 6-9 epilogue: TMEM -> registers (tcgen05.ld) -> fp16 (RNE) or
//             fp32 -> global, each thread writing whole 32-byte sectors of
//             its row (fp32 partials to the workspace under split-K); with
//             M = 128 row r of the tile lives in TMEM lane r, with M = 64 in
//             lane 32*(r/16) + r%16 (lanes 16..31 of each quarter unused).
//   warp 10   B producer (kTcTiled, kTcLift): TMA tiles of 64 columns x 128
//             rows, or one tile_n-wide box for 16- and 32-column tiles.
//   warps 11+ (kTcGather) the B gather: each warp owns whole blocks of 4
//             selected rows of every stage; every lane reads the blocks'
//             column-loc words (loaded a few stages ahead) and copies
//             16-byte chunks with cp.async, coalesced along each row,
//             straight into the 128B-swizzled operand layout (zero-filled
//             past N); each thread's copies arrive on the stage's barrier
//             (cp.async.mbarrier.arrive.noinc) and the MMA thread fences the
//             generic-proxy writes into the async proxy after its wait.
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

constexpr int kTcWarpsFixed = 11;  // warps 0-10; gathering CTAs add gather warps after them
constexpr int kEpiWarp0 = 6;       // warps 6-9: epilogue
constexpr int kBProducerWarp = 10; // B by TMA (M == 4)
constexpr int kKSteps = kTcStageK / 32;        // MMA k-steps (K = 32) per stage
constexpr int kValsPerStage = kTcStageK / 2;   // stored values per row per stage (128 bytes)
constexpr int kMetaSlotCols = 8;   // TMEM columns between consecutive MMAs' m-index words
constexpr int kMetaStageCols = kKSteps * kMetaSlotCols;
// Sleep between polls of a barrier, per role (ns): the MMA thread polls
// flat out; the others park so that ~20 waiting warps do not take the issue
// slots of the ones doing work. The epilogue waits a whole tile.
constexpr uint32_t kSleepProducer = 32;
constexpr uint32_t kSleepMeta = 32;
constexpr uint32_t kSleepGather = 32;
constexpr uint32_t kSleepEpilogue = 256;
// m-index word of a row that lies beyond R: slots (0, 1) in all 8 groups
constexpr uint32_t kPadMeta = 0x44444444u;
// stages ahead of their use at which the m-index warps load the m-index
// words of their rows (fewer when they also drain half of the accumulator)
__host__ __device__ constexpr int meta_prefetch(bool split_epilogue) { return split_epilogue ? 2 : 4; }

struct TcArgs {
    const uint32_t* colidx;  // [R/V][nblk] words of 4 column bytes
    const uint32_t* values;  // [R][vpr_words] words of 2 values, read by the re-encoding warps (kTcLift)
    int64_t vpr_words;
    const uint16_t* B;       // K x N fp16 (ld_b), read by the gather warps
    const uint8_t* meta;     // [R][mpitch] m-indices, read by the m-index warps
    int64_t mpitch;
    int64_t ld_b;
    OutSpec out;             // C (strides, type, bias, activation)
    int plain_out;           // C row-major with no bias or activation (the vector stores below)
    int b_kmajor;            // B K-major (tiled and lift modes): TMA boxes of 64 K x BN rows
    float* partial;          // [splits][R][N] fp32, or null
    int64_t R, N;
    int V, M;
    int64_t nblk;
    int num_kt;              // MMA K / kTcStageK: B stages of a whole row
    int kt_per_split;        // B stages per K split
    int n_tiles, m_tiles;    // tile grid (see tile_geom for the order)
    int group_m;             // row tiles per group of the tile order
    int total_tiles;
    int vec_store;           // C row starts 16-byte aligned
    int vec32;               // C row starts 32-byte aligned (32-byte stores)
    int part_vec32;          // split-K partial rows 32-byte aligned
    int skip_stage;          // tests of the bounded waits: CTA 0 never issues this stage's loads (-1: none)
    int* status;
};

__host__ __device__ constexpr int pow2_at_least(int x) {
    int p = 32;
    while (p < x) p *= 2;
    return p;
}

// Gather warps of a gathering CTA (each owns 32 / warps blocks of a stage):
// 16 for wide tiles (one CTA per SM), 8 for tiles of at most 64 columns
// (two CTAs per SM).
__host__ __device__ constexpr int gather_warps(int bn) { return bn <= 64 ? 8 : 16; }

// Groups of 4 warps that re-encode A (kTcLift), each taking every
// kLiftGroups-th stage (at most the B stages: see the lift warps' waits).
constexpr int kLiftGroups = 3;

template <int TM, int BN, int MODE>
__host__ __device__ constexpr int tc_threads() {
    return kTcWarpsFixed * 32 +
           (MODE == kTcGather ? 32 * gather_warps(BN) : MODE == kTcLift ? 32 * 4 * (kLiftGroups - 1) : 0);
}

// B stages ahead of their use at which a gather warp loads their column-loc
// words (8 words per warp in flight)
__host__ __device__ constexpr int col_prefetch(int blocks_per_warp) { return 8 / blocks_per_warp; }

template <int TM, int BN, int MODE>
struct TcCfg {
    static constexpr bool kNarrow = tc_narrow_b(BN, MODE == kTcGather);
    static constexpr int kAtoms = (BN + 63) / 64;      // 64-column swizzle atoms of B
    static constexpr int kABytes = tc_a_stage_bytes(TM);
    static constexpr int kBBytes = tc_b_stage_bytes(BN, kNarrow);
    static constexpr int kStages = tc_stages(TM, BN, kNarrow);
    static constexpr int kAStages = tc_a_stages(TM, kStages);
    // two accumulators (the epilogue of one tile overlaps the next tile's
    // main loop) when they fit TMEM beside the m-index slots
    static constexpr int kAccBufs = 2 * BN + kStages * kMetaStageCols <= 512 ? 2 : 1;
    static constexpr int kTmemCols = pow2_at_least(kAccBufs * BN + kStages * kMetaStageCols);
    static constexpr int kSmemBytes = kStages * kBBytes + kAStages * kABytes + 1024;  // + alignment
    static constexpr int kMinBlocks = BN <= 64 && MODE != kTcLift ? 2 : 1;
    static_assert(kStages >= 2, "pipeline depth");
    static_assert(kAStages >= 2 && kAStages <= kStages, "A ring depth");
    static_assert(BN + kStages * kMetaStageCols <= 512, "TMEM budget");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(TM == 64 || TM == 128, "MMA M");
    // a lift group waits on b_empty of stage it - AS having last waited on stage
    // it - kLiftGroups - AS: the barrier cannot be two phases behind
    static_assert(MODE != kTcLift || kLiftGroups <= kStages, "lift groups");
    static_assert(kBBytes % 1024 == 0 || kNarrow, "B stages keep the 1024-byte swizzle alignment");
};

// TMEM lane quarter q (warp % 4), lane l -> row of the tile (or -1).
template <int TM>
__device__ __forceinline__ int tile_row_of_lane(int q, int l) {
    if (TM == 128) return 32 * q + l;
    return l < 16 ? 16 * q + l : -1;
}

// Write a row's four m-index words of a stage (one per MMA k-step) to the
// stage's TMEM slot `te` in this warp's lane quarter (`lane_addr`), paired
// the way the sparse MMA reads them: rows i and i+8 of each 16-row group
// share 16-bit halves, TMEM lane i taking both rows' low halves and lane i+8
// both rows' high halves. Each lane sends its partner the four halves the
// partner needs, packed in two words. Whole warp.
__device__ __forceinline__ void store_meta_words(uint32_t te, uint32_t lane_addr, int lane, const uint32_t (&own)[4]) {
    const bool hi = (lane & 8) != 0;
    const uint32_t send01 = hi ? ((own[0] & 0xFFFFu) | (own[1] << 16)) : ((own[0] >> 16) | (own[1] & 0xFFFF0000u));
    const uint32_t send23 = hi ? ((own[2] & 0xFFFFu) | (own[3] << 16)) : ((own[2] >> 16) | (own[3] & 0xFFFF0000u));
    const uint32_t got01 = __shfl_xor_sync(0xFFFFFFFFu, send01, 8);
    const uint32_t got23 = __shfl_xor_sync(0xFFFFFFFFu, send23, 8);
    const uint32_t got[4] = {got01 & 0xFFFFu, got01 >> 16, got23 & 0xFFFFu, got23 >> 16};
#pragma unroll
    for (int s = 0; s < kKSteps; ++s) {
        // low lane: [own low | partner low]; high lane: [partner high | own high]
        const uint32_t word = hi ? (got[s] | (own[s] & 0xFFFF0000u)) : ((own[s] & 0xFFFFu) | (got[s] << 16));
        tmem_st_32x32b_x1(te + s * kMetaSlotCols + lane_addr, word);
    }
}

// 2:4 form of one block of 8 columns (kTcLift) that keeps columns d0 < d1,
// for the block's values word u (value of column d0 in the low half, of d1
// in the high half): .x holds two byte-permute selectors, applied to
// (u, 0), that give the 2-value words of the block's two groups of 4
// columns (low 16 bits: columns 0-3; high: columns 4-7); .y the two groups'
// 4-bit slot codes (lower slot in the low 2 bits; columns 0-3 in the low
// nibble). A group that holds one kept column pairs it with a zero in slot
// 0, or in slot 1 when the kept column is column 0 of the group; a group
// that holds none takes zeros in slots 0 and 1. A pair with d0 >= d1 (which
// vnm_compress never writes) gives zeros.
__host__ __device__ constexpr uint2 lift_entry(uint32_t d0, uint32_t d1) {
    constexpr uint32_t kBoth = 0x3210u;     // (u.lo, u.hi)
    constexpr uint32_t kNone = 0x4444u;     // (0, 0)
    constexpr uint32_t kLoZero = 0x4410u;   // (u.lo, 0)
    constexpr uint32_t kZeroLo = 0x1044u;   // (0, u.lo)
    constexpr uint32_t kHiZero = 0x4432u;   // (u.hi, 0)
    constexpr uint32_t kZeroHi = 0x3244u;   // (0, u.hi)
    constexpr uint32_t kPad = 0x4u;         // slots 0 and 1
    if (d0 >= d1 || d1 > 7) return uint2{kNone | (kNone << 16), kPad | (kPad << 4)};
    if (d1 < 4) return uint2{kBoth | (kNone << 16), (d0 | (d1 << 2)) | (kPad << 4)};
    if (d0 >= 4) return uint2{kNone | (kBoth << 16), kPad | (((d0 - 4) | ((d1 - 4) << 2)) << 4)};
    const uint32_t e = d1 - 4;
    const uint32_t sel0 = d0 == 0 ? kLoZero : kZeroLo, code0 = d0 == 0 ? kPad : (d0 << 2);
    const uint32_t sel1 = e == 0 ? kHiZero : kZeroHi, code1 = e == 0 ? kPad : (e << 2);
    return uint2{sel0 | (sel1 << 16), code0 | (code1 << 4)};
}

struct TileGeom {
    int64_t m0, n0;  // first row and column of the C tile
    int split;       // K split
    int kt0, nkt;    // first stage (of kTcStageK condensed columns) and stage count
};

// Tile t: split = t / (m_tiles * n_tiles); within a split, groups of group_m
// row tiles (the last group may be smaller) by n_tiles column tiles, the row
// tile varying fastest within a group.
__device__ __forceinline__ TileGeom tile_geom(const TcArgs& p, int t, int tm, int bn) {
    TileGeom g;
    const int per_split = p.m_tiles * p.n_tiles;
    g.split = t / per_split;
    int r = t - g.split * per_split;
    const int group_tiles = p.group_m * p.n_tiles;
    const int grp = r / group_tiles;
    const int first_m = grp * p.group_m;
    const int gm = min(p.group_m, p.m_tiles - first_m);
    r -= grp * group_tiles;
    const int m_idx = first_m + r % gm;
    const int n_idx = r / gm;
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
template <int BN, bool GEN>
__device__ __forceinline__ void drain_columns(const TcArgs& p, const TileGeom& g, uint32_t tacc, int64_t row, int c0,
                                              int c1) {
    // one 16-column chunk of this thread's row: fp32 partials, fp32 or fp16 C
    auto store16 = [&](const uint32_t (&v)[16], int c) {
        const int64_t col = g.n0 + c;
        if (row >= p.R || col >= p.N) return;
        const bool full = col + 16 <= p.N;
        if (p.partial != nullptr) {
            float* dst = p.partial + (static_cast<int64_t>(g.split) * p.R + row) * p.N + col;
            if (full && p.part_vec32) {
                st_global_v8(dst, v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
                st_global_v8(dst + 8, v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]);
            } else if (full && (p.N % 4) == 0) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    reinterpret_cast<uint4*>(dst)[u] = make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            } else {
                for (int u = 0; u < 16 && col + u < p.N; ++u) dst[u] = __uint_as_float(v[u]);
            }
        } else if (GEN && !p.plain_out) {
            // a bias, an activation or a transposed C: the 16 values transformed, then stored one
            // by one (with a transposed C the lanes' rows are consecutive, so each store of the
            // warp covers 32 consecutive elements of one row of Y)
            float t[16];
            const float bb = p.out.bias != nullptr ? __half2float(p.out.bias[row]) : 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                float x = __uint_as_float(v[u]) + bb;
                if (p.out.act == VNM_ACT_RELU) x = fmaxf(x, 0.f);
                else if (p.out.act == VNM_ACT_GELU) x = 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
                t[u] = x;
            }
            const int64_t ns = p.out.ns;
            if (p.out.f32) {
                float* dst = static_cast<float*>(p.out.C) + row * p.out.rs + col * ns;
                if (full) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) dst[u * ns] = t[u];
                } else {
                    for (int u = 0; u < 16 && col + u < p.N; ++u) dst[u * ns] = t[u];
                }
            } else {
                __half* dst = static_cast<__half*>(p.out.C) + row * p.out.rs + col * ns;
                if (full) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) dst[u * ns] = __float2half_rn(t[u]);
                } else {
                    for (int u = 0; u < 16 && col + u < p.N; ++u) dst[u * ns] = __float2half_rn(t[u]);
                }
            }
        } else if (p.out.f32) {
            float* dst = static_cast<float*>(p.out.C) + row * p.out.rs + col;
            if (full && p.vec32) {
                st_global_v8(dst, v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
                st_global_v8(dst + 8, v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]);
            } else if (full && p.vec_store) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    reinterpret_cast<uint4*>(dst)[u] = make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            } else {
                for (int u = 0; u < 16 && col + u < p.N; ++u) dst[u] = __uint_as_float(v[u]);
            }
        } else {
            __half* dst = static_cast<__half*>(p.out.C) + row * p.out.rs + col;
            uint32_t h[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const __half2 t2 = __floats2half2_rn(__uint_as_float(v[2 * u]), __uint_as_float(v[2 * u + 1]));
                h[u] = *reinterpret_cast<const uint32_t*>(&t2);
            }
            if (full && p.vec32) {
                st_global_v8(dst, h[0], h[1], h[2], h[3], h[4], h[5], h[6], h[7]);
            } else if (full && p.vec_store) {
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

// Iterator over a CTA's (tile, stage) sequence; every role walks the same
// one, so their stage and accumulator counters agree.
struct StageIt {
    int t, k;
    TileGeom g;
    bool valid;
};

template <int TM, int BN>
__device__ __forceinline__ void stage_start(const TcArgs& p, StageIt& x) {
    x.t = static_cast<int>(blockIdx.x);
    x.k = 0;
    x.valid = x.t < p.total_tiles;
    if (x.valid) x.g = tile_geom(p, x.t, TM, BN);
}

template <int TM, int BN>
__device__ __forceinline__ void stage_next(const TcArgs& p, StageIt& x) {
    if (++x.k < x.g.nkt) return;
    x.k = 0;
    x.t += static_cast<int>(gridDim.x);
    x.valid = x.t < p.total_tiles;
    if (x.valid) x.g = tile_geom(p, x.t, TM, BN);
}

// Persistent: CTA b takes tiles b, b + gridDim.x, ...
// GEN: the general output (bias, activation, transposed C) and a K-major B
// (the Linear-layer form); without it the kernel is the plain SpMM's.
template <int TM, int BN, int MODE, bool GEN>
__global__ void __launch_bounds__(tc_threads<TM, BN, MODE>(), TcCfg<TM, BN, MODE>::kMinBlocks)
    spmm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const TcArgs p) {
    constexpr bool GATHER = MODE == kTcGather;
    constexpr bool LIFT = MODE == kTcLift;
    using Cfg = TcCfg<TM, BN, MODE>;
    constexpr int ST = Cfg::kStages;
    constexpr int AS = Cfg::kAStages;
    constexpr int ACC = Cfg::kAccBufs;
    constexpr int kGatherThreads = 32 * gather_warps(BN);
    // The m-index warps never drain the accumulator: their m-index loads run
    // ahead of the MMAs, and a drain between tiles made them late.
    constexpr bool kSplitEpi = false;
    constexpr int kEpiCols = kSplitEpi ? BN / 2 : BN;  // columns [0, kEpiCols) drained by the epilogue warps
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t b_full[ST];    // B landed (TMA, or every gather thread)
    __shared__ __align__(8) uint64_t meta_bar[ST];  // the stage's m-indices written to TMEM (4 warps)
    // b_empty[s % ST]: the MMAs of stage s (and all before it) are done, so
    // its B rows, its m-index slot and its A stage (s % AS) may be reused
    __shared__ __align__(8) uint64_t b_empty[ST];
    __shared__ __align__(8) uint64_t a_full[AS];    // A stage landed (TMA)
    __shared__ __align__(8) uint64_t accf_bar[ACC]; // accumulator complete (MMA commit)
    __shared__ __align__(8) uint64_t acce_bar[ACC]; // accumulator read out (4 epilogue warps)
    __shared__ __align__(8) uint64_t done_bar;      // every MMA of this CTA complete
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ uint2 lift_tab[LIFT ? 64 : 1];       // lift_entry(d0, d1) at 8 * d0 + d1

    // B stages first: a B descriptor read stays inside this CTA's allocation
    // even if its two strides were interpreted the other way round.
    const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sB0 = smem_base;
    const uint32_t sA0 = sB0 + ST * Cfg::kBBytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&b_full[s]), GATHER ? kGatherThreads : 1);
            mbar_init(smem_u32(&meta_bar[s]), 4);
            mbar_init(smem_u32(&b_empty[s]), 1);
        }
        for (int s = 0; s < AS; ++s) mbar_init(smem_u32(&a_full[s]), 1);
        for (int b = 0; b < ACC; ++b) {
            mbar_init(smem_u32(&accf_bar[b]), 1);
            mbar_init(smem_u32(&acce_bar[b]), kSplitEpi ? 8 : 4);
        }
        mbar_init(smem_u32(&done_bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        if (!LIFT) tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
    }
    if (LIFT && threadIdx.x < 64) lift_tab[threadIdx.x] = lift_entry(threadIdx.x >> 3, threadIdx.x & 7u);
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_acc = tmem_slot;           // columns [0, ACC*BN): fp32 accumulators
    const uint32_t tmem_e = tmem_slot + ACC * BN;  // then ST*32 columns of m-index words
    volatile int* abort = &abort_flag;

    if (warp == 0) {
        // ------------------------------------------------ A producer (TMA; none when A is re-encoded)
        if (LIFT) {
            // idle
        } else {
        int last_it[AS];
#pragma unroll
        for (int s = 0; s < AS; ++s) last_it[s] = -1;
        int st = 0;
        bool run = true;
        for (int t = static_cast<int>(blockIdx.x); run && t < p.total_tiles; t += static_cast<int>(gridDim.x)) {
            const TileGeom g = tile_geom(p, t, TM, BN);
            for (int k = 0; k < g.nkt; ++k, ++st) {
                const int aslot = st % AS;
                // A stage aslot was last read by stage st - AS: free once that stage's MMAs are done
                // (AS <= ST, and the MMAs cannot pass stage st - 1 before this load, so the phase
                // of b_empty waited on here is unambiguous)
                if (st >= AS && !mbar_wait_warp(smem_u32(&b_empty[(st - AS) % ST]),
                                                static_cast<uint32_t>((st - AS) / ST) & 1u, abort, kSleepProducer)) {
                    run = false;
                    break;
                }
                // test hook: CTA 0 leaves this stage's A load unissued, so the wait on it runs out
                if (lane == 0 && !(GATHER && blockIdx.x == 0 && st == p.skip_stage)) {
                    const uint32_t fb = smem_u32(&a_full[aslot]);
                    mbar_arrive_expect_tx(fb, Cfg::kABytes);
                    tma_load_2d(sA0 + aslot * Cfg::kABytes, &tm_a, (g.kt0 + k) * kValsPerStage,
                                static_cast<int32_t>(g.m0), fb);
                    last_it[aslot] = st;
                }
            }
        }
        if (lane == 0 && *abort) {
            // let every copy already issued land before the CTA exits
            for (int s = 0; s < AS; ++s)
                if (last_it[s] >= 0) mbar_drain(smem_u32(&a_full[s]), static_cast<uint32_t>(last_it[s] / AS) & 1u);
        }
        }
    } else if (warp == kBProducerWarp) {
        // ------------------------------------------------ B producer (TMA tiles: kTcTiled, kTcLift)
        if (!GATHER) {
            int last_it[ST];
#pragma unroll
            for (int s = 0; s < ST; ++s) last_it[s] = -1;
            int it = 0;
            bool run = true;
            for (int t = static_cast<int>(blockIdx.x); run && t < p.total_tiles; t += static_cast<int>(gridDim.x)) {
                const TileGeom g = tile_geom(p, t, TM, BN);
                for (int k = 0; k < g.nkt; ++k, ++it) {
                    const int slot = it % ST;
                    if (!mbar_wait_warp(smem_u32(&b_empty[slot]), (static_cast<uint32_t>(it / ST) & 1u) ^ 1u, abort,
                                        kSleepProducer)) {
                        run = false;
                        break;
                    }
                    // test hook: CTA 0 leaves this stage's B loads unissued
                    if (lane == 0 && !(blockIdx.x == 0 && it == p.skip_stage)) {
                        const uint32_t fb = smem_u32(&b_full[slot]);
                        const uint32_t sB = sB0 + slot * Cfg::kBBytes;
                        const int32_t row = (g.kt0 + k) * kTcStageK;
                        mbar_arrive_expect_tx(fb, Cfg::kBBytes);
                        if (GEN && p.b_kmajor) {
                            // two boxes of 64 K x BN rows (128-byte rows, 128B swizzle)
                            tma_load_2d(sB, &tm_b, row, static_cast<int32_t>(g.n0), fb);
                            tma_load_2d(sB + BN * 128, &tm_b, row + 64, static_cast<int32_t>(g.n0), fb);
                        } else if (Cfg::kNarrow) {
                            tma_load_2d(sB, &tm_b, static_cast<int32_t>(g.n0), row, fb);
                        } else {
#pragma unroll
                            for (int a = 0; a < Cfg::kAtoms; ++a)
                                tma_load_2d(sB + a * kTcStageK * 128, &tm_b, static_cast<int32_t>(g.n0 + 64 * a), row,
                                            fb);
                        }
                        last_it[slot] = it;
                    }
                }
            }
            if (lane == 0 && *abort) {
                for (int s = 0; s < ST; ++s)
                    if (last_it[s] >= 0) mbar_drain(smem_u32(&b_full[s]), static_cast<uint32_t>(last_it[s] / ST) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // One thread; per stage one combined wait (m-indices, B, A), the four
        // MMAs and two commits. The shared-memory descriptors are computed
        // once and advanced by adding the (16-byte unit) offsets of the stage
        // and the k-step to their start-address field.
        if (lane == 0) {
            constexpr uint32_t idesc_n = make_idesc_f16_f32(TM, BN, /*sparse=*/true, /*a_mn=*/false, /*b_mn=*/true);
            constexpr uint32_t idesc_k = make_idesc_f16_f32(TM, BN, /*sparse=*/true, /*a_mn=*/false, /*b_mn=*/false);
            const uint32_t idesc = GEN && p.b_kmajor ? idesc_k : idesc_n;
            // A: K-major, 128B swizzle, 128-byte rows (64 values), 8-row groups 1024 bytes apart;
            // MMA k-step s takes bytes 32s .. 32s+31 of every row
            const uint64_t adesc0 = make_smem_desc(sA0, 16, 1024, kLayoutSw128);
            // B: N-major, 128B swizzle; 64-column atoms 128*128 bytes apart (leading dimension),
            // 8-row groups of K 1024 bytes apart (stride dimension); narrow: BN * 2-byte rows,
            // 32B/64B swizzle, 8-row groups 16 * BN bytes apart
            const uint64_t bdesc0 =
                Cfg::kNarrow ? make_smem_desc(sB0, 16, 16 * BN, BN == 16 ? kLayoutSw32 : kLayoutSw64)
                             : make_smem_desc(sB0, Cfg::kAtoms > 1 ? kTcStageK * 128 : 1024, 1024, kLayoutSw128);
            constexpr uint32_t kBRowBytes = Cfg::kNarrow ? BN * 2 : 128;
            // K-major B: BN rows of 128 bytes (64 K) per box, two boxes per stage; MMA k-step s
            // (K = 32, 64 bytes of each row) starts 64 * (s % 2) bytes into box s / 2
            const uint64_t bkdesc0 = make_smem_desc(sB0, 16, 1024, kLayoutSw128);
            int it = 0, ti = 0;
            bool run = true;
            for (int t = static_cast<int>(blockIdx.x); run && t < p.total_tiles;
                 t += static_cast<int>(gridDim.x), ++ti) {
                const TileGeom g = tile_geom(p, t, TM, BN);
                const int buf = ti % ACC;
                const uint32_t use = static_cast<uint32_t>(ti / ACC) & 1u;
                // the epilogue must have read this accumulator out (first use passes)
                if (!mbar_wait(smem_u32(&acce_bar[buf]), use ^ 1u, abort)) break;
                tc_fence_after_sync();
                const uint32_t d = tmem_acc + buf * BN;
                bool ready = false;  // this stage's barriers already seen complete
                for (int k = 0; k < g.nkt; ++k, ++it) {
                    const int slot = it % ST;
                    const int aslot = it % AS;
                    const uint32_t ph = static_cast<uint32_t>(it / ST) & 1u;
                    // (re-encoded A is written together with the m-indices: one barrier)
                    if (!ready && !(LIFT ? mbar_wait2(smem_u32(&meta_bar[slot]), ph, smem_u32(&b_full[slot]), ph, abort)
                                         : mbar_wait3(smem_u32(&meta_bar[slot]), ph, smem_u32(&b_full[slot]), ph,
                                                      smem_u32(&a_full[aslot]), static_cast<uint32_t>(it / AS) & 1u,
                                                      abort))) {
                        run = false;
                        break;
                    }
                    // gathered B rows (cp.async) and re-encoded A (st.shared) came through the generic proxy
                    if (GATHER || LIFT) fence_proxy_async_smem();
                    tc_fence_after_sync();
                    const uint64_t ad = adesc0 + ((aslot * Cfg::kABytes) >> 4);
                    const uint64_t bd = bdesc0 + ((slot * Cfg::kBBytes) >> 4);
                    const uint32_t te = tmem_e + slot * kMetaStageCols;
#pragma unroll
                    for (int s = 0; s < kKSteps; ++s) {
                        const uint64_t bs = GEN && p.b_kmajor ? bkdesc0 + ((slot * Cfg::kBBytes + (s >> 1) * BN * 128 + (s & 1) * 64) >> 4)
                                                       : bd + ((s * 32 * kBRowBytes) >> 4);
                        tc_mma_sp_f16(d, ad + 2 * s, bs, te + s * kMetaSlotCols, idesc, (k > 0 || s > 0) ? 1u : 0u);
                        if (s == 1) {
                            // test the next stage of this tile while these MMAs run
                            const int nx = it + 1;
                            const uint32_t nph = static_cast<uint32_t>(nx / ST) & 1u;
                            ready = k + 1 < g.nkt &&
                                    (LIFT ? mbar_test2(smem_u32(&meta_bar[nx % ST]), nph, smem_u32(&b_full[nx % ST]), nph)
                                          : mbar_test3(smem_u32(&meta_bar[nx % ST]), nph, smem_u32(&b_full[nx % ST]),
                                                       nph, smem_u32(&a_full[nx % AS]),
                                                       static_cast<uint32_t>(nx / AS) & 1u));
                        }
                    }
                    tc_commit(smem_u32(&b_empty[slot]));
                }
                if (run) tc_commit(smem_u32(&accf_bar[buf]));
            }
            // every MMA issued must finish before TMEM is released
            tc_commit(smem_u32(&done_bar));
            mbar_drain(smem_u32(&done_bar), 0);
        }
        __syncwarp();
    } else if (LIFT && (warp < kEpiWarp0 || warp >= kTcWarpsFixed)) {
        // ------------------------------------------------ A re-encoded as 2:4 (kTcLift)
        // kLiftGroups groups of 4 warps (warps 2-5, then 11-14, 15-18, ...);
        // group g prepares the stages it with it % kLiftGroups == g, each
        // lane one row of the tile, so that every warp has kLiftGroups
        // stage-times for the re-encoding and for its loads to land. A stage
        // is 16 blocks of 8 columns: the lane loads the row's 32 values of
        // the stage (16 words), its 64 bits of m-indices and one column-loc
        // word of its V-block (lane l: block l % 16; the 16 rows of a
        // half-warp lie in one V-block); re-encodes every block as 2:4 over
        // the block's 8 columns (lift_entry); issues the loads of its next
        // stage; and, once the stage's A slot and TMEM slot are free, writes
        // the row's 64 values into the A slot in the layout a 128B-swizzled
        // TMA box would have, and its four m-index words to TMEM.
        const int grp = warp < kEpiWarp0 ? 0 : 1 + (warp - kTcWarpsFixed) / 4;
        const int q = warp & 3;
        const int trow = tile_row_of_lane<TM>(q, lane);
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        struct Raw {
            uint4 v[4];   // the row's 32 values of the stage
            uint2 m;      // their 2-bit slots (block b at bits 4b)
            uint32_t c;   // column-loc word of block lane % 16 of the stage
        };
        int col_t = -1;         // tile whose column-loc row base is cached
        int64_t col_base = 0;   // first column-loc word of this lane's V-block row
        auto load_raw = [&](const StageIt& x, Raw& r) {
#pragma unroll
            for (int j = 0; j < 4; ++j) r.v[j] = make_uint4(0u, 0u, 0u, 0u);
            r.m = make_uint2(0u, 0u);  // rows past R: slots (0, 0) in every block encode zeros
            r.c = 0u;
            if (!x.valid || trow < 0) return;
            const int64_t row = x.g.m0 + trow;
            if (row >= p.R) return;
            if (x.t != col_t) {
                col_t = x.t;
                col_base = (row / p.V) * p.nblk;
            }
            const int kt = x.g.kt0 + x.k;
            const uint4* vs = reinterpret_cast<const uint4*>(p.values + row * p.vpr_words) + 4 * kt;
#pragma unroll
            for (int j = 0; j < 4; ++j) r.v[j] = __ldg(vs + j);
            r.m = __ldg(reinterpret_cast<const uint2*>(p.meta + row * p.mpitch) + kt);
            r.c = __ldg(p.colidx + col_base + 16 * static_cast<int64_t>(kt) + (lane & 15));
        };
        auto advance = [&](StageIt& x, int n) {
            for (int i = 0; i < n && x.valid; ++i) stage_next<TM, BN>(p, x);
        };
        StageIt cur;
        stage_start<TM, BN>(p, cur);
        advance(cur, grp);
        StageIt ahead = cur;
        advance(ahead, kLiftGroups);
        Raw r;
        load_raw(cur, r);
        int it = grp;
        while (cur.valid) {
            uint32_t aw[32];  // the row's 64 values of the stage, 2 per word
            uint32_t mw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int b = 0; b < 16; ++b) {
                const uint32_t cw = __shfl_sync(0xFFFFFFFFu, r.c, (lane & 16) | b);
                const uint4& v4 = r.v[b >> 2];
                const uint32_t u = (b & 3) == 0 ? v4.x : (b & 3) == 1 ? v4.y : (b & 3) == 2 ? v4.z : v4.w;
                const uint32_t nib = ((b < 8 ? r.m.x : r.m.y) >> (4 * (b & 7))) & 15u;
                const uint32_t d0 = (cw >> ((nib & 3u) << 3)) & 7u;
                const uint32_t d1 = (cw >> ((nib >> 2) << 3)) & 7u;
                const uint2 e = lift_tab[8 * d0 + d1];
                aw[2 * b] = __byte_perm(u, 0u, e.x);
                aw[2 * b + 1] = __byte_perm(u, 0u, e.x >> 16);
                mw[b >> 2] |= e.y << (8 * (b & 3));
            }
            // the next stage's loads only now: a wait for this stage's words never covers them
            asm volatile("" ::: "memory");
            load_raw(ahead, r);
            advance(ahead, kLiftGroups);
            const int slot = it % ST;
            const int aslot = it % AS;
            // A slot aslot was last read by stage it - AS, TMEM slot `slot` by stage
            // it - ST <= it - AS: both free once the MMAs of stage it - AS are done
            if (it >= AS && !mbar_wait_warp(smem_u32(&b_empty[(it - AS) % ST]),
                                            static_cast<uint32_t>((it - AS) / ST) & 1u, abort, kSleepMeta))
                break;
            tc_fence_after_sync();
            if (trow >= 0) {
                // 128B swizzle: 16-byte chunk c of row trow at chunk c ^ (trow % 8)
                const uint32_t rowa = sA0 + aslot * Cfg::kABytes + static_cast<uint32_t>(trow) * 128u;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(rowa + ((static_cast<uint32_t>(c) ^ (trow & 7u)) << 4), aw[4 * c], aw[4 * c + 1],
                                 aw[4 * c + 2], aw[4 * c + 3]);
            }
            fence_proxy_async_smem();  // these generic-proxy writes are read by the MMAs
            store_meta_words(tmem_e + slot * kMetaStageCols, lane_addr, lane, mw);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&meta_bar[slot]));
            it += kLiftGroups;
            advance(cur, kLiftGroups);
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------ m-indices -> TMEM (warps 2-5)
        // Each lane owns one row of the tile: it loads that row's m-index
        // words of a stage (4 words, one per MMA k-step) from global memory
        // kMetaPrefetch stages ahead, and once the stage's TMEM slot is free
        // (the MMAs of its previous use are done) writes them to TMEM.
        const int q = warp & 3;  // this warp may access TMEM lanes 32q .. 32q+31
        const int trow = tile_row_of_lane<TM>(q, lane);
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        bool run = true;
        // upper half of tile ti's accumulator (single buffer: use ti & 1), when the split applies
        auto drain_upper = [&](const TileGeom& g, int ti) -> bool {
            const bool ok = mbar_wait_warp(smem_u32(&accf_bar[0]), static_cast<uint32_t>(ti) & 1u, abort, kSleepMeta) &&
                            !*abort;
            if (!ok) return false;
            tc_fence_after_sync();
            drain_columns<BN, GEN>(p, g, tmem_acc + lane_addr, trow >= 0 ? g.m0 + trow : p.R, kEpiCols, BN);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acce_bar[0]));
            return true;
        };
        // this lane's four m-index words of a stage (padding past R)
        auto load_meta = [&](const StageIt& x) -> uint4 {
            uint4 w = make_uint4(kPadMeta, kPadMeta, kPadMeta, kPadMeta);
            if (x.valid && trow >= 0 && x.g.m0 + trow < p.R)
                w = __ldg(reinterpret_cast<const uint4*>(p.meta + (x.g.m0 + trow) * p.mpitch) + (x.g.kt0 + x.k));
            return w;
        };
        constexpr int kMetaPrefetch = meta_prefetch(kSplitEpi);
        StageIt cur, ahead;
        stage_start<TM, BN>(p, cur);
        ahead = cur;
        uint4 ring[kMetaPrefetch];
#pragma unroll
        for (int d = 0; d < kMetaPrefetch; ++d) {
            ring[d] = load_meta(ahead);
            if (ahead.valid) stage_next<TM, BN>(p, ahead);
        }
        int it = 0, ti = 0, last_t = cur.t;
        TileGeom prev = cur.g;
        while (run && cur.valid) {
#pragma unroll
            for (int d = 0; d < kMetaPrefetch; ++d) {
                const uint4 w = ring[d];  // loaded kMetaPrefetch stages ago
                if (cur.t != last_t) {
                    // a new tile: with the split epilogue, drain the previous one's upper half first
                    if (kSplitEpi && !drain_upper(prev, ti)) {
                        run = false;
                        break;
                    }
                    ++ti;
                    last_t = cur.t;
                    prev = cur.g;
                }
                const int slot = it % ST;
                const uint32_t ph = static_cast<uint32_t>(it / ST) & 1u;
                // the stage's TMEM m-index slot is free once the MMAs of its previous use are done
                if (!mbar_wait_warp(smem_u32(&b_empty[slot]), ph ^ 1u, abort, kSleepMeta)) {
                    run = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t own[4] = {w.x, w.y, w.z, w.w};
                store_meta_words(tmem_e + slot * kMetaStageCols, lane_addr, lane, own);
                // the ring slot is reused only after its words were used: a wait for them then
                // never covers the load issued for a later stage
                asm volatile("" ::: "memory");
                ring[d] = load_meta(ahead);
                if (ahead.valid) stage_next<TM, BN>(p, ahead);
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&meta_bar[slot]));
                ++it;
                stage_next<TM, BN>(p, cur);
                if (!cur.valid) break;
            }
        }
        if (kSplitEpi && run) drain_upper(prev, ti);
    } else if (warp < kEpiWarp0 + 4) {
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
            drain_columns<BN, GEN>(p, g, tmem_acc + buf * BN + lane_addr, row, 0, kEpiCols);
            // this warp's lanes of the accumulator are in registers: release it
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acce_bar[buf]));
        }
    } else if (GATHER && warp >= kTcWarpsFixed) {
        // ------------------------------------------------ B gather (cp.async), warps 11+
        // A stage holds 32 blocks of 4 selected rows of B; gather warp gw
        // owns blocks gw*BPW .. gw*BPW+BPW-1 of every stage. A block's 4 rows
        // are 4 * CPR 16-byte chunks, copied in P passes of the warp: in pass
        // i lane l takes chunk q = 32i + l, i.e. chunk q % CPR of row q / CPR
        // (consecutive lanes read consecutive chunks of a row: coalesced).
        constexpr int GW = gather_warps(BN);
        constexpr int kBlocks = kTcStageK / 4;
        constexpr int BPW = kBlocks / GW;
        constexpr int CPR = BN / 8;
        constexpr int P = (4 * CPR + 31) / 32;
        static_assert(kBlocks % GW == 0, "gather split");
        const int gw = warp - kTcWarpsFixed;
        int rb_shift[P];       // 8 * (row of the block) of this lane's chunk in pass i
        uint32_t dst[P][BPW];  // its offset in the stage, for each of the warp's blocks
        bool pv[P];
        int cc[P];
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const int q = 32 * i + lane;
            pv[i] = q < 4 * CPR;
            const int rb = pv[i] ? q / CPR : 0;
            cc[i] = pv[i] ? q % CPR : 0;
            rb_shift[i] = 8 * rb;
#pragma unroll
            for (int j = 0; j < BPW; ++j) {
                const int qq = 4 * (gw * BPW + j) + rb;  // row of the stage
                // 128B swizzle: chunk c of row qq sits at chunk (c % 8) ^ (qq % 8) of its atom
                dst[i][j] = static_cast<uint32_t>((cc[i] >> 3) * (kTcStageK * 128) + qq * 128 +
                                                  (((cc[i] & 7) ^ (qq & 7)) << 4));
            }
        }
        const int64_t ldb_bytes = p.ld_b * 2;
        // column-loc words of this warp's blocks of a stage (every lane loads the same words)
        int col_t = -1;        // tile whose column-loc row base is cached
        int64_t col_base = 0;  // its first column-loc word
        auto load_words = [&](const StageIt& x, uint32_t (&w)[BPW]) {
#pragma unroll
            for (int j = 0; j < BPW; ++j) w[j] = 0u;
            if (!x.valid) return;
            if (x.t != col_t) {
                col_t = x.t;
                col_base = (x.g.m0 / p.V) * p.nblk;
            }
            const uint32_t* src = p.colidx + col_base + static_cast<int64_t>(x.g.kt0 + x.k) * kBlocks + gw * BPW;
#pragma unroll
            for (int j = 0; j < BPW; ++j) w[j] = __ldg(src + j);
        };
        StageIt cur, ahead;
        stage_start<TM, BN>(p, cur);
        ahead = cur;
        constexpr int kColPrefetch = col_prefetch(BPW);
        uint32_t ring[kColPrefetch][BPW];
#pragma unroll
        for (int d = 0; d < kColPrefetch; ++d) {
            load_words(ahead, ring[d]);
            if (ahead.valid) stage_next<TM, BN>(p, ahead);
        }
        const char* bsrc[P];  // this lane's column of B in pass i for the current tile
        uint32_t fill[P];     // bytes of that 16-byte chunk inside B (the rest is zero-filled)
        int src_tile = -1;
        int it = 0;
        bool stop = !cur.valid;
        while (!stop) {
#pragma unroll
            for (int d = 0; d < kColPrefetch; ++d) {
                const uint32_t (&words)[BPW] = ring[d];  // loaded kColPrefetch stages ago

                const int slot = it % ST;
                const uint32_t ph = static_cast<uint32_t>(it / ST) & 1u;
                if (!mbar_wait_warp(smem_u32(&b_empty[slot]), ph ^ 1u, abort, kSleepGather)) {
                    stop = true;
                    break;
                }
                const TileGeom& g = cur.g;
                if (cur.t != src_tile) {
                    src_tile = cur.t;
#pragma unroll
                    for (int i = 0; i < P; ++i) {
                        const int64_t col = g.n0 + 8 * cc[i];
                        const int64_t left = p.N - col;
                        fill[i] = left >= 8 ? 16u : (left > 0 ? static_cast<uint32_t>(2 * left) : 0u);
                        bsrc[i] = reinterpret_cast<const char*>(p.B + (fill[i] ? col : 0));
                    }
                }
                // test hook: CTA 0 leaves this stage's B copies unissued (the MMA's wait on it runs out)
                if (!(blockIdx.x == 0 && it == p.skip_stage)) {
                    const uint32_t sB = sB0 + slot * Cfg::kBBytes;
                    // first row of B of block 0 of this stage
                    const int64_t kbase = static_cast<int64_t>(g.kt0 + cur.k) * kBlocks * p.M;
#pragma unroll
                    for (int j = 0; j < BPW; ++j) {
                        const int64_t rowbase = kbase + static_cast<int64_t>(gw * BPW + j) * p.M;
#pragma unroll
                        for (int i = 0; i < P; ++i) {
                            if (!pv[i]) continue;
                            // column-loc byte, clamped so that a corrupt array cannot address past K
                            const uint32_t cb = min((words[j] >> rb_shift[i]) & 0xFFu, static_cast<uint32_t>(p.M - 1));
                            cp_async_16(sB + dst[i][j], bsrc[i] + (rowbase + cb) * ldb_bytes, fill[i]);
                        }
                    }
                    cp_async_arrive_noinc(smem_u32(&b_full[slot]));
                }
                // the ring slot is reused only after its words were used (see the m-index warps)
                asm volatile("" ::: "memory");
                load_words(ahead, ring[d]);
                if (ahead.valid) stage_next<TM, BN>(p, ahead);
                ++it;
                stage_next<TM, BN>(p, cur);
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

template <int TM, int BN, int MODE, bool GEN>
cudaError_t launch_variant(const TcLaunch& L, const TcArgs& p, cudaStream_t stream) {
    using Cfg = TcCfg<TM, BN, MODE>;
    auto kern = spmm_tc_kernel<TM, BN, MODE, GEN>;
    constexpr int threads = tc_threads<TM, BN, MODE>();
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
    kern<<<static_cast<unsigned>(units), threads, Cfg::kSmemBytes, stream>>>(L.tm_a, L.tm_b, p);
    return cudaGetLastError();
}

template <int TM, int MODE, bool GEN>
cudaError_t dispatch_bn(const TcLaunch& L, const TcArgs& p, cudaStream_t stream) {
    switch (L.tile_n) {
        case 16: return launch_variant<TM, 16, MODE, GEN>(L, p, stream);
        case 32: return launch_variant<TM, 32, MODE, GEN>(L, p, stream);
        case 64: return launch_variant<TM, 64, MODE, GEN>(L, p, stream);
        case 128: return launch_variant<TM, 128, MODE, GEN>(L, p, stream);
        case 192: return GEN ? cudaErrorInvalidValue : launch_variant<TM, 192, MODE, false>(L, p, stream);
        case 256: return launch_variant<TM, 256, MODE, GEN>(L, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

// The 2:4 form of an M = 8 matrix over the whole K, written out (the
// workspace form of the re-encoding): every row's block j becomes the two
// 4-column groups 2j, 2j+1 of a plain 2:4 row (values2 [R][K/2], meta2
// [R][K/8]: one byte of two 4-bit codes per block). A thread takes four
// consecutive blocks of a row: 16 bytes of values, 16 bits of m-indices and
// 16 bytes of column-loc in; 32 bytes of values and 4 m-index bytes out. The
// grid is (quads of a row, rows): the row and its V-block row come from the
// block index, with no per-element division.
constexpr int kLiftThreads = 128;

__global__ void __launch_bounds__(kLiftThreads) lift_expand_kernel(const uint32_t* __restrict__ values,
                                                                   const uint8_t* __restrict__ meta,
                                                                   const uint32_t* __restrict__ colidx, int64_t R,
                                                                   int64_t nblk, int64_t mpitch, int V,
                                                                   uint32_t* __restrict__ values2,
                                                                   uint32_t* __restrict__ meta2) {
    __shared__ uint2 tab[64];
    if (threadIdx.x < 64) tab[threadIdx.x] = lift_entry(threadIdx.x >> 3, threadIdx.x & 7u);
    __syncthreads();
    const int64_t quads = nblk / 4;  // nblk = K / 8, K % 128 == 0: whole quads
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kLiftThreads + threadIdx.x;
    if (t >= quads) return;  // no barrier follows
    const int64_t j0 = 4 * t;
    for (int64_t r = blockIdx.y; r < R; r += gridDim.y) {
        const int64_t vrow = static_cast<int64_t>(static_cast<uint32_t>(r) / static_cast<uint32_t>(V));  // R < 2^31
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(values + r * nblk + j0));
        const uint32_t m = __ldg(reinterpret_cast<const uint16_t*>(meta + r * mpitch + j0 / 2));
        const uint4 c = __ldg(reinterpret_cast<const uint4*>(colidx + vrow * nblk + j0));
        const uint32_t vs[4] = {v.x, v.y, v.z, v.w}, cs[4] = {c.x, c.y, c.z, c.w};
        uint32_t out[8], codes = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t nib = (m >> (4 * b)) & 15u;
            const uint32_t d0 = (cs[b] >> ((nib & 3u) << 3)) & 7u;
            const uint32_t d1 = (cs[b] >> ((nib >> 2) << 3)) & 7u;
            const uint2 e = tab[8 * d0 + d1];
            out[2 * b] = __byte_perm(vs[b], 0u, e.x);
            out[2 * b + 1] = __byte_perm(vs[b], 0u, e.x >> 16);
            codes |= e.y << (8 * b);
        }
        uint4* dst = reinterpret_cast<uint4*>(values2 + r * (2 * nblk) + 2 * j0);
        dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
        dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
        meta2[(r * nblk + j0) / 4] = codes;
    }
}

}  // namespace

cudaError_t launch_lift_expand(const vnm_matrix_s& A, void* values2, void* meta2, cudaStream_t stream) {
    const int64_t nblk = A.K / A.M;
    if (A.M != 8 || A.K % kTcStageK != 0) return cudaErrorInvalidValue;
    const int64_t quads = nblk / 4;
    if (A.R == 0 || quads == 0) return cudaSuccess;
    // about 16 CTAs of 128 threads per SM, each a slice of a row's quads over a stride of rows
    const int64_t gx = (quads + kLiftThreads - 1) / kLiftThreads;
    const int64_t gy = std::max<int64_t>(1, std::min<int64_t>({A.R, 65535, 16 * static_cast<int64_t>(A.sm_count) / gx}));
    if (gx > 0x7FFFFFFF) return cudaErrorInvalidValue;
    lift_expand_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), kLiftThreads, 0, stream>>>(
        static_cast<const uint32_t*>(A.values), static_cast<const uint8_t*>(A.meta),
        static_cast<const uint32_t*>(A.colidx), A.R, nblk, meta_pitch(A.K, A.M), A.V,
        static_cast<uint32_t*>(values2), static_cast<uint32_t*>(meta2));
    return cudaGetLastError();
}

int tc_default_stages(int tile_m, int tile_n, bool gather) {
    if (tile_m != 64 && tile_m != 128) return 0;
    if (tile_n != 16 && tile_n != 32 && tile_n != 64 && tile_n != 128 && tile_n != 192 && tile_n != 256) return 0;
    return tc_stages(tile_m, tile_n, tc_narrow_b(tile_n, gather));
}

cudaError_t launch_spmm_tc(const vnm_matrix_s& A, const TcLaunch& L, const void* B, int64_t ld_b, int64_t N,
                           const OutSpec& out, float* partial, cudaStream_t stream) {
    const bool gather = L.mode == kTcGather;
    const bool lift = L.mode == kTcLift;
    if (L.mode != kTcTiled && L.mode != kTcGather && L.mode != kTcLift) return cudaErrorInvalidValue;
    if (lift && (A.M != 8 || L.tile_m != 128)) return cudaErrorInvalidValue;
    if (L.b_kmajor && gather) return cudaErrorInvalidValue;  // the gather copies rows of a row-major B
    if (tc_default_stages(L.tile_m, L.tile_n, gather) == 0 || L.stages != tc_default_stages(L.tile_m, L.tile_n, gather))
        return cudaErrorInvalidValue;
    TcArgs p;
    p.colidx = static_cast<const uint32_t*>(A.colidx);
    p.values = static_cast<const uint32_t*>(A.values);
    p.vpr_words = values_per_row(A.K, A.M) / 2;
    p.B = static_cast<const uint16_t*>(B);
    p.ld_b = ld_b;
    p.out = out;
    p.plain_out = out.ns == 1 && out.bias == nullptr && out.act == VNM_ACT_NONE;
    p.b_kmajor = L.b_kmajor ? 1 : 0;
    p.R = A.R;
    p.N = N;
    p.V = A.V;
    p.M = A.M;
    p.nblk = A.K / A.M;
    p.meta = static_cast<const uint8_t*>(A.meta);
    p.mpitch = meta_pitch(A.K, A.M);
    // K splits are whole 128-column units of the MMAs' K (the host sizes the
    // workspace by the same rule), one B stage each
    static_assert(kTcStageK == 128, "one B stage per 128-column unit");
    const int units = static_cast<int>(tc_k_units(A.K, A.M, lift));
    const int splits_req = max(1, min(L.splits, units));
    const int units_per_split = (units + splits_req - 1) / splits_req;
    const int splits = (units + units_per_split - 1) / units_per_split;
    p.num_kt = units;
    p.kt_per_split = units_per_split;
    p.partial = splits > 1 ? partial : nullptr;
    const int64_t esz = out.f32 ? 4 : 2;
    p.vec_store = p.plain_out && (reinterpret_cast<uintptr_t>(out.C) % 16 == 0) && ((out.rs * esz) % 16 == 0);
    p.vec32 = p.plain_out && (reinterpret_cast<uintptr_t>(out.C) % 32 == 0) && ((out.rs * esz) % 32 == 0);
    p.part_vec32 = (reinterpret_cast<uintptr_t>(partial) % 32 == 0) && (N % 8 == 0);
    p.status = A.status;
    p.skip_stage = L.skip_stage;
    if (splits > 1 && partial == nullptr) return cudaErrorInvalidValue;
    p.n_tiles = static_cast<int>((N + L.tile_n - 1) / L.tile_n);
    p.m_tiles = static_cast<int>((A.R + L.tile_m - 1) / L.tile_m);
    // row tiles per group: as many as keep the group's A values and m-indices
    // (read once per column tile) within about a third of the 126 MB L2
    {
        const int64_t a_tile = static_cast<int64_t>(L.tile_m) * (values_per_row(A.K, A.M) * 2 + meta_pitch(A.K, A.M));
        const int64_t budget = int64_t(40) << 20;
        p.group_m = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(p.m_tiles, budget / std::max<int64_t>(a_tile, 1))));
    }
    const int64_t total = static_cast<int64_t>(p.n_tiles) * p.m_tiles * splits;
    if (total > INT32_MAX) return cudaErrorInvalidValue;
    p.total_tiles = static_cast<int>(total);
    cudaError_t e;
    // the plain SpMM runs kernels without the general output and K-major B
    if (p.plain_out && !p.b_kmajor) {
        if (lift)
            e = dispatch_bn<128, kTcLift, false>(L, p, stream);
        else if (L.tile_m == 128)
            e = gather ? dispatch_bn<128, kTcGather, false>(L, p, stream) : dispatch_bn<128, kTcTiled, false>(L, p, stream);
        else
            e = gather ? dispatch_bn<64, kTcGather, false>(L, p, stream) : dispatch_bn<64, kTcTiled, false>(L, p, stream);
    } else {
        if (lift)
            e = dispatch_bn<128, kTcLift, true>(L, p, stream);
        else if (L.tile_m == 128)
            e = gather ? dispatch_bn<128, kTcGather, true>(L, p, stream) : dispatch_bn<128, kTcTiled, true>(L, p, stream);
        else
            e = gather ? dispatch_bn<64, kTcGather, true>(L, p, stream) : dispatch_bn<64, kTcTiled, true>(L, p, stream);
    }
    if (e != cudaSuccess) return e;
    if (splits > 1) return launch_splitk_reduce(partial, splits, A.R, N, out, stream);
    return cudaSuccess;
}

}  // namespace vnm
