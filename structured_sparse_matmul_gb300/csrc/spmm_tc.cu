// V:N:M SpMM on Blackwell's 2:4 sparse tensor cores (tcgen05.mma.sp).
//
// VENOM: A Vectorized N:M Format for Unleashing the Power of Sparse Tensor
// Cores, section 4 (Figure 4): the V:N:M matrix is run on 2:4 sparse tensor
// cores as an R x (K/M*4) operand, each block's column-loc selecting 4 of
// its M rows of B; section 4.1 (Figures 5-8): a thread-block tile spans V
// rows (BSr = V), column-loc is fetched ahead of the B rows it selects, and
// the output tile is written back with wide, coalesced stores.
//
// GB300 design (one CTA = one tile_m x tile_n tile of C, over a range of the
// condensed K; tile_m = 128, or 64 when V = 64 and column-loc differs per
// 64-row block). Per 128-column stage of the condensed K (4 MMA k-steps):
//   warp 0    TMA producer. Per stage: four tiled loads of the A values
//             (one per MMA k-step: tile_m rows x 16 values, 32B swizzle, each
//             in its own aligned buffer), one of the m-indices (tile_m rows x
//             16 bytes) and, when M == 4 (column-loc is the identity), the B
//             rows as plain tiled loads.
//   warps 6-9 (M > 4) the B gather: the column-loc words of the CTA's
//             k-range (at most kCidxStages stages; the planner splits K to
//             keep it so) are staged in shared memory before the main loop;
//             per stage these warps copy the 128 selected B rows (4 per
//             block, tile_n columns each) with 16-byte cp.async, coalesced
//             along each row, straight into the 128B-swizzled operand layout
//             (zero-filled past N); each thread's copies arrive on the
//             stage's barrier by themselves when they land
//             (cp.async.mbarrier.arrive), so every pipeline stage can be in
//             flight; the MMA thread fences the generic-proxy writes into the
//             async proxy after acquiring the barrier.
//   warps 2-5 per stage: read their rows' m-index words from shared memory,
//             pair them the way the sparse MMA reads them (rows i and i+8 of
//             each 16-row group share their 16-bit halves between TMEM lanes
//             i and i+8) and write them to TMEM (tcgen05.st), each MMA's word
//             in its own 8-column-aligned slot; after the main loop they are
//             the epilogue: TMEM -> registers (tcgen05.ld) -> fp16 (RNE) or
//             fp32 -> global, each thread writing whole 32-byte sectors of its
//             row (fp32 partials to the workspace under split-K).
//   warp 1    TMEM owner and MMA issuer (one thread): 4 sparse MMAs of
//             M=tile_m, N=tile_n, K=32 per stage into an fp32 accumulator in
//             TMEM; tcgen05.commit releases the stage. With M=128 row r of
//             the tile lives in TMEM lane r; with M=64 in lane
//             32*(r/16) + r%16 (lanes 16..31 of each quarter stay unused).
// Every mbarrier wait is bounded: on time-out the CTA records
// VNM_ERR_TIMEOUT, drains what it already issued, frees TMEM and returns.
#include <cuda_fp16.h>

#include "vnm_internal.h"
#include "vnm_ptx.cuh"

namespace vnm {
namespace {

constexpr int kTcThreadsTile = 192;    // warps 0-5; gathering CTAs add gather warps after them
constexpr int kKTile = 128;        // condensed K per stage = 4 MMAs of K = 32
constexpr int kValsPerKTile = 64;  // stored values per row per stage (128 bytes)
constexpr int kMetaSlotCols = 8;   // TMEM columns between consecutive MMAs' m-index words
constexpr int kMetaStageCols = 4 * kMetaSlotCols;
constexpr int kCidxStages = 64;    // most stages one gathering CTA covers (column-loc words in shared memory)
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
    int c_f32;
    int vec_store;           // C row starts 16-byte aligned
    int* status;
};

__host__ __device__ constexpr int pow2_at_least(int x) {
    int p = 32;
    while (p < x) p *= 2;
    return p;
}

template <int TM, int BN>
struct TcCfg {
    static constexpr int kAtoms = (BN + 63) / 64;            // 64-column swizzle atoms of B
    static constexpr int kAStepBytes = TM * 32;              // one MMA's A: TM rows x 16 values
    static constexpr int kABytes = 4 * kAStepBytes;
    static constexpr int kBBytes = kAtoms * kKTile * 128;    // per atom: 128 rows x 128 B
    static constexpr int kEBytes = TM * 16;                  // 4 m-index words per row
    static constexpr int kStageTx = kABytes + kBBytes + kEBytes;
    static constexpr int kStages = tc_stages_for(TM, BN);
    static constexpr int kTmemCols = pow2_at_least(BN + kStages * kMetaStageCols);
    static constexpr int kSmemBytes = kStages * kStageTx + 1024;  // + alignment slack
    static_assert(kStages >= 2, "pipeline depth");
    static_assert(BN + kStages * kMetaStageCols <= 512, "TMEM budget");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(TM == 64 || TM == 128, "MMA M");
};

// Gather threads of a gathering CTA: the gathered B tile needs many 16-byte
// copies in flight per SM (one CTA per SM), and a 64-row tile has half the
// A bytes per gathered B byte, so it takes twice the gather warps; never
// more threads than 16-byte chunks per stage (kKTile * BN / 8).
__host__ __device__ constexpr int gather_threads(int tm, int bn) {
    return (tm == 64 ? 512 : 256) < kKTile * bn / 8 ? (tm == 64 ? 512 : 256) : kKTile * bn / 8;
}

template <int TM, int BN, bool GATHER>
__host__ __device__ constexpr int tc_threads() {
    return kTcThreadsTile + (GATHER ? gather_threads(TM, BN) : 0);
}

// TMEM lane quarter q (warp % 4), lane l -> row of the tile (or -1).
template <int TM>
__device__ __forceinline__ int tile_row_of_lane(int q, int l) {
    if (TM == 128) return 32 * q + l;
    return l < 16 ? 16 * q + l : -1;
}

template <int TM, int BN, bool GATHER>
__global__ void __launch_bounds__(tc_threads<TM, BN, GATHER>(), 1)
    spmm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_e,
                   const __grid_constant__ CUtensorMap tm_b, const TcArgs p) {
    using Cfg = TcCfg<TM, BN>;
    constexpr int STAGES = Cfg::kStages;
    constexpr int kGatherThreads = gather_threads(TM, BN);
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];   // TMA bytes landed
    __shared__ __align__(8) uint64_t meta_bar[STAGES];   // m-indices written to TMEM (4 warps)
    __shared__ __align__(8) uint64_t empty_bar[STAGES];  // MMAs done with the stage
    __shared__ __align__(8) uint64_t acc_bar;            // accumulator complete
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ __align__(16) uint32_t s_cidx[GATHER ? kCidxStages * 32 : 1];

    // B stages first: a B descriptor read stays inside this CTA's allocation
    // even if its two strides were interpreted the other way round.
    const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sB0 = smem_base;
    const uint32_t sA0 = sB0 + STAGES * Cfg::kBBytes;
    const uint32_t sE0 = sA0 + STAGES * Cfg::kABytes;
    const uint8_t* sE_generic = smem_raw + (sE0 - smem_u32(smem_raw));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TM;
    const int split = blockIdx.z;
    const int kt0 = split * p.kt_per_split;
    const int nkt = min(p.num_kt, kt0 + p.kt_per_split) - kt0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), GATHER ? 1 + kGatherThreads : 1);
            mbar_init(smem_u32(&meta_bar[s]), 4);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&acc_bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_e);
        tma_prefetch_desc(&tm_b);
    }
    if (GATHER) {
        if (nkt > kCidxStages) {  // the host never launches this; refuse rather than overrun
            if (threadIdx.x == 0) record_error(p.status, VNM_ERR_INTERNAL, 20);
            return;
        }
        // column-loc words of this CTA's k-range, for the gather warps
        const uint32_t* crow = p.colidx + (m0 / p.V) * p.nblk + static_cast<int64_t>(kt0) * 32;
        for (int u = threadIdx.x; u < nkt * 32; u += blockDim.x) s_cidx[u] = __ldg(crow + u);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_acc = tmem_slot;        // columns [0, BN): fp32 accumulator
    const uint32_t tmem_e = tmem_slot + BN;     // columns [BN, BN + STAGES*32): m-index words
    volatile int* abort = &abort_flag;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        int last_it[STAGES];
#pragma unroll
        for (int s = 0; s < STAGES; ++s) last_it[s] = -1;
        for (int it = 0; it < nkt; ++it) {
            const int slot = it % STAGES;
            const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(smem_u32(&empty_bar[slot]), ph ^ 1u, abort);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            const int kt = kt0 + it;
            const uint32_t fb = smem_u32(&full_bar[slot]);
            const uint32_t sA = sA0 + slot * Cfg::kABytes;
            const uint32_t sB = sB0 + slot * Cfg::kBBytes;
            const uint32_t sE = sE0 + slot * Cfg::kEBytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, GATHER ? Cfg::kABytes + Cfg::kEBytes : Cfg::kStageTx);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tma_load_2d(sA + s * Cfg::kAStepBytes, &tm_a, kt * kValsPerKTile + 16 * s,
                                static_cast<int32_t>(m0), fb);
                tma_load_2d(sE, &tm_e, kt * 4, static_cast<int32_t>(m0), fb);
                if (!GATHER) {
#pragma unroll
                    for (int a = 0; a < Cfg::kAtoms; ++a)
                        tma_load_2d(sB + a * kKTile * 128, &tm_b, static_cast<int32_t>(n0 + 64 * a), kt * kKTile,
                                    fb);
                }
                last_it[slot] = it;
            }
        }
        if (lane == 0 && *abort) {
            // let every copy already issued land before the CTA exits
            for (int s = 0; s < STAGES; ++s)
                if (last_it[s] >= 0) mbar_drain(smem_u32(&full_bar[s]), static_cast<uint32_t>(last_it[s] / STAGES) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc_f16_f32(TM, BN, /*sparse=*/true, /*a_mn=*/false, /*b_mn=*/true);
            for (int it = 0; it < nkt; ++it) {
                const int slot = it % STAGES;
                const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
                // the m-index warps arrive only after this stage's TMA bytes landed
                if (!mbar_wait(smem_u32(&meta_bar[slot]), ph, abort)) break;
                if (GATHER) fence_proxy_async_smem();  // gathered B rows were written by cp.async
                tc_fence_after_sync();
                const uint32_t sA = sA0 + slot * Cfg::kABytes;
                const uint32_t sB = sB0 + slot * Cfg::kBBytes;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    // A: K-major, 32B swizzle, 32-byte rows, 8-row groups 256 bytes apart
                    const uint64_t ad = make_smem_desc(sA + s * Cfg::kAStepBytes, 16, 256, kLayoutSw32);
                    // B: N-major, 128B swizzle; 64-column atoms kKTile*128 bytes apart (leading
                    // dimension), 8-row groups of K 1024 bytes apart (stride dimension)
                    const uint64_t bd =
                        make_smem_desc(sB + s * 32 * 128, Cfg::kAtoms > 1 ? kKTile * 128 : 1024, 1024, kLayoutSw128);
                    const uint32_t te = tmem_e + slot * kMetaStageCols + s * kMetaSlotCols;
                    tc_mma_sp_f16(tmem_acc, ad, bd, te, idesc, (it > 0 || s > 0) ? 1u : 0u);
                }
                tc_commit(smem_u32(&empty_bar[slot]));
            }
            tc_commit(smem_u32(&acc_bar));
            // all issued MMAs must finish before TMEM is released
            mbar_drain(smem_u32(&acc_bar), 0);
        }
        __syncwarp();
    } else if (GATHER && warp >= 6) {
        // ------------------------------------------------ B gather (cp.async)
        constexpr int kChunksPerRow = BN / 8;                       // 16-byte chunks of a gathered row
        constexpr int kChunks = kKTile * kChunksPerRow;             // per stage
        static_assert(kChunks % kGatherThreads == 0, "gather split");
        const int gt = threadIdx.x - 6 * 32;
        // Fixed thread -> (chunk, row) map: thread gt copies chunk c of rows
        // q = u * kRowsPerPass + q0, u = 0 .. kPasses-1; consecutive threads
        // cover consecutive 16-byte chunks of one row (coalesced reads).
        constexpr int kRowsPerPass = kGatherThreads / kChunksPerRow;
        constexpr int kPasses = kChunks / kGatherThreads;
        const int c = gt % kChunksPerRow;
        const int q0 = gt / kChunksPerRow;
        const int64_t col = n0 + 8 * c;
        const int64_t left = p.N - col;
        const uint32_t bytes = left >= 8 ? 16u : (left > 0 ? static_cast<uint32_t>(2 * left) : 0u);
        const uint16_t* bcol = p.B + (bytes ? col : 0);
        const uint32_t dst_atom = (c >> 3) * (kKTile * 128);  // 64-column atom of chunk c
        const int cx = c & 7;                                  // chunk within the atom's 128-byte row
        for (int it = 0; it < nkt; ++it) {
            const int slot = it % STAGES;
            const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(smem_u32(&empty_bar[slot]), ph ^ 1u, abort);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            const int kt = kt0 + it;
            const uint32_t sB = sB0 + slot * Cfg::kBBytes + dst_atom;
            const uint32_t* sel_row = s_cidx + it * 32;
            const int32_t kbase = kt * 32 * p.M;
#pragma unroll
            for (int u = 0; u < kPasses; ++u) {
                const int q = u * kRowsPerPass + q0;  // row of the gathered tile: block q/4, slot q%4
                const uint32_t sel = sel_row[q >> 2];
                const int32_t kr = kbase + (q >> 2) * p.M + static_cast<int32_t>((sel >> (8 * (q & 3))) & 0xFFu);
                // 128B swizzle: chunk cx of row q sits at chunk cx ^ (q % 8)
                cp_async_16(sB + q * 128 + ((cx ^ (q & 7)) << 4), bcol + static_cast<int64_t>(kr) * p.ld_b, bytes);
            }
            cp_async_arrive_noinc(smem_u32(&full_bar[slot]));
        }
        cp_async_wait_all();  // nothing may still be landing when the CTA exits
    } else {
        const int q = warp & 3;  // this warp may access TMEM lanes 32q .. 32q+31
        const int trow = tile_row_of_lane<TM>(q, lane);
        const int64_t row = trow >= 0 ? m0 + trow : p.R;  // lanes with no row act as padding
        const int srow = trow >= 0 ? trow : tile_row_of_lane<TM>(q, lane & 15);  // an in-tile row to read
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        // ------------------------------------------------ m-indices -> TMEM
        for (int it = 0; it < nkt; ++it) {
            const int slot = it % STAGES;
            const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(smem_u32(&full_bar[slot]), ph, abort);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            uint4 w = *reinterpret_cast<const uint4*>(sE_generic + slot * Cfg::kEBytes + srow * 16);
            if (row >= p.R) w = make_uint4(kPadMeta, kPadMeta, kPadMeta, kPadMeta);
            const uint32_t own[4] = {w.x, w.y, w.z, w.w};
            uint32_t v[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) v[u] = 0u;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint32_t mine = own[s];
                const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, mine, 8);
                v[s * kMetaSlotCols] = (lane & 8) ? ((other >> 16) | (mine & 0xFFFF0000u))
                                                  : ((mine & 0xFFFFu) | (other << 16));
            }
            tmem_st_32x32b_x32(tmem_e + slot * kMetaStageCols + lane_addr, v);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&meta_bar[slot]));
        }
        // ------------------------------------------------ epilogue
        int ok = 1;
        if (lane == 0) ok = mbar_wait(smem_u32(&acc_bar), 0, abort) && !*abort;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        tc_fence_after_sync();
        if (ok) {
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem_acc + lane_addr + c, v);
                tmem_wait_ld();
                const int64_t col = n0 + c;
                if (row >= p.R || col >= p.N) continue;
                const bool full = col + 16 <= p.N;
                if (p.partial != nullptr) {
                    float* dst = p.partial + (static_cast<int64_t>(split) * p.R + row) * p.N + col;
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
                        const __half2 t = __floats2half2_rn(__uint_as_float(v[2 * u]), __uint_as_float(v[2 * u + 1]));
                        h[u] = *reinterpret_cast<const uint32_t*>(&t);
                    }
                    if (full && p.vec_store) {
                        reinterpret_cast<uint4*>(dst)[0] = make_uint4(h[0], h[1], h[2], h[3]);
                        reinterpret_cast<uint4*>(dst)[1] = make_uint4(h[4], h[5], h[6], h[7]);
                    } else {
                        for (int u = 0; u < 16 && col + u < p.N; ++u)
                            dst[u] = __float2half_rn(__uint_as_float(v[u]));
                    }
                }
            }
        }
    }

    // ---------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) record_error(p.status, VNM_ERR_TIMEOUT, 10 + blockIdx.z);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_acc, Cfg::kTmemCols);
    }
}

template <int TM, int BN, bool GATHER>
cudaError_t launch_variant(const TcLaunch& L, const TcArgs& p, dim3 grid, cudaStream_t stream) {
    using Cfg = TcCfg<TM, BN>;
    auto kern = spmm_tc_kernel<TM, BN, GATHER>;
    static bool configured = false;  // once per process (the attribute is per function)
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<grid, tc_threads<TM, BN, GATHER>(), Cfg::kSmemBytes, stream>>>(L.tm_a, L.tm_e, L.tm_b, p);
    return cudaGetLastError();
}

template <int TM, bool GATHER>
cudaError_t dispatch_bn(const TcLaunch& L, const TcArgs& p, dim3 grid, cudaStream_t stream) {
    switch (L.tile_n) {
        case 16: return launch_variant<TM, 16, GATHER>(L, p, grid, stream);
        case 32: return launch_variant<TM, 32, GATHER>(L, p, grid, stream);
        case 64: return launch_variant<TM, 64, GATHER>(L, p, grid, stream);
        case 128: return launch_variant<TM, 128, GATHER>(L, p, grid, stream);
        case 256: return launch_variant<TM, 256, GATHER>(L, p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int tc_gather_max_stages() { return kCidxStages; }

int tc_default_stages(int tile_m, int tile_n) {
    if (tile_m != 64 && tile_m != 128) return 0;
    if (tile_n != 16 && tile_n != 32 && tile_n != 64 && tile_n != 128 && tile_n != 256) return 0;
    return tc_stages_for(tile_m, tile_n);
}

cudaError_t launch_spmm_tc(const vnm_matrix_s& A, const TcLaunch& L, const void* B, int64_t ld_b, int64_t N, void* C,
                           int64_t ld_c, bool c_f32, float* partial, cudaStream_t stream) {
    if (tc_default_stages(L.tile_m, L.tile_n) == 0 || L.stages != tc_default_stages(L.tile_m, L.tile_n))
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
    if (splits > 1 && partial == nullptr) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>((N + L.tile_n - 1) / L.tile_n),
              static_cast<unsigned>((A.R + L.tile_m - 1) / L.tile_m), static_cast<unsigned>(splits));
    cudaError_t e;
    if (L.tile_m == 128)
        e = L.gather ? dispatch_bn<128, true>(L, p, grid, stream) : dispatch_bn<128, false>(L, p, grid, stream);
    else
        e = L.gather ? dispatch_bn<64, true>(L, p, grid, stream) : dispatch_bn<64, false>(L, p, grid, stream);
    if (e != cudaSuccess) return e;
    if (splits > 1) return launch_splitk_reduce(partial, splits, A.R, N, C, ld_c, c_f32, stream);
    return cudaSuccess;
}

}  // namespace vnm
