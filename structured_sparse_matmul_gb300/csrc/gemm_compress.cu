// Fused dense GEMM + V:N:M prune-and-encode: W = X . Y^T (fp16 operands,
// fp32 accumulation, W rounded once to fp16, RNE) is pruned and encoded tile
// by tile in the GEMM's epilogue; the dense W never goes to global memory
// (unless a caller asks for it).
//
// Dynamic N:M fine-grained structured sparse attention (DFSS), sections
// 4.2-4.3: the N:M selection and the encoding of the kept values and their
// metadata run in the epilogue of the dense GEMM that produces the sparse
// operand (there the attention scores Q K^T), which leaves the dense result
// in registers and on-chip memory. The selection applied here is the V:N:M
// rule of VENOM section 3 (Figure 2), the same as vnm_compress.
//
// GB300 design: one CTA per 128 x 128 tile of W, two CTAs per SM (one's
// epilogue overlaps the other's main loop).
//   warp 0    TMA producer: per stage the X tile (128 rows x 64 D-columns)
//             and the Y tile (128 rows x 64 D-columns), 128B swizzle.
//   warp 1    TMEM owner and MMA issuer (one thread): 4 dense MMAs
//             (tcgen05.mma kind::f16, M = N = 128, K = 16, both operands
//             K-major) per stage into a 128-column fp32 accumulator.
//   warps 2-5 epilogue, one row of the tile per thread:
//             1. the row of the accumulator (tcgen05.ld) rounded to fp16
//                into a shared-memory tile of 65-word rows (a column read
//                across rows then hits 32 banks), and to W_out if asked;
//             2. thread c sums the exact magnitudes of column c over each
//                V-row block (integers in units of 2^-24); the (row block,
//                block) pairs are spread over the threads, each picking its
//                block's 4 columns;
//             3. the (row, block) items, numbered row-major over the
//                threads so that a warp's stores are coalesced: per block the
//                2 largest of the 4 selected values, and their slots.
// The epilogue's shared memory is the stage ring's: the MMAs are done with
// it once the accumulator is complete. Every mbarrier wait is bounded.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "vnm_internal.h"
#include "vnm_ptx.cuh"
#include "vnm_select.cuh"

namespace vnm {
namespace {

constexpr int kGcTile = 128;                    // rows and columns of a W tile
constexpr int kGcStageD = 64;                   // D-columns per stage (4 MMA k-steps)
constexpr int kGcStages = 2;
constexpr int kGcOperandBytes = kGcTile * 128;  // one operand tile per stage (16 KB)
constexpr int kGcStageBytes = 2 * kGcOperandBytes;
constexpr int kGcSmemBytes = kGcStages * kGcStageBytes + 1024;
constexpr int kGcEpiWarp0 = 2;
constexpr int kGcEpiThreads = 8 * 32;           // warps 2-9, two per TMEM lane quarter
constexpr int kGcThreads = 2 * 32 + kGcEpiThreads;
constexpr int kGcPitchWords = kGcTile / 2 + 1;  // shared W tile: 65 words (130 halves) per row
constexpr uint32_t kSleepEpilogue = 256;
constexpr int kMaxDevicesGc = 64;

// |h| of an fp16 bit pattern, as fp32 (exact).
__device__ __forceinline__ float abs_half_f32(uint16_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0x7FFFu)));
}

// Top 4 of n >= 5 fp32 column sums of V magnitudes each, when fp32 decides
// it: `word` gets the 4 columns ascending and the result is true if the
// 4th largest sum exceeds the 5th by more than both sums' rounding error
// (at most V * 2^-24 of the larger, for V - 1 additions of non-negative
// exact terms), so that the exact sums select the same 4 columns. Equal
// or nearly equal sums return false (the caller sums exactly).
__device__ __forceinline__ bool top4_f32_sure(const float* s, int n, int V, uint32_t& word) {
    float k0 = -1.f, k1 = -1.f, k2 = -1.f, k3 = -1.f, k4 = -1.f;  // the 5 best, k0 largest
    uint32_t i0 = 0, i1 = 0, i2 = 0, i3 = 0;
    for (int c = 0; c < n; ++c) {
        const float k = s[c];
        if (k <= k4) continue;
        if (k <= k3) {
            k4 = k;
            continue;
        }
        k4 = k3;
        if (k > k2) {
            k3 = k2;
            i3 = i2;
            if (k > k1) {
                k2 = k1;
                i2 = i1;
                if (k > k0) {
                    k1 = k0;
                    i1 = i0;
                    k0 = k;
                    i0 = static_cast<uint32_t>(c);
                } else {
                    k1 = k;
                    i1 = static_cast<uint32_t>(c);
                }
            } else {
                k2 = k;
                i2 = static_cast<uint32_t>(c);
            }
        } else {
            k3 = k;
            i3 = static_cast<uint32_t>(c);
        }
    }
    // each sum is within V * 2^-24 * (its value) of the exact one: a gap above twice
    // that of the larger keeps the order (2^-23 per term, with margin)
    if (!(k3 - k4 > static_cast<float>(V) * 0x1p-22f * k3)) return false;
    auto cx = [](uint32_t& a, uint32_t& b) {
        const uint32_t lo = min(a, b), hi = max(a, b);
        a = lo;
        b = hi;
    };
    cx(i0, i1);
    cx(i2, i3);
    cx(i0, i2);
    cx(i1, i3);
    cx(i1, i2);
    word = i0 | (i1 << 8) | (i2 << 16) | (i3 << 24);
    return true;
}

struct GcArgs {
    int64_t R, K;
    int V, M;
    int num_k;            // stages of kGcStageD over D (0: D = 0, W = 0)
    int n_tiles;          // column tiles of W
    uint16_t* values;     // [R][vpr]
    uint8_t* meta;        // [R][mpitch]
    uint32_t* colidx;     // [R/V][nblk] words of 4 column bytes
    int64_t vpr, mpitch, nblk;
    uint16_t* w_out;      // optional dense W (fp16, ld_w), else null
    int64_t ld_w;
    int* status;
};

// Shared-memory layout of the epilogue (inside the stage ring).
constexpr int kGcTileBytes = kGcTile * kGcPitchWords * 4;         // 33280
constexpr int kGcGroupBlocks = 16;                                 // V-row blocks summed per pass
constexpr int kGcScoreOff = (kGcTileBytes + 15) & ~15;             // fp32 column sums of a group
constexpr int kGcColwOff = kGcScoreOff + kGcGroupBlocks * kGcTile * 4;  // column-loc words of the tile
constexpr int kGcColwMax = kGcTile * (kGcTile / 8);                // (128 / V) x (128 / M) words, M > 4
static_assert(kGcColwOff + kGcColwMax * 4 <= kGcStages * kGcStageBytes, "epilogue fits the stage ring");

__global__ void __launch_bounds__(kGcThreads, 3)
    gemm_compress_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
                         const GcArgs p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kGcStages];
    __shared__ __align__(8) uint64_t empty_bar[kGcStages];
    __shared__ __align__(8) uint64_t acc_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int epi_go;  // the epilogue's one decision to proceed (all 4 warps or none)

    const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* const smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = static_cast<int>(blockIdx.x) / p.n_tiles;
    const int n_tile = static_cast<int>(blockIdx.x) - m_tile * p.n_tiles;
    const int64_t m0 = static_cast<int64_t>(m_tile) * kGcTile;
    const int64_t n0 = static_cast<int64_t>(n_tile) * kGcTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGcStages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&acc_bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_y);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), kGcTile);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_acc = tmem_slot;
    volatile int* abort = &abort_flag;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last = -1;
            for (int k = 0; k < p.num_k; ++k) {
                const int slot = k % kGcStages;
                if (!mbar_wait(smem_u32(&empty_bar[slot]), (static_cast<uint32_t>(k / kGcStages) & 1u) ^ 1u, abort))
                    break;
                const uint32_t fb = smem_u32(&full_bar[slot]);
                const uint32_t sx = smem_base + slot * kGcStageBytes;
                mbar_arrive_expect_tx(fb, kGcStageBytes);
                tma_load_2d(sx, &tm_x, k * kGcStageD, static_cast<int32_t>(m0), fb);
                tma_load_2d(sx + kGcOperandBytes, &tm_y, k * kGcStageD, static_cast<int32_t>(n0), fb);
                last = k;
            }
            if (*abort) {
                // every copy issued must land before the CTA exits
                for (int k = last >= kGcStages ? last - kGcStages + 1 : 0; k <= last; ++k)
                    mbar_drain(smem_u32(&full_bar[k % kGcStages]), static_cast<uint32_t>(k / kGcStages) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && p.num_k > 0) {
            constexpr uint32_t idesc = make_idesc_f16_f32(kGcTile, kGcTile, /*sparse=*/false, /*a_mn=*/false,
                                                          /*b_mn=*/false);
            // both operands K-major, 128B swizzle, 128-byte rows, 8-row groups 1024 bytes apart;
            // MMA k-step s (K = 16) takes bytes 32s .. 32s+31 of every row
            const uint64_t xdesc0 = make_smem_desc(smem_base, 16, 1024, kLayoutSw128);
            const uint64_t ydesc0 = make_smem_desc(smem_base + kGcOperandBytes, 16, 1024, kLayoutSw128);
            bool run = true;
            for (int k = 0; k < p.num_k && run; ++k) {
                const int slot = k % kGcStages;
                if (!mbar_wait(smem_u32(&full_bar[slot]), static_cast<uint32_t>(k / kGcStages) & 1u, abort)) {
                    run = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t off = static_cast<uint64_t>((slot * kGcStageBytes) >> 4);
#pragma unroll
                for (int s = 0; s < kGcStageD / 16; ++s)
                    tc_mma_f16(tmem_acc, xdesc0 + off + 2 * s, ydesc0 + off + 2 * s, idesc, (k > 0 || s > 0) ? 1u : 0u);
                tc_commit(smem_u32(&empty_bar[slot]));
            }
            // the accumulator is complete (or abandoned) once every MMA issued is done
            tc_commit(smem_u32(&acc_bar));
            mbar_drain(smem_u32(&acc_bar), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2-9)
        const int q = warp & 3;            // TMEM lane quarter of this warp
        const int eh = (warp - kGcEpiWarp0) >> 2;  // which half of the columns it reads out
        const int trow = 32 * q + lane;    // row of the tile (step 1)
        const int t = threadIdx.x - 32 * kGcEpiWarp0;  // 0..255
        const int64_t row = m0 + trow;
        if (p.num_k > 0) mbar_wait_warp(smem_u32(&acc_bar), 0u, abort, kSleepEpilogue);
        // one thread decides for the eight warps, so that all or none of them
        // reach the named barriers below (the abort flag may rise meanwhile)
        named_barrier(1, kGcEpiThreads);
        if (t == 0) epi_go = *abort ? 0 : 1;
        named_barrier(1, kGcEpiThreads);
        if (epi_go) {
            tc_fence_after_sync();
            uint32_t* tile = reinterpret_cast<uint32_t*>(smem_gen);
            const uint16_t* tile_h = reinterpret_cast<const uint16_t*>(smem_gen);
            const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(32 * q) << 16);
            bool bad = false;
            // 1. half of the row, rounded to fp16, into the shared tile (and W_out)
#pragma unroll 1
            for (int c = (kGcTile / 2) * eh; c < (kGcTile / 2) * (eh + 1); c += 16) {
                uint32_t v[16];
                if (p.num_k > 0) {
                    tmem_ld_32x32b_x16(taddr + c, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) v[u] = 0u;
                }
                uint32_t h[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const __half2 t2 = __floats2half2_rn(__uint_as_float(v[2 * u]), __uint_as_float(v[2 * u + 1]));
                    h[u] = *reinterpret_cast<const uint32_t*>(&t2);
                    tile[trow * kGcPitchWords + c / 2 + u] = h[u];
                }
                if (row < p.R) {
                    if (n0 + c + 16 <= p.K) {
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            bad |= ((h[u] & 0x7C00u) == 0x7C00u) | ((h[u] & 0x7C000000u) == 0x7C000000u);
                    } else {
                        for (int u = 0; u < 16; ++u)
                            if (n0 + c + u < p.K) bad |= half_nonfinite(static_cast<uint16_t>(h[u / 2] >> (16 * (u & 1))));
                    }
                    if (p.w_out != nullptr) {
                        uint16_t* dst = p.w_out + row * p.ld_w + n0 + c;
                        for (int u = 0; u < 16 && n0 + c + u < p.K; ++u)
                            dst[u] = static_cast<uint16_t>(h[u / 2] >> (16 * (u & 1)));
                    }
                }
            }
            if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) record_error(p.status, VNM_ERR_NONFINITE, 7);
            // every row of the tile is in shared memory (and the TMEM reads are done)
            tc_fence_before_sync();
            named_barrier(1, kGcEpiThreads);

            const int nb_tile = kGcTile / p.M;  // blocks per tile row (a power of 2, as is V)
            const int lg_nb = __ffs(nb_tile) - 1, lg_v = __ffs(p.V) - 1;
            uint32_t* colw = reinterpret_cast<uint32_t*>(smem_gen + kGcColwOff);
            float* fscore = reinterpret_cast<float*>(smem_gen + kGcScoreOff);
            // 2. column-loc of every V-row block of the tile (rows past R: none), in
            //    groups of up to kGcGroupBlocks row blocks: thread t sums column t % 128
            //    over every other row block of the group, then the (row block, block)
            //    pairs are spread over the threads, each picking that block's 4 columns
            const int64_t rows_here = p.R - m0 < kGcTile ? p.R - m0 : kGcTile;
            const int rblocks = static_cast<int>(rows_here / p.V);
            if (p.M > 4) {
                const int c = t & (kGcTile - 1), part = t >> 7;
                for (int g0 = 0; g0 < rblocks; g0 += kGcGroupBlocks) {
                    const int g1 = min(rblocks, g0 + kGcGroupBlocks);
                    for (int rb = g0 + part; rb < g1; rb += 2) {
                        const uint16_t* col = tile_h + rb * p.V * (2 * kGcPitchWords) + c;
                        float s0 = 0.f, s1 = 0.f;
                        int r = 0;
                        for (; r + 2 <= p.V; r += 2) {
                            s0 += abs_half_f32(col[r * (2 * kGcPitchWords)]);
                            s1 += abs_half_f32(col[(r + 1) * (2 * kGcPitchWords)]);
                        }
                        if (r < p.V) s0 += abs_half_f32(col[r * (2 * kGcPitchWords)]);
                        fscore[(rb - g0) * kGcTile + c] = s0 + s1;
                    }
                    named_barrier(1, kGcEpiThreads);
                    for (int pi = t; pi < (g1 - g0) * nb_tile; pi += kGcEpiThreads) {
                        const int rbl = pi >> lg_nb, j = pi & (nb_tile - 1);
                        if (n0 + static_cast<int64_t>(j) * p.M >= p.K) continue;
                        uint32_t w;
                        if (!top4_f32_sure(fscore + rbl * kGcTile + j * p.M, p.M, p.V, w)) {
                            // too close to call in fp32: exact integer sums of the block's columns
                            Top4 best;
                            for (int cc = 0; cc < p.M; ++cc) {
                                const uint16_t* col = tile_h + (g0 + rbl) * p.V * (2 * kGcPitchWords) + j * p.M + cc;
                                uint64_t e = 0;
                                for (int r = 0; r < p.V; ++r) e += mag_units(col[r * (2 * kGcPitchWords)]);
                                best.offer(e, static_cast<uint32_t>(cc));
                            }
                            w = best.word();
                        }
                        colw[(g0 + rbl) * nb_tile + j] = w;
                        p.colidx[(m0 / p.V + g0 + rbl) * p.nblk + n0 / p.M + j] = w;
                    }
                    named_barrier(1, kGcEpiThreads);
                }
            } else {
                // M = 4: every block keeps its 4 columns
                for (int pi = t; pi < rblocks * nb_tile; pi += kGcEpiThreads) {
                    const int rb = pi >> lg_nb, j = pi & (nb_tile - 1);
                    if (n0 + static_cast<int64_t>(j) * p.M < p.K)
                        p.colidx[(m0 / p.V + rb) * p.nblk + n0 / p.M + j] = 0x03020100u;
                }
            }
            // 3. per (row, block) item, 2 of the block's 4 selected values and their
            //    slots. Items are numbered row-major, so the lanes of a warp hold
            //    consecutive blocks of a row and its stores are coalesced: values
            //    as 4-byte words, the slots of two neighbouring blocks as one byte
            //    (the even lane of the pair writes it)
            const int64_t left = (p.K - n0) / p.M;  // blocks of the tile inside K
            const int nvalid = static_cast<int>(left < nb_tile ? left : nb_tile);
            const int items = static_cast<int>(rows_here) * nb_tile;  // nb_tile is a power of 2, >= 2
            const int lane_e = t & 31;
            uint16_t* const vtile = p.values + m0 * p.vpr + (n0 / p.M) * 2;   // the tile's first value
            uint8_t* const mtile = p.meta + m0 * p.mpitch + n0 / (2 * p.M);  // and m-index byte
            for (int i0 = t - lane_e; i0 < items; i0 += kGcEpiThreads) {
                const int i = i0 + lane_e;
                const int er = i >> lg_nb, j = i & (nb_tile - 1);
                const bool live = i < items && j < nvalid;
                uint32_t code = 0;
                if (live) {
                    const uint32_t w = p.M > 4 ? colw[((er >> lg_v) << lg_nb) + j] : 0x03020100u;
                    const uint16_t* trow_h = tile_h + er * (2 * kGcPitchWords) + j * p.M;
                    uint16_t a[4];
#pragma unroll
                    for (int s = 0; s < 4; ++s) a[s] = trow_h[(w >> (8 * s)) & 0xFFu];
                    uint16_t v0, v1;
                    code = keep2of4(a, v0, v1);
                    *reinterpret_cast<uint32_t*>(vtile + er * p.vpr + 2 * j) =
                        static_cast<uint32_t>(v0) | (static_cast<uint32_t>(v1) << 16);
                }
                // the odd neighbour's code (0 when it lies past K: upper nibble 0)
                const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, code, 1);
                if (live && (j & 1) == 0)
                    mtile[er * p.mpitch + j / 2] = static_cast<uint8_t>(code | (hi << 4));
            }
        }
    }

    // ---------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) record_error(p.status, VNM_ERR_TIMEOUT, 11);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_acc, kGcTile);
    }
}

}  // namespace

bool gemm_compress_shape_ok(int V, int M) {
    return V >= 1 && V <= kGcTile && (kGcTile % V) == 0 && (M == 4 || M == 8 || M == 16 || M == 32 || M == 64);
}

cudaError_t launch_gemm_compress(const vnm_matrix_s& A, const CUtensorMap& tm_x, const CUtensorMap& tm_y, int64_t D,
                                 void* w_out, int64_t ld_w, cudaStream_t stream) {
    GcArgs p;
    p.R = A.R;
    p.K = A.K;
    p.V = A.V;
    p.M = A.M;
    p.num_k = static_cast<int>((D + kGcStageD - 1) / kGcStageD);
    p.n_tiles = static_cast<int>((A.K + kGcTile - 1) / kGcTile);
    p.values = static_cast<uint16_t*>(A.values);
    p.meta = static_cast<uint8_t*>(A.meta);
    p.colidx = static_cast<uint32_t*>(A.colidx);
    p.vpr = values_per_row(A.K, A.M);
    p.mpitch = meta_pitch(A.K, A.M);
    p.nblk = A.K / A.M;
    p.w_out = static_cast<uint16_t*>(w_out);
    p.ld_w = ld_w;
    p.status = A.status;
    const int64_t m_tiles = (A.R + kGcTile - 1) / kGcTile;
    const int64_t tiles = m_tiles * p.n_tiles;
    if (tiles > INT32_MAX) return cudaErrorInvalidValue;
    static std::atomic<bool> attr_set[kMaxDevicesGc];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevicesGc) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(gemm_compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGcSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    gemm_compress_kernel<<<static_cast<unsigned>(tiles), kGcThreads, kGcSmemBytes, stream>>>(tm_x, tm_y, p);
    return cudaGetLastError();
}

}  // namespace vnm
