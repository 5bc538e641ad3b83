// Magnitude V:N:M prune-and-encode (and its inverse) on the GPU.
//
// VENOM: A Vectorized N:M Format for Unleashing the Power of Sparse Tensor
// Cores, section 3 "The V:N:M format", Figure 2 (block-wise split, vector-
// wise pruning to the 4 most significant columns of each V x M block, 2:4
// pruning of each row of 4) and Figure 3 (values, m-indices, column-loc).
// The 2:4 packing follows the lecture notes "2:4 sparsity on sparse tensor
// cores" ("The compressed format": survivors pushed left, one 2-bit slot
// tag per survivor).
//
// Significance of a column = its L1 norm over the block's V rows, summed
// exactly as integers: |fp16| is an integer multiple of 2^-24 below 2^41
// units, so a uint64 sum of up to 4096 of them is exact and independent of
// the summation order. Ties go to the lower column, then to the lower slot.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "vnm_internal.h"
#include "vnm_ptx.cuh"
#include "vnm_select.cuh"

namespace vnm {
namespace {

constexpr int kCompressThreads = 256;
constexpr int kTileElems = 16384;  // V x TK elements of W staged per CTA (32 KB)
constexpr int kTileMaxCols = 4096; // TK cap (bounds the column-sum array)

// Bytes of the staged W tile, rounded up so the column sums that follow
// are 16-byte aligned.
__host__ __device__ __forceinline__ size_t tile_bytes_aligned(int V, int tk) {
    return (sizeof(uint16_t) * static_cast<size_t>(V) * tk + 15) & ~static_cast<size_t>(15);
}

struct CompressArgs {
    const uint16_t* W;
    int64_t ld_w;
    int64_t R, K;
    int V, M;
    int tk;             // columns per tile (multiple of 2*M)
    uint16_t* values;   // [R][2K/M]
    uint8_t* meta;      // [R][mpitch]
    uint32_t* colidx;   // [R/V][K/M] words of 4 bytes
    int64_t nblk, mpitch;
    bool vec_load;      // W rows 16-byte aligned at every tile start
    int* status;
};

// One CTA compresses V rows x tk columns: stage the tile in shared memory,
// sum |w| per column, pick 4 columns per block, then 2 of 4 per row.
__global__ void __launch_bounds__(kCompressThreads) compress_tiled_kernel(const CompressArgs p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int V = p.V, M = p.M, TK = p.tk;
    const int64_t i = blockIdx.y;
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * TK;
    const int tk = static_cast<int>(p.K - k0 < TK ? p.K - k0 : TK);  // multiple of M
    const int nb = tk / M;
    uint16_t* sW = reinterpret_cast<uint16_t*>(smem);                       // [V][TK]
    uint64_t* sL1 = reinterpret_cast<uint64_t*>(smem + tile_bytes_aligned(V, TK));  // [TK]
    uint32_t* sSel = reinterpret_cast<uint32_t*>(sL1 + TK);                 // [TK / M]
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();

    // stage the tile
    const uint16_t* Wt = p.W + i * V * p.ld_w + k0;
    int nonfinite = 0;
    if (p.vec_load && (tk % 8) == 0) {
        const int vpr = tk / 8;
        for (int q = threadIdx.x; q < V * vpr; q += kCompressThreads) {
            const int r = q / vpr, c8 = q % vpr;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(Wt + r * p.ld_w) + c8);
            *reinterpret_cast<uint4*>(sW + r * TK + 8 * c8) = v;
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
                nonfinite |= half_nonfinite(w[h] & 0xFFFFu) | half_nonfinite(w[h] >> 16);
        }
    } else {
        for (int q = threadIdx.x; q < V * tk; q += kCompressThreads) {
            const int r = q / tk, c = q % tk;
            const uint16_t h = Wt[r * p.ld_w + c];
            sW[r * TK + c] = h;
            nonfinite |= half_nonfinite(h);
        }
    }
    if (nonfinite) bad = 1;
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) record_error(p.status, VNM_ERR_NONFINITE, 1);
        return;
    }

    // exact column sums
    for (int c = threadIdx.x; c < tk; c += kCompressThreads) {
        uint64_t s = 0;
        for (int r = 0; r < V; ++r) s += mag_units(sW[r * TK + c]);
        sL1[c] = s;
    }
    __syncthreads();

    // 4 columns per block
    const int64_t jt = k0 / M;
    for (int b = threadIdx.x; b < nb; b += kCompressThreads) {
        const uint32_t sel = top4_ascending(sL1 + b * M, M);
        sSel[b] = sel;
        p.colidx[i * p.nblk + jt + b] = sel;
    }
    __syncthreads();

    // 2 of 4 per row; one item = one row x 4 consecutive blocks
    const int ngroups = (nb + 3) / 4;
    const bool vec_store = (p.nblk % 4 == 0) && (jt % 4 == 0);
    for (int q = threadIdx.x; q < V * ngroups; q += kCompressThreads) {
        const int r = q / ngroups, g = q % ngroups;
        const int64_t row = i * V + r;
        uint16_t out[8];
        uint32_t code = 0;
        const int nblk_here = min(4, nb - 4 * g);
        for (int u = 0; u < nblk_here; ++u) {
            const int b = 4 * g + u;
            const uint32_t sel = sSel[b];
            uint16_t a[4];
#pragma unroll
            for (int s = 0; s < 4; ++s) a[s] = sW[r * TK + b * M + ((sel >> (8 * s)) & 0xFFu)];
            code |= keep2of4(a, out[2 * u], out[2 * u + 1]) << (4 * u);
        }
        uint16_t* vrow = p.values + row * (2 * p.nblk) + 2 * (jt + 4 * g);
        uint8_t* mrow = p.meta + row * p.mpitch + (jt + 4 * g) / 2;
        if (vec_store && nblk_here == 4) {
            uint4 v;
            v.x = out[0] | (static_cast<uint32_t>(out[1]) << 16);
            v.y = out[2] | (static_cast<uint32_t>(out[3]) << 16);
            v.z = out[4] | (static_cast<uint32_t>(out[5]) << 16);
            v.w = out[6] | (static_cast<uint32_t>(out[7]) << 16);
            *reinterpret_cast<uint4*>(vrow) = v;
            *reinterpret_cast<uint16_t*>(mrow) = static_cast<uint16_t>(code);
        } else {
            for (int u = 0; u < 2 * nblk_here; ++u) vrow[u] = out[u];
            // blocks jt+4g .. : two per byte, low nibble = even block
            for (int u = 0; u < nblk_here; u += 2) mrow[u / 2] = static_cast<uint8_t>(code >> (4 * u));
        }
    }
}

// Fallback for large blocks (V x 2M above the tile budget): one CTA per
// pair of blocks of one block-row, columns summed straight from global
// memory. Owning a block pair means owning whole m-index bytes.
__global__ void __launch_bounds__(kCompressThreads) compress_block_kernel(const CompressArgs p) {
    __shared__ uint64_t sL1[2][256];
    __shared__ uint32_t sSel[2];
    __shared__ int bad;
    const int V = p.V, M = p.M;
    const int64_t i = blockIdx.y;
    const int64_t j0 = 2 * static_cast<int64_t>(blockIdx.x);
    const int nb = p.nblk - j0 < 2 ? static_cast<int>(p.nblk - j0) : 2;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    int nonfinite = 0;
    for (int q = threadIdx.x; q < nb * M; q += kCompressThreads) {
        const int b = q / M, c = q % M;
        const uint16_t* col = p.W + i * V * p.ld_w + (j0 + b) * M + c;
        uint64_t s = 0;
        for (int r = 0; r < V; ++r) {
            const uint16_t h = col[r * p.ld_w];
            nonfinite |= half_nonfinite(h);
            s += mag_units(h);
        }
        sL1[b][c] = s;
    }
    if (nonfinite) bad = 1;
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) record_error(p.status, VNM_ERR_NONFINITE, 2);
        return;
    }
    if (threadIdx.x < nb) {
        const uint32_t sel = top4_ascending(sL1[threadIdx.x], M);
        sSel[threadIdx.x] = sel;
        p.colidx[i * p.nblk + j0 + threadIdx.x] = sel;
    }
    __syncthreads();
    for (int r = threadIdx.x; r < V; r += kCompressThreads) {
        const int64_t row = i * V + r;
        uint32_t code = 0;
        for (int b = 0; b < nb; ++b) {
            uint16_t a[4], v0, v1;
            for (int s = 0; s < 4; ++s)
                a[s] = p.W[row * p.ld_w + (j0 + b) * M + ((sSel[b] >> (8 * s)) & 0xFFu)];
            code |= keep2of4(a, v0, v1) << (4 * b);
            p.values[row * (2 * p.nblk) + 2 * (j0 + b)] = v0;
            p.values[row * (2 * p.nblk) + 2 * (j0 + b) + 1] = v1;
        }
        p.meta[row * p.mpitch + j0 / 2] = static_cast<uint8_t>(code);
    }
}

// Streaming compress: a persistent grid walks the V x tk tiles; each CTA
// double-buffers its tiles in shared memory with 16-byte cp.async, so the
// next tile loads while this one is processed.
//   M == 4: column-loc is the identity; only the 2:4 step runs.
//   M > 4:  columns are ranked by fp32 sums of |w| (rows added in order);
//           when the gap between the 4th and 5th largest is not wider than
//           the fp32 error bound of such a sum (V * 2^-24 relative), the
//           block's columns are re-summed exactly as integers (units of
//           2^-24) and ranked on those. Either way the result is the exact
//           ranking, ties to the lower column.
constexpr int kStreamCtasPerSm = 3;

__device__ __forceinline__ float half_abs_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0x7FFFu)));
}

// Rank the M columns of one block (one warp): keep the 4 largest sums,
// lower column first on ties; return them ascending, one per byte. Lanes
// own columns lane, lane + 32, ...; `score` is either the fp32 or the exact
// sums (compared as given). `sRank` is per-block scratch of M bytes.
template <typename T>
__device__ __forceinline__ void rank_columns(const T* score, int M, uint8_t* sRank, int lane) {
    for (int c = lane; c < M; c += 32) {
        const T v = score[c];
        int rank = 0;
        for (int d = 0; d < M; ++d) {
            const T w = score[d];
            rank += (w > v) || (w == v && d < c);
        }
        sRank[c] = static_cast<uint8_t>(rank < 255 ? rank : 255);
    }
    __syncwarp();
}

// The 4 columns of rank < 4, ascending, packed one per byte.
__device__ __forceinline__ uint32_t selected_columns(const uint8_t* sRank, int M, int lane) {
    uint32_t word = 0;
    for (int c0 = 0; c0 < M; c0 += 32) {
        const int c = c0 + lane;
        const bool sel = c < M && sRank[c] < 4;
        const uint32_t mask = __ballot_sync(0xFFFFFFFFu, sel);
        if (sel) {
            // position among the selected columns = selected columns before c
            int pos = __popc(mask & ((1u << lane) - 1u));
            for (int d = 0; d < c0; ++d) pos += sRank[d] < 4;
            word |= static_cast<uint32_t>(c) << (8 * pos);
        }
    }
    // OR the partial words of all lanes
    for (int off = 16; off > 0; off >>= 1) word |= __shfl_xor_sync(0xFFFFFFFFu, word, off);
    return word;
}

// Value of the column of rank r (0-based) among `score`, via sRank.
template <typename T>
__device__ __forceinline__ T value_of_rank(const T* score, const uint8_t* sRank, int M, int r, int lane) {
    T v = T(0);
    int found = 0;
    for (int c0 = 0; c0 < M; c0 += 32) {
        const int c = c0 + lane;
        const bool hit = c < M && sRank[c] == r;
        const uint32_t mask = __ballot_sync(0xFFFFFFFFu, hit);
        if (!found && mask) {
            const int src = __ffs(mask) - 1;
            v = __shfl_sync(0xFFFFFFFFu, hit ? score[c] : T(0), src);
            found = 1;
        }
    }
    return v;
}

// Warp-wide: the 4 selected columns of the block whose columns start at
// col0 of the staged tile. fp32 sums decide unless the 4th/5th gap is inside
// the fp32 error bound (relative 2.5 * V * 2^-24); then exact integer sums.
__device__ uint32_t rank_block_warp(const uint16_t* sW, int TK, int V, int M, int col0, const float* sF,
                                    uint64_t* sExact, uint8_t* sRank, int lane) {
    rank_columns(sF + col0, M, sRank, lane);
    const float v4 = value_of_rank(sF + col0, sRank, M, 3, lane);
    const float v5 = value_of_rank(sF + col0, sRank, M, 4, lane);
    if (v4 - v5 > 2.5f * static_cast<float>(V) * 5.9604645e-8f * v4) return selected_columns(sRank, M, lane);
    for (int c = lane; c < M; c += 32) {
        uint64_t e = 0;
        for (int r = 0; r < V; ++r) e += mag_units(sW[r * TK + col0 + c]);
        sExact[col0 + c] = e;
    }
    __syncwarp();
    rank_columns(sExact + col0, M, sRank, lane);
    return selected_columns(sRank, M, lane);
}

__global__ void __launch_bounds__(kCompressThreads) compress_stream_kernel(const CompressArgs p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int V = p.V, M = p.M, TK = p.tk;
    const size_t tile_bytes = tile_bytes_aligned(V, TK);
    uint16_t* sBuf[2] = {reinterpret_cast<uint16_t*>(smem), reinterpret_cast<uint16_t*>(smem + tile_bytes)};
    float* sF = reinterpret_cast<float*>(smem + 2 * tile_bytes);                    // [TK]
    uint64_t* sExact = reinterpret_cast<uint64_t*>(sF + TK + (TK & 1));            // [TK]
    uint32_t* sSel = reinterpret_cast<uint32_t*>(sExact + TK);                      // [TK / M]
    float* sPart = reinterpret_cast<float*>(sSel + TK / M + 4);                     // [kCompressThreads * 8]
    uint8_t* sRankAll = reinterpret_cast<uint8_t*>(sPart + kCompressThreads * 8);    // [8 warps][256]
    __shared__ int bad;
    const int64_t tiles_x = (p.K + TK - 1) / TK;
    const int64_t n_tiles = (p.R / V) * tiles_x;
    const int cpr = TK / 8;  // 16-byte chunks per tile row
    const bool cpr_pow2 = (cpr & (cpr - 1)) == 0;
    const int cpr_log2 = 31 - __clz(cpr);

    auto issue = [&](int64_t t, uint16_t* dst) {
        const int64_t i = t / tiles_x, k0 = (t % tiles_x) * TK;
        const int tk = static_cast<int>(p.K - k0 < TK ? p.K - k0 : TK);
        const uint16_t* Wt = p.W + i * V * p.ld_w + k0;
        for (int q = threadIdx.x; q < V * cpr; q += kCompressThreads) {
            const int r = cpr_pow2 ? (q >> cpr_log2) : q / cpr;
            const int c8 = q - r * cpr;
            const int left = tk - 8 * c8;
            const uint32_t bytes = left >= 8 ? 16u : (left > 0 ? 2u * left : 0u);
            cp_async_16(smem_u32(dst + r * TK + 8 * c8), Wt + r * p.ld_w + (bytes ? 8 * c8 : 0), bytes);
        }
        cp_async_commit();
    };

    if (threadIdx.x == 0) bad = 0;
    int64_t t = blockIdx.x;
    if (t < n_tiles) issue(t, sBuf[0]);
    for (int n = 0; t < n_tiles; ++n, t += gridDim.x) {
        const int64_t tn = t + gridDim.x;
        if (tn < n_tiles) {
            issue(tn, sBuf[(n + 1) & 1]);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint16_t* sW = sBuf[n & 1];
        const int64_t i = t / tiles_x, k0 = (t % tiles_x) * TK;
        const int tk = static_cast<int>(p.K - k0 < TK ? p.K - k0 : TK);
        const int nb = tk / M;
        const int64_t jt = k0 / M;
        int nonfinite = 0;
        if (M == 4) {
            for (int b = threadIdx.x; b < nb; b += kCompressThreads) sSel[b] = 0x03020100u;
        } else {
            // fp32 column sums: thread = (8-column chunk, row group); partials per row group
            const int cpr = TK / 8;
            if (kCompressThreads % cpr == 0) {
                const int rgs = kCompressThreads / cpr;
                const int cc = threadIdx.x % cpr, rg = threadIdx.x / cpr;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int r = rg; r < V; r += rgs) {
                    const uint4 v = *reinterpret_cast<const uint4*>(sW + r * TK + 8 * cc);
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        acc[2 * h] += half_abs_to_float(static_cast<uint16_t>(w[h] & 0xFFFFu));
                        acc[2 * h + 1] += half_abs_to_float(static_cast<uint16_t>(w[h] >> 16));
                    }
                }
#pragma unroll
                for (int h = 0; h < 8; ++h) sPart[rg * TK + 8 * cc + h] = acc[h];
                __syncthreads();
                for (int c = threadIdx.x; c < tk; c += kCompressThreads) {
                    float sum = 0.f;
                    for (int g = 0; g < rgs; ++g) sum += sPart[g * TK + c];
                    sF[c] = sum;
                    nonfinite |= !(sum <= 3.4e38f);  // Inf or NaN in the column
                }
            } else {
                for (int c = threadIdx.x; c < tk; c += kCompressThreads) {
                    float sum = 0.f;
                    for (int r = 0; r < V; ++r) sum += half_abs_to_float(sW[r * TK + c]);
                    sF[c] = sum;
                    nonfinite |= !(sum <= 3.4e38f);
                }
            }
            __syncthreads();
            const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
            for (int b = warp; b < nb; b += kCompressThreads / 32) {
                const uint32_t sel = rank_block_warp(sW, TK, V, M, b * M, sF, sExact, sRankAll + 256 * warp, lane);
                if (lane == 0) sSel[b] = sel;
            }
        }
        __syncthreads();
        for (int b = threadIdx.x; b < nb; b += kCompressThreads) p.colidx[i * p.nblk + jt + b] = sSel[b];

        // 2 of 4 per row; one item = one row x 4 consecutive blocks
        const int ngroups = (nb + 3) / 4;
        const bool vec_store = (p.nblk % 4 == 0) && (jt % 4 == 0);
        for (int q = threadIdx.x; q < V * ngroups; q += kCompressThreads) {
            const int r = q / ngroups, g = q % ngroups;
            const int64_t row = i * V + r;
            uint16_t out[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            uint32_t code = 0;
            const int nblk_here = min(4, nb - 4 * g);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (u < nblk_here) {
                    const int b = 4 * g + u;
                    const uint32_t sel = sSel[b];
                    const uint16_t* wr = sW + r * TK + b * M;
                    const uint16_t a[4] = {wr[sel & 0xFFu], wr[(sel >> 8) & 0xFFu], wr[(sel >> 16) & 0xFFu],
                                           wr[sel >> 24]};
                    if (M == 4) nonfinite |= half_nonfinite(a[0]) | half_nonfinite(a[1]) | half_nonfinite(a[2]) |
                                             half_nonfinite(a[3]);
                    code |= keep2of4(a, out[2 * u], out[2 * u + 1]) << (4 * u);
                }
            }
            uint16_t* vrow = p.values + row * (2 * p.nblk) + 2 * (jt + 4 * g);
            uint8_t* mrow = p.meta + row * p.mpitch + (jt + 4 * g) / 2;
            if (vec_store && nblk_here == 4) {
                uint4 v;
                v.x = out[0] | (static_cast<uint32_t>(out[1]) << 16);
                v.y = out[2] | (static_cast<uint32_t>(out[3]) << 16);
                v.z = out[4] | (static_cast<uint32_t>(out[5]) << 16);
                v.w = out[6] | (static_cast<uint32_t>(out[7]) << 16);
                *reinterpret_cast<uint4*>(vrow) = v;
                *reinterpret_cast<uint16_t*>(mrow) = static_cast<uint16_t>(code);
            } else {
                for (int u = 0; u < 2 * nblk_here; ++u) vrow[u] = out[u];
                for (int u = 0; u < nblk_here; u += 2) mrow[u / 2] = static_cast<uint8_t>(code >> (4 * u));
            }
        }
        if (nonfinite) bad = 1;
        __syncthreads();  // this tile's buffer is refilled two tiles from now
    }
    if (threadIdx.x == 0 && bad) record_error(p.status, VNM_ERR_NONFINITE, 3);
}

__device__ __forceinline__ float shfl_any(float v, int src) { return __shfl_sync(0xFFFFFFFFu, v, src); }
__device__ __forceinline__ uint64_t shfl_any(uint64_t v, int src) {
    const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), src);
    const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), src);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Lane c < n of a warp holds the score of column c. Column order: larger
// score first, lower index first on equal scores. Returns the bit mask of
// the 4 leading columns and puts this lane's place in that order in *rank
// (32 for lanes >= n).
template <typename T>
__device__ __forceinline__ uint32_t warp_top4_mask(T score, int n, int lane, int* rank) {
    int rk = 0;
    for (int c = 0; c < n; ++c) {
        const T o = shfl_any(score, c);
        rk += (o > score) || (o == score && c < lane);
    }
    *rank = lane < n ? rk : 32;
    return __ballot_sync(0xFFFFFFFFu, lane < n && rk < 4);
}

// The 4 lowest set bits of `mask` as ascending bytes of a word.
__device__ __forceinline__ uint32_t mask_to_cols(uint32_t mask) {
    uint32_t sel = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int c = __ffs(mask) - 1;
        sel |= static_cast<uint32_t>(c & 0xFF) << (8 * q);
        mask &= mask - 1;
    }
    return sel;
}

// sum += (float)h for the fp16 h in the low 16 bits of x (exact conversion,
// one rounding: the same value as converting then adding).
__device__ __forceinline__ void add_f16(float& sum, uint32_t x) {
    const unsigned short h = static_cast<unsigned short>(x & 0xFFFFu);
    asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(sum) : "h"(h));
}

// Word pair holding half `col` of a block row of NW words: words 2*(col/4)
// and 2*(col/4)+1, picked by a select tree on the bits of col/4.
template <int NW>
__device__ __forceinline__ void pair_of(const uint32_t (&w)[NW], int pair, uint32_t& x, uint32_t& y) {
    constexpr int NP = NW / 2;
    uint32_t xs[NP], ys[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        xs[q] = w[2 * q];
        ys[q] = w[2 * q + 1];
    }
#pragma unroll
    for (int lvl = 1; lvl < NP; lvl <<= 1) {
        const bool hi = (pair & lvl) != 0;
#pragma unroll
        for (int q = 0; q < NP; q += 2 * lvl) {
            xs[q] = hi ? xs[q + lvl] : xs[q];
            ys[q] = hi ? ys[q + lvl] : ys[q];
        }
    }
    x = xs[0];
    y = ys[0];
}

// Byte-permute selector that moves half (col % 4) of a word pair into the
// low 16 bits.
__device__ __forceinline__ uint32_t half_selector(int col) {
    const uint32_t b = 2u * static_cast<uint32_t>(col & 3);
    return b | ((b + 1u) << 4);
}

// 2 of the 4 values packed as P = a0 | a1 << 16, Q = a2 | a3 << 16: the two
// with the largest |a| (lower slot on ties), in slot order, as one word
// v0 | v1 << 16; returns the 4-bit code s0 | s1 << 2.
__device__ __forceinline__ uint32_t keep2of4_packed(uint32_t P, uint32_t Q, uint32_t& out) {
    // unique keys (|a| << 2 | 3 - slot): larger |a| first, then the lower slot
    const uint32_t mP = P & 0x7FFF7FFFu, mQ = Q & 0x7FFF7FFFu;
    const uint32_t k0 = ((mP & 0xFFFFu) << 2) | 3u, k1 = ((mP >> 16) << 2) | 2u;
    const uint32_t k2 = ((mQ & 0xFFFFu) << 2) | 1u, k3 = (mQ >> 16) << 2;
    const uint32_t a = max(k0, k1), b = min(k0, k1), c = max(k2, k3), d = min(k2, k3);
    const uint32_t t1 = max(a, c), t2 = max(min(a, c), max(b, d));  // largest and second largest
    const uint32_t i1 = 3u - (t1 & 3u), i2 = 3u - (t2 & 3u);
    const uint32_t s0 = min(i1, i2), s1 = max(i1, i2);
    // bytes 2s, 2s+1 of the 8-byte (P, Q) for s0 then s1
    const uint32_t sel = (2u * s0) | ((2u * s0 + 1u) << 4) | ((2u * s1) << 8) | ((2u * s1 + 1u) << 12);
    out = __byte_perm(P, Q, sel);
    return s0 | (s1 << 2);
}

constexpr int kColsBlocks = 8;   // blocks per CTA: consecutive blocks of one block row

// Compress for M in {8, 16, 32}. A CTA owns blocks (i, j0 .. j0+7) over all
// V rows. Lane (b, g) = (lane % 8, lane / 8) of warp w handles block j0+b in
// rows r = 4w + g + 32t, so each row a warp reads is 8 adjacent block rows
// (coalesced 16-byte loads). Pass 1: fp32 column sums of |w|, combined over
// g by shuffles and over warps in shared memory. Ranking: warp w ranks block
// j0+w with lane c holding column c; the fp32 ranking is the exact one
// whenever the gap between the 4th and 5th sums is beyond the fp32 error
// bound of such a sum (relative V * 2^-24; 2.5 x that is required), else that
// warp re-sums the block's columns exactly as integers (units of 2^-24).
// Pass 2: keep 2 of the 4 selected values per row, write values and m-index
// bytes (two blocks per byte, paired by a shuffle). With RPL > 0 (V <= 32 *
// RPL) the rows stay in registers between the passes; with RPL == 0 pass 2
// re-reads them (L1-resident: a CTA's rows are V * 16 * M bytes).
// Two resident CTAs per SM bound the registers; measured faster for every
// variant except M = 16 with four rows per lane, which runs best unbounded.
template <int MB, int RPL, int kColsWarps>
__global__ void __launch_bounds__(kColsWarps * 32, (MB == 16 && RPL == 4) ? 1 : 2)
    compress_cols_kernel(const CompressArgs p) {
    constexpr int kVec = MB / 8;     // 16-byte chunks per block row
    constexpr int kNW = MB / 2;      // 32-bit words per block row
    constexpr int kRowStep = 4 * kColsWarps;
    __shared__ float s_sum[kColsWarps][kColsBlocks][MB];
    __shared__ uint32_t s_sel[kColsBlocks];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = lane & 7, g = lane >> 3;
    // grid: x = tiles of 8 blocks along a block row, (y, z) = block row
    const int64_t i = static_cast<int64_t>(blockIdx.z) * 65535 + blockIdx.y;
    if (i >= p.R / p.V) return;  // the whole CTA (before any barrier)
    const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kColsBlocks;
    const int64_t j = j0 + b;
    const bool valid = j < p.nblk;
    const int V = p.V;
    const int64_t ld = p.ld_w;
    const uint16_t* Wrow = p.W + (i * V) * ld;  // row 0 of block row i
    const uint16_t* Wb = Wrow + (valid ? j : 0) * MB;

    // ---- pass 1: partial column sums
    float sum[MB];
#pragma unroll
    for (int c = 0; c < MB; ++c) sum[c] = 0.f;
    uint4 x[RPL > 0 ? RPL : 1][kVec];
    auto add_pair = [&](uint32_t w, int c) {  // |w| of two fp16 (sign bits cleared) into sum[c], sum[c+1]
        const uint32_t m = w & 0x7FFF7FFFu;
        add_f16(sum[c], m);
        add_f16(sum[c + 1], m >> 16);
    };
    auto accumulate = [&](const uint4 (&xr)[kVec]) {
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            add_pair(xr[v].x, 8 * v);
            add_pair(xr[v].y, 8 * v + 2);
            add_pair(xr[v].z, 8 * v + 4);
            add_pair(xr[v].w, 8 * v + 6);
        }
    };
    if constexpr (RPL > 0) {
#pragma unroll
        for (int t = 0; t < RPL; ++t) {
            const int r = 4 * warp + g + kRowStep * t;
            const bool act = valid && r < V;
#pragma unroll
            for (int v = 0; v < kVec; ++v)
                x[t][v] = act ? __ldg(reinterpret_cast<const uint4*>(Wb + r * ld) + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int t = 0; t < RPL; ++t) accumulate(x[t]);
    } else {
#pragma unroll 2
        for (int r = 4 * warp + g; r < V; r += kRowStep) {
            if (!valid) break;
#pragma unroll
            for (int v = 0; v < kVec; ++v) x[0][v] = __ldg(reinterpret_cast<const uint4*>(Wb + r * ld) + v);
            accumulate(x[0]);
        }
    }
#pragma unroll
    for (int c = 0; c < MB; ++c) {
        sum[c] += __shfl_xor_sync(0xFFFFFFFFu, sum[c], 8);
        sum[c] += __shfl_xor_sync(0xFFFFFFFFu, sum[c], 16);
    }
    if (g == 0) {
#pragma unroll
        for (int c = 0; c < MB; ++c) s_sum[warp][b][c] = sum[c];
    }
    __syncthreads();

    // ---- ranking: 32/MB blocks per warp, lane = MB * group + column; the
    // first MB/4 warps rank the CTA's 8 blocks
    constexpr int kGroups = 32 / MB;
    constexpr int kRankWarps = kColsBlocks / kGroups;
    for (int rw = warp; rw < kRankWarps; rw += kColsWarps) {  // warp-uniform
        const int grp = lane / MB, c = lane % MB;
        const int blk = rw * kGroups + grp;
        const bool has = j0 + blk < p.nblk;  // per lane group
        const uint32_t gshift = static_cast<uint32_t>(grp * MB);
        const uint32_t gbits = MB == 32 ? 0xFFFFFFFFu : ((1u << MB) - 1u);
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kColsWarps; ++w) s += s_sum[w][blk][c];
        const bool any_bad = ((__ballot_sync(0xFFFFFFFFu, has && !(s <= 3.4e38f)) >> gshift) & gbits) != 0;
        int rk = 0;
#pragma unroll
        for (int c2 = 0; c2 < MB; ++c2) {
            const float o = __shfl_sync(0xFFFFFFFFu, s, c2, MB);
            rk += (o > s) || (o == s && c2 < c);
        }
        uint32_t mask = (__ballot_sync(0xFFFFFFFFu, rk < 4) >> gshift) & gbits;
        const int l3 = __ffs((__ballot_sync(0xFFFFFFFFu, rk == 3) >> gshift) & gbits) - 1;
        const int l4 = __ffs((__ballot_sync(0xFFFFFFFFu, rk == 4) >> gshift) & gbits) - 1;
        const float v3 = __shfl_sync(0xFFFFFFFFu, s, l3 & (MB - 1), MB);
        const float v4 = __shfl_sync(0xFFFFFFFFu, s, l4 & (MB - 1), MB);
        const bool safe = !any_bad && l3 >= 0 && l4 >= 0 &&
                          (v3 - v4 > 2.5f * static_cast<float>(V) * 5.9604645e-8f * v3);
        if (__any_sync(0xFFFFFFFFu, has && !safe)) {
            // exact sums in units of 2^-24 (the whole warp, for the groups that need them)
            uint64_t e = 0;
            if (has) {
                const uint16_t* col = Wrow + (j0 + blk) * MB + c;
                for (int r = 0; r < V; ++r) e += mag_units(col[r * ld]);
            }
            int rk2 = 0;
#pragma unroll
            for (int c2 = 0; c2 < MB; ++c2) {
                const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(e), c2, MB);
                const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(e >> 32), c2, MB);
                const uint64_t o = (static_cast<uint64_t>(hi) << 32) | lo;
                rk2 += (o > e) || (o == e && c2 < c);
            }
            const uint32_t m2 = (__ballot_sync(0xFFFFFFFFu, rk2 < 4) >> gshift) & gbits;
            if (!safe) mask = m2;
        }
        if (has && c == 0) {
            const uint32_t sel = mask_to_cols(mask);
            s_sel[blk] = sel;
            p.colidx[i * p.nblk + j0 + blk] = sel;
            if (any_bad) record_error(p.status, VNM_ERR_NONFINITE, 5);
        }
    }
    __syncthreads();

    // ---- pass 2: 2 of the 4 selected values per row
    const uint32_t sel = s_sel[b];
    const int col0 = sel & 0xFF, col1 = (sel >> 8) & 0xFF, col2 = (sel >> 16) & 0xFF, col3 = sel >> 24;
    const uint32_t bs0 = half_selector(col0), bs1 = half_selector(col1), bs2 = half_selector(col2),
                   bs3 = half_selector(col3);
    const bool pair_lo = (j & 1) == 0;
    auto emit = [&](const uint4 (&xr)[kVec], int r, bool act) {
        uint32_t w[kNW];
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            w[4 * v] = xr[v].x;
            w[4 * v + 1] = xr[v].y;
            w[4 * v + 2] = xr[v].z;
            w[4 * v + 3] = xr[v].w;
        }
        // the 4 selected values as P = a0 | a1 << 16, Q = a2 | a3 << 16
        uint32_t x, y;
        pair_of<kNW>(w, col0 >> 2, x, y);
        const uint32_t h0 = __byte_perm(x, y, bs0);
        pair_of<kNW>(w, col1 >> 2, x, y);
        const uint32_t h1 = __byte_perm(x, y, bs1);
        pair_of<kNW>(w, col2 >> 2, x, y);
        const uint32_t h2 = __byte_perm(x, y, bs2);
        pair_of<kNW>(w, col3 >> 2, x, y);
        const uint32_t h3 = __byte_perm(x, y, bs3);
        const uint32_t P = __byte_perm(h0, h1, 0x5410u), Q = __byte_perm(h2, h3, 0x5410u);
        uint32_t vals;
        uint32_t code = keep2of4_packed(P, Q, vals);
        if (!act) code = 0;
        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, code, 1);  // the neighbouring block's code
        if (act) {
            const int64_t row = i * V + r;
            *reinterpret_cast<uint32_t*>(p.values + row * (2 * p.nblk) + 2 * j) = vals;
            if (pair_lo) p.meta[row * p.mpitch + (j >> 1)] = static_cast<uint8_t>(code | (other << 4));
        }
    };
    if constexpr (RPL > 0) {
#pragma unroll
        for (int t = 0; t < RPL; ++t) {
            const int r = 4 * warp + g + kRowStep * t;
            emit(x[t], r, valid && r < V);
        }
    } else {
        // r0 is uniform over the warp, so every lane reaches the shuffle in emit
        for (int r0 = 4 * warp; r0 < V; r0 += kRowStep) {
            const int r = r0 + g;
            const bool act = valid && r < V;
#pragma unroll
            for (int v = 0; v < kVec; ++v)
                x[0][v] = act ? __ldg(reinterpret_cast<const uint4*>(Wb + r * ld) + v) : make_uint4(0, 0, 0, 0);
            emit(x[0], r, act);
        }
    }
}

// Warp-tile compress for M in {8, 16} when a lane can hold all its rows
// (RPL = V/4 rows, RPL * M/8 16-byte chunks <= 16): each warp owns blocks
// (i, j0 .. j0+7) over all V rows on its own, with warp-level
// synchronisation only. Lane (b, g) = (lane % 8, lane / 8) holds rows
// r = g + 4t of block j0 + b in registers; the column sums are reduced over g
// by shuffles, handed to the ranking lanes (32/M blocks per pass, lane =
// M * group + column) through the warp's shared-memory slot, and the 2-of-4
// step runs from the registers.
constexpr int kTileWarps = 4;  // warp tiles per CTA (consecutive along a block row)

template <int MB, int RPL>
__global__ void __launch_bounds__(kTileWarps * 32) compress_warp_kernel(const CompressArgs p) {
    constexpr int kVec = MB / 8;
    constexpr int kNW = MB / 2;
    constexpr int kGroups = 32 / MB;
    __shared__ float s_sum[kTileWarps][kColsBlocks][MB];
    __shared__ uint32_t s_sel[kTileWarps][kColsBlocks];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = lane & 7, g = lane >> 3;
    const int64_t i = static_cast<int64_t>(blockIdx.z) * 65535 + blockIdx.y;
    const int64_t j0 = (static_cast<int64_t>(blockIdx.x) * kTileWarps + warp) * kColsBlocks;
    if (i >= p.R / p.V || j0 >= p.nblk) return;  // the whole warp; no CTA barrier follows
    const int64_t j = j0 + b;
    const bool valid = j < p.nblk;
    const int V = p.V;
    const int64_t ld = p.ld_w;
    const uint16_t* Wrow = p.W + (i * V) * ld;
    const uint16_t* Wb = Wrow + (valid ? j : 0) * MB;

    // ---- pass 1: all rows of this lane in flight, column sums
    uint4 x[RPL][kVec];
#pragma unroll
    for (int t = 0; t < RPL; ++t) {
        const int r = g + 4 * t;
        const bool act = valid && r < V;
#pragma unroll
        for (int v = 0; v < kVec; ++v)
            x[t][v] = act ? __ldg(reinterpret_cast<const uint4*>(Wb + r * ld) + v) : make_uint4(0, 0, 0, 0);
    }
    float sum[MB];
#pragma unroll
    for (int c = 0; c < MB; ++c) sum[c] = 0.f;
#pragma unroll
    for (int t = 0; t < RPL; ++t) {
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            const uint32_t w4[4] = {x[t][v].x & 0x7FFF7FFFu, x[t][v].y & 0x7FFF7FFFu, x[t][v].z & 0x7FFF7FFFu,
                                    x[t][v].w & 0x7FFF7FFFu};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                add_f16(sum[8 * v + 2 * h], w4[h]);
                add_f16(sum[8 * v + 2 * h + 1], w4[h] >> 16);
            }
        }
    }
#pragma unroll
    for (int c = 0; c < MB; ++c) {
        sum[c] += __shfl_xor_sync(0xFFFFFFFFu, sum[c], 8);
        sum[c] += __shfl_xor_sync(0xFFFFFFFFu, sum[c], 16);
    }
    if (g == 0) {
#pragma unroll
        for (int c = 0; c < MB; ++c) s_sum[warp][b][c] = sum[c];
    }
    __syncwarp();

    // ---- ranking: 32/M blocks per pass
    for (int pass = 0; pass < kColsBlocks / kGroups; ++pass) {
        const int grp = lane / MB, c = lane % MB;
        const int blk = pass * kGroups + grp;
        const bool has = j0 + blk < p.nblk;
        const uint32_t gshift = static_cast<uint32_t>(grp * MB);
        const uint32_t gbits = (1u << MB) - 1u;
        const float s = s_sum[warp][blk][c];
        const bool any_bad = ((__ballot_sync(0xFFFFFFFFu, has && !(s <= 3.4e38f)) >> gshift) & gbits) != 0;
        int rk = 0;
#pragma unroll
        for (int c2 = 0; c2 < MB; ++c2) {
            const float o = __shfl_sync(0xFFFFFFFFu, s, c2, MB);
            rk += (o > s) || (o == s && c2 < c);
        }
        uint32_t mask = (__ballot_sync(0xFFFFFFFFu, rk < 4) >> gshift) & gbits;
        const int l3 = __ffs((__ballot_sync(0xFFFFFFFFu, rk == 3) >> gshift) & gbits) - 1;
        const int l4 = __ffs((__ballot_sync(0xFFFFFFFFu, rk == 4) >> gshift) & gbits) - 1;
        const float v3 = __shfl_sync(0xFFFFFFFFu, s, l3 & (MB - 1), MB);
        const float v4 = __shfl_sync(0xFFFFFFFFu, s, l4 & (MB - 1), MB);
        const bool safe = !any_bad && l3 >= 0 && l4 >= 0 &&
                          (v3 - v4 > 2.5f * static_cast<float>(V) * 5.9604645e-8f * v3);
        if (__any_sync(0xFFFFFFFFu, has && !safe)) {
            uint64_t e = 0;
            if (has) {
                const uint16_t* col = Wrow + (j0 + blk) * MB + c;
                for (int r = 0; r < V; ++r) e += mag_units(col[r * ld]);
            }
            int rk2 = 0;
#pragma unroll
            for (int c2 = 0; c2 < MB; ++c2) {
                const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(e), c2, MB);
                const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(e >> 32), c2, MB);
                const uint64_t o = (static_cast<uint64_t>(hi) << 32) | lo;
                rk2 += (o > e) || (o == e && c2 < c);
            }
            const uint32_t m2 = (__ballot_sync(0xFFFFFFFFu, rk2 < 4) >> gshift) & gbits;
            if (!safe) mask = m2;
        }
        if (has && c == 0) {
            const uint32_t sel = mask_to_cols(mask);
            s_sel[warp][blk] = sel;
            p.colidx[i * p.nblk + j0 + blk] = sel;
            if (any_bad) record_error(p.status, VNM_ERR_NONFINITE, 6);
        }
    }
    __syncwarp();

    // ---- pass 2: 2 of the 4 selected values per row, from the registers
    const uint32_t sel = valid ? s_sel[warp][b] : 0x03020100u;
    const int col0 = sel & 0xFF, col1 = (sel >> 8) & 0xFF, col2 = (sel >> 16) & 0xFF, col3 = sel >> 24;
    const uint32_t bs0 = half_selector(col0), bs1 = half_selector(col1), bs2 = half_selector(col2),
                   bs3 = half_selector(col3);
    const bool pair_lo = (j & 1) == 0;
#pragma unroll
    for (int t = 0; t < RPL; ++t) {
        const int r = g + 4 * t;
        const bool act = valid && r < V;
        uint32_t w[kNW];
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            w[4 * v] = x[t][v].x;
            w[4 * v + 1] = x[t][v].y;
            w[4 * v + 2] = x[t][v].z;
            w[4 * v + 3] = x[t][v].w;
        }
        uint32_t xx, yy;
        pair_of<kNW>(w, col0 >> 2, xx, yy);
        const uint32_t h0 = __byte_perm(xx, yy, bs0);
        pair_of<kNW>(w, col1 >> 2, xx, yy);
        const uint32_t h1 = __byte_perm(xx, yy, bs1);
        pair_of<kNW>(w, col2 >> 2, xx, yy);
        const uint32_t h2 = __byte_perm(xx, yy, bs2);
        pair_of<kNW>(w, col3 >> 2, xx, yy);
        const uint32_t h3 = __byte_perm(xx, yy, bs3);
        const uint32_t P = __byte_perm(h0, h1, 0x5410u), Q = __byte_perm(h2, h3, 0x5410u);
        uint32_t vals;
        uint32_t code = keep2of4_packed(P, Q, vals);
        if (!act) code = 0;
        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, code, 1);  // the neighbouring block's code
        if (act) {
            const int64_t row = i * V + r;
            *reinterpret_cast<uint32_t*>(p.values + row * (2 * p.nblk) + 2 * j) = vals;
            if (pair_lo) p.meta[row * p.mpitch + (j >> 1)] = static_cast<uint8_t>(code | (other << 4));
        }
    }
}

template <int MB>
void launch_cols(const CompressArgs& p, dim3 grid, cudaStream_t stream) {
    const int V = p.V;
    constexpr int W = 8;  // warps per CTA (4 measured slower: fewer rows in flight per CTA)
    if (V <= 32) compress_cols_kernel<MB, 1, W><<<grid, 32 * W, 0, stream>>>(p);
    else if (V <= 64) compress_cols_kernel<MB, 2, W><<<grid, 32 * W, 0, stream>>>(p);
    else if (V <= 128) compress_cols_kernel<MB, 4, W><<<grid, 32 * W, 0, stream>>>(p);
    else compress_cols_kernel<MB, 0, W><<<grid, 32 * W, 0, stream>>>(p);
}

// M == 4: column-loc is the identity, so prune-and-encode is the 2:4 step
// alone, on each group of 4 consecutive weights of a row. One thread turns
// 16 consecutive weights (32 bytes) into 8 values (16 bytes) and 4 nibbles
// of m-indices (2 bytes); consecutive threads take consecutive chunks of a
// row, so loads and stores are fully coalesced and no shared memory is used.
constexpr int kM4Threads = 256;

__global__ void __launch_bounds__(kM4Threads) compress_m4_kernel(const CompressArgs p) {
    const int64_t cpr = p.K / 16;  // 16-weight chunks per row
    const int64_t total = p.R * cpr;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kM4Threads;
    const int64_t sr = stride / cpr, sx = stride % cpr;  // the stride in rows and chunks
    int64_t q = static_cast<int64_t>(blockIdx.x) * kM4Threads + threadIdx.x;
    int64_t r = q / cpr, x = q % cpr;
    uint32_t nonfinite = 0;
#pragma unroll 2
    for (; q < total; q += stride) {
        const uint4* src = reinterpret_cast<const uint4*>(p.W + r * p.ld_w + 16 * x);
        const uint4 a = __ldg(src), b = __ldg(src + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t v[4];
        uint32_t code = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            // a group of 4 weights is the word pair (w[2g], w[2g+1])
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t e = w[2 * g + h] & 0x7C007C00u;  // exponent fields of both halves
                nonfinite |= ((e & 0xFFFFu) == 0x7C00u) | ((e >> 16) == 0x7C00u);
            }
            code |= keep2of4_packed(w[2 * g], w[2 * g + 1], v[g]) << (4 * g);
        }
        *reinterpret_cast<uint4*>(p.values + r * (p.K / 2) + 8 * x) = make_uint4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<uint16_t*>(p.meta + r * p.mpitch + 2 * x) = static_cast<uint16_t>(code);
        x += sx;
        r += sr;
        if (x >= cpr) {
            x -= cpr;
            ++r;
        }
    }
    const int64_t ncw = (p.R / p.V) * p.nblk;  // column-loc words: always 0, 1, 2, 3
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kM4Threads + threadIdx.x; q < ncw; q += stride)
        p.colidx[q] = 0x03020100u;
    if (__any_sync(0xFFFFFFFFu, nonfinite) && (threadIdx.x & 31) == 0) record_error(p.status, VNM_ERR_NONFINITE, 4);
}

struct DecompressArgs {
    const uint16_t* values;
    const uint8_t* meta;
    const uint32_t* colidx;
    uint16_t* W;
    int64_t ld_w, R, K;
    int V, M;
    int64_t nblk, mpitch;
};

// One thread per (row, block): write the block's M columns of that row.
__global__ void decompress_kernel(const DecompressArgs p) {
    const int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (q >= p.R * p.nblk) return;
    const int64_t row = q / p.nblk, j = q % p.nblk;
    const uint32_t sel = p.colidx[(row / p.V) * p.nblk + j];
    const uint32_t code = (p.meta[row * p.mpitch + j / 2] >> (4 * (j & 1))) & 0xFu;
    const int c0 = (sel >> (8 * (code & 3u))) & 0xFF;
    const int c1 = (sel >> (8 * (code >> 2))) & 0xFF;
    const uint16_t v0 = p.values[row * 2 * p.nblk + 2 * j];
    const uint16_t v1 = p.values[row * 2 * p.nblk + 2 * j + 1];
    uint16_t* out = p.W + row * p.ld_w + j * p.M;
    for (int c = 0; c < p.M; ++c) out[c] = c == c0 ? v0 : (c == c1 ? v1 : static_cast<uint16_t>(0));
}

}  // namespace

cudaError_t launch_compress(const vnm_matrix_s& A, const void* W, int64_t ld_w, cudaStream_t stream) {
    CompressArgs p;
    p.W = static_cast<const uint16_t*>(W);
    p.ld_w = ld_w;
    p.R = A.R;
    p.K = A.K;
    p.V = A.V;
    p.M = A.M;
    p.values = static_cast<uint16_t*>(A.values);
    p.meta = static_cast<uint8_t*>(A.meta);
    p.colidx = static_cast<uint32_t*>(A.colidx);
    p.nblk = A.K / A.M;
    p.mpitch = meta_pitch(A.K, A.M);
    p.status = A.status;
    if (A.R == 0 || A.K == 0) return cudaSuccess;
    if (A.M == 4 && A.K % 16 == 0 && reinterpret_cast<uintptr_t>(W) % 16 == 0 && ld_w % 8 == 0) {
        // one full wave of resident CTAs, each striding over the chunks
        static std::atomic<int> per_sm_cache{0};  // resident CTAs per SM, once per process
        int per_sm = per_sm_cache.load(std::memory_order_relaxed);
        if (per_sm == 0) {
            int occ = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, compress_m4_kernel, kM4Threads, 0) != cudaSuccess)
                occ = 4;
            per_sm = std::max(1, occ);
            per_sm_cache.store(per_sm, std::memory_order_relaxed);
        }
        const int64_t chunks = A.R * (A.K / 16);
        const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((chunks + kM4Threads - 1) / kM4Threads,
                                                                      static_cast<int64_t>(A.sm_count) * per_sm));
        compress_m4_kernel<<<static_cast<unsigned>(blocks), kM4Threads, 0, stream>>>(p);
        return cudaGetLastError();
    }
    // M in {8, 16, 32}: eight blocks x V rows per CTA, no staging
    if ((A.M == 8 || A.M == 16 || A.M == 32) && reinterpret_cast<uintptr_t>(W) % 16 == 0 && ld_w % 8 == 0) {
        const int64_t rows = A.R / A.V;  // block rows: grid y (then z past 65535)
        const int64_t tiles = (p.nblk + kColsBlocks - 1) / kColsBlocks;
        // one warp per tile when a lane holds all its rows (V <= 64 at M = 8, V <= 32 at M = 16)
        if ((A.M == 8 && A.V <= 64 && A.V % 4 == 0) || (A.M == 16 && A.V <= 32 && A.V % 4 == 0)) {
            const dim3 wgrid(static_cast<unsigned>((tiles + kTileWarps - 1) / kTileWarps),
                             static_cast<unsigned>(std::min<int64_t>(rows, 65535)),
                             static_cast<unsigned>((rows + 65534) / 65535));
            const unsigned th = kTileWarps * 32;
            if (A.M == 8) {
                if (A.V <= 16) compress_warp_kernel<8, 4><<<wgrid, th, 0, stream>>>(p);
                else if (A.V <= 32) compress_warp_kernel<8, 8><<<wgrid, th, 0, stream>>>(p);
                else compress_warp_kernel<8, 16><<<wgrid, th, 0, stream>>>(p);
            } else {
                if (A.V <= 16) compress_warp_kernel<16, 4><<<wgrid, th, 0, stream>>>(p);
                else compress_warp_kernel<16, 8><<<wgrid, th, 0, stream>>>(p);
            }
            return cudaGetLastError();
        }
        const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(std::min<int64_t>(rows, 65535)),
                        static_cast<unsigned>((rows + 65534) / 65535));
        if (A.M == 8) launch_cols<8>(p, grid, stream);
        else if (A.M == 16) launch_cols<16>(p, grid, stream);
        else launch_cols<32>(p, grid, stream);
        return cudaGetLastError();
    }
    // tile width: an even number of blocks, as many as fit the budget
    int64_t pairs = kTileElems / (static_cast<int64_t>(A.V) * 2 * A.M);
    pairs = std::min<int64_t>(pairs, kTileMaxCols / (2 * A.M));
    if (pairs >= 1) {
        p.tk = static_cast<int>(pairs * 2 * A.M);
        p.vec_load = (reinterpret_cast<uintptr_t>(W) % 16 == 0) && (ld_w % 8 == 0) && (p.tk % 8 == 0);
        const size_t smem = tile_bytes_aligned(A.V, p.tk) + sizeof(uint64_t) * p.tk +
                            sizeof(uint32_t) * (p.tk / A.M);
        // largest dynamic shared memory sizes set so far (one lock for check and set,
        // so that concurrent calls never lower a size another call relies on)
        static std::mutex smem_mutex;
        static size_t configured = 0;
        std::lock_guard<std::mutex> smem_lock(smem_mutex);
        if (smem > 48 * 1024 && smem > configured) {
            cudaError_t e = cudaFuncSetAttribute(compress_tiled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            configured = smem;
        }
        if (p.vec_load) {
            // persistent, double-buffered: two tiles + column sums + exact sums + selections
            const size_t ssmem = 2 * tile_bytes_aligned(A.V, p.tk) + sizeof(float) * (p.tk + 1) +
                                 sizeof(uint64_t) * p.tk + sizeof(uint32_t) * (p.tk / A.M + 4) +
                                 sizeof(float) * kCompressThreads * 8 + 8 * 256 + 16;
            static size_t sconfigured = 0;
            if (ssmem > 48 * 1024 && ssmem > sconfigured) {
                cudaError_t e = cudaFuncSetAttribute(compress_stream_kernel,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     static_cast<int>(ssmem));
                if (e != cudaSuccess) return e;
                sconfigured = ssmem;
            }
            const int64_t n_tiles = (A.R / A.V) * ((A.K + p.tk - 1) / p.tk);
            const int64_t fit = std::max<int64_t>(1, std::min<int64_t>(kStreamCtasPerSm, (220 * 1024) / ssmem));
            const int64_t ctas = std::min<int64_t>(n_tiles, static_cast<int64_t>(A.sm_count) * fit);
            compress_stream_kernel<<<static_cast<unsigned>(ctas), kCompressThreads, ssmem, stream>>>(p);
            return cudaGetLastError();
        }
        dim3 grid(static_cast<unsigned>((A.K + p.tk - 1) / p.tk), static_cast<unsigned>(A.R / A.V));
        compress_tiled_kernel<<<grid, kCompressThreads, smem, stream>>>(p);
    } else {
        p.tk = 0;
        p.vec_load = false;
        dim3 grid(static_cast<unsigned>((p.nblk + 1) / 2), static_cast<unsigned>(A.R / A.V));
        compress_block_kernel<<<grid, kCompressThreads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_decompress(const vnm_matrix_s& A, void* W, int64_t ld_w, cudaStream_t stream) {
    if (A.R == 0 || A.K == 0) return cudaSuccess;
    DecompressArgs p;
    p.values = static_cast<const uint16_t*>(A.values);
    p.meta = static_cast<const uint8_t*>(A.meta);
    p.colidx = static_cast<const uint32_t*>(A.colidx);
    p.W = static_cast<uint16_t*>(W);
    p.ld_w = ld_w;
    p.R = A.R;
    p.K = A.K;
    p.V = A.V;
    p.M = A.M;
    p.nblk = A.K / A.M;
    p.mpitch = meta_pitch(A.K, A.M);
    const int64_t n = A.R * p.nblk;
    const int threads = 256;
    decompress_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace vnm
