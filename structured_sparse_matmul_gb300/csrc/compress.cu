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

#include "vnm_internal.h"

namespace vnm {
namespace {

constexpr int kCompressThreads = 256;
constexpr int kTileElems = 16384;  // V x TK elements of W staged per CTA (32 KB)
constexpr int kTileMaxCols = 4096; // TK cap (bounds the column-sum array)

// |h| in units of 2^-24 (binary16: 5 exponent bits, bias 15, 10 fraction bits).
__device__ __forceinline__ uint64_t mag_units(uint16_t h) {
    const uint32_t e = (h >> 10) & 0x1Fu, f = h & 0x3FFu;
    return e == 0 ? static_cast<uint64_t>(f) : static_cast<uint64_t>(1024u + f) << (e - 1u);
}

__device__ __forceinline__ bool half_nonfinite(uint16_t h) { return (h & 0x7C00u) == 0x7C00u; }

// Top 4 of n scores: largest first, lower index first on ties; returned as
// 4 ascending column indices packed in bytes 0..3 of a word.
__device__ __forceinline__ uint32_t top4_ascending(const uint64_t* score, int n) {
    uint64_t bv[4] = {0, 0, 0, 0};
    int bi[4] = {-1, -1, -1, -1};
    for (int c = 0; c < n; ++c) {
        const uint64_t v = score[c];
        // insert after every entry that is >= v (keeps equal scores in index order)
        if (bi[3] >= 0 && v <= bv[3]) continue;
        int p = 3;
        while (p > 0 && (bi[p - 1] < 0 || v > bv[p - 1])) {
            bv[p] = bv[p - 1];
            bi[p] = bi[p - 1];
            --p;
        }
        bv[p] = v;
        bi[p] = c;
    }
    // sort the four indices ascending
    for (int a = 1; a < 4; ++a)
        for (int b = a; b > 0 && bi[b - 1] > bi[b]; --b) {
            const int t = bi[b];
            bi[b] = bi[b - 1];
            bi[b - 1] = t;
        }
    return static_cast<uint32_t>(bi[0]) | (static_cast<uint32_t>(bi[1]) << 8) |
           (static_cast<uint32_t>(bi[2]) << 16) | (static_cast<uint32_t>(bi[3]) << 24);
}

// 2 of the 4 values a[0..3] with the largest |a| (lower slot on ties), in
// ascending slot order. Returns the 4-bit code s0 | s1 << 2 and the two
// fp16 bit patterns.
__device__ __forceinline__ uint32_t keep2of4(const uint16_t a[4], uint16_t& v0, uint16_t& v1) {
    uint32_t m[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) m[s] = a[s] & 0x7FFFu;  // finite fp16 magnitudes order like integers
    int first = 0;
#pragma unroll
    for (int s = 1; s < 4; ++s)
        if (m[s] > m[first]) first = s;
    int second = first == 0 ? 1 : 0;
#pragma unroll
    for (int s = 0; s < 4; ++s)
        if (s != first && m[s] > m[second]) second = s;
    const int s0 = first < second ? first : second;
    const int s1 = first < second ? second : first;
    v0 = a[s0];
    v1 = a[s1];
    return static_cast<uint32_t>(s0) | (static_cast<uint32_t>(s1) << 2);
}

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
    // tile width: an even number of blocks, as many as fit the budget
    int64_t pairs = kTileElems / (static_cast<int64_t>(A.V) * 2 * A.M);
    pairs = std::min<int64_t>(pairs, kTileMaxCols / (2 * A.M));
    if (pairs >= 1) {
        p.tk = static_cast<int>(pairs * 2 * A.M);
        p.vec_load = (reinterpret_cast<uintptr_t>(W) % 16 == 0) && (ld_w % 8 == 0) && (p.tk % 8 == 0);
        const size_t smem = tile_bytes_aligned(A.V, p.tk) + sizeof(uint64_t) * p.tk +
                            sizeof(uint32_t) * (p.tk / A.M);
        static size_t configured = 0;  // largest dynamic shared memory size set so far
        if (smem > 48 * 1024 && smem > configured) {
            cudaError_t e = cudaFuncSetAttribute(compress_tiled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            configured = smem;
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
