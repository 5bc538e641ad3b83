// Energy (magnitude preservation) of a pruning pattern: the sum of the kept
// |w| over the sum of all |w| of a dense fp16 matrix W, at the V:N:M
// density 2/M, for three selection policies.
//
// VENOM: A Vectorized N:M Format for Unleashing the Power of Sparse Tensor
// Cores, section 5 (Figure 11): the energy metric, and the comparison of
// unstructured magnitude pruning (the ideal selection), V:N:M with several V,
// and vector-wise pruning with vector length l.
//   V:N:M         the kept values of the compressed matrix (vnm_compress).
//   unstructured  the 2RK/M largest |w| of the whole matrix.
//   vector-wise   per panel of l = V consecutive rows, the 2K/M columns of
//                 largest L1 norm over the panel (vectors of l x 1).
// All sums are exact integers in units of 2^-24 (|fp16| is an integer
// multiple of 2^-24 below 2^41 units); ties between equal magnitudes or
// column norms cannot change a kept sum, so each energy is unique.
//
// GB300 design: memory-bound passes over W with per-CTA 128-bit partial sums;
// the unstructured threshold from a 32768-bin histogram of the 15-bit
// magnitude codes (shared-memory histogram per CTA, one CTA per SM); the
// vector-wise threshold per panel by an 8-pass radix select over the panel's
// exact column norms. The host adds the partials.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>

#include "vnm_internal.h"
#include "vnm_select.cuh"

namespace vnm {
namespace {

constexpr int kEnThreads = 256;
constexpr int kHistBins = 1 << 15;   // |fp16| bit patterns 0 .. 0x7FFF
constexpr int kSelThreads = 1024;

typedef unsigned __int128 u128;

struct EnergyArgs {
    const uint16_t* W;
    int64_t ld_w, R, K;
    int V;
    int* flags;      // [0]: a non-finite weight seen
};

__device__ __forceinline__ u128 block_sum_u128(u128 v, u128* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // warp: through two 64-bit halves
    uint64_t lo = static_cast<uint64_t>(v), hi = static_cast<uint64_t>(v >> 64);
    for (int off = 16; off > 0; off >>= 1) {
        const uint64_t olo = __shfl_xor_sync(0xFFFFFFFFu, lo, off);
        const uint64_t ohi = __shfl_xor_sync(0xFFFFFFFFu, hi, off);
        const uint64_t nlo = lo + olo;
        hi = hi + ohi + (nlo < lo ? 1u : 0u);
        lo = nlo;
    }
    if (lane == 0) red[warp] = (static_cast<u128>(hi) << 64) | lo;
    __syncthreads();
    u128 s = 0;
    if (threadIdx.x == 0)
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += red[w];
    __syncthreads();
    return s;  // valid in thread 0
}

// Sum of |w| over W (and the non-finite flag): one 128-bit partial per CTA.
__global__ void __launch_bounds__(kEnThreads) energy_total_kernel(const EnergyArgs p, uint64_t* partial) {
    __shared__ u128 red[kEnThreads / 32];
    u128 acc = 0;
    bool bad = false;
    for (int64_t r = blockIdx.x; r < p.R; r += gridDim.x)
        for (int64_t c = threadIdx.x; c < p.K; c += blockDim.x) {
            const uint16_t h = p.W[r * p.ld_w + c];
            bad |= half_nonfinite(h);
            acc += mag_units(h);
        }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicExch(p.flags, 1);
    const u128 s = block_sum_u128(acc, red);
    if (threadIdx.x == 0) {
        partial[2 * blockIdx.x] = static_cast<uint64_t>(s);
        partial[2 * blockIdx.x + 1] = static_cast<uint64_t>(s >> 64);
    }
}

// Sum of |v| over n stored fp16 values (the kept weights of V:N:M).
__global__ void __launch_bounds__(kEnThreads) energy_values_kernel(const uint16_t* values, int64_t n,
                                                                   uint64_t* partial) {
    __shared__ u128 red[kEnThreads / 32];
    u128 acc = 0;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x)
        acc += mag_units(values[e]);
    const u128 s = block_sum_u128(acc, red);
    if (threadIdx.x == 0) {
        partial[2 * blockIdx.x] = static_cast<uint64_t>(s);
        partial[2 * blockIdx.x + 1] = static_cast<uint64_t>(s >> 64);
    }
}

// Counts of each 15-bit magnitude code of W: a shared histogram per CTA,
// added into the global one.
__global__ void __launch_bounds__(kEnThreads) energy_hist_kernel(const EnergyArgs p, unsigned long long* hist) {
    extern __shared__ uint32_t sh[];  // kHistBins counts
    for (int b = threadIdx.x; b < kHistBins; b += blockDim.x) sh[b] = 0u;
    __syncthreads();
    for (int64_t r = blockIdx.x; r < p.R; r += gridDim.x)
        for (int64_t c = threadIdx.x; c < p.K; c += blockDim.x) atomicAdd(&sh[p.W[r * p.ld_w + c] & 0x7FFFu], 1u);
    __syncthreads();
    for (int b = threadIdx.x; b < kHistBins; b += blockDim.x)
        if (sh[b]) atomicAdd(&hist[b], static_cast<unsigned long long>(sh[b]));
}

// |h| in units of 2^-24 for a 15-bit magnitude code.
__device__ __forceinline__ uint64_t code_units(uint32_t b) { return mag_units(static_cast<uint16_t>(b)); }

// The sum of the nnz largest magnitudes, from the histogram: bins above the
// threshold bin in full, the threshold bin for the remainder. One CTA.
__global__ void __launch_bounds__(kSelThreads) energy_select_kernel(const unsigned long long* hist, uint64_t nnz,
                                                                    uint64_t* out) {
    constexpr int kPer = kHistBins / kSelThreads;  // 32 bins per thread, thread 0 the highest
    __shared__ unsigned long long cnt[kSelThreads];
    __shared__ u128 red[kSelThreads / 32];
    const int t = threadIdx.x;
    const int top = kHistBins - 1 - t * kPer;  // this thread's bins: top, top-1, ..., top-kPer+1
    unsigned long long mine = 0;
    for (int q = 0; q < kPer; ++q) mine += hist[top - q];
    cnt[t] = mine;
    __syncthreads();
    // exclusive prefix from the highest bins down (serial over 1024 partials in thread 0
    // would do; a Hillis-Steele scan keeps it short)
    for (int off = 1; off < kSelThreads; off <<= 1) {
        const unsigned long long v = t >= off ? cnt[t - off] : 0ull;
        __syncthreads();
        cnt[t] += v;
        __syncthreads();
    }
    const unsigned long long above = t > 0 ? cnt[t - 1] : 0ull;  // count in higher threads' bins
    u128 acc = 0;
    unsigned long long run = above;
    for (int q = 0; q < kPer && run < nnz; ++q) {
        const uint32_t b = static_cast<uint32_t>(top - q);
        const unsigned long long c = hist[b];
        const unsigned long long take = c < nnz - run ? c : nnz - run;
        acc += static_cast<u128>(take) * code_units(b);
        run += take;
    }
    const u128 s = block_sum_u128(acc, red);
    if (t == 0) {
        out[0] = static_cast<uint64_t>(s);
        out[1] = static_cast<uint64_t>(s >> 64);
    }
}

// Exact L1 norm of every column over every panel of V rows: colsum[panel][c].
__global__ void __launch_bounds__(kEnThreads) energy_colsum_kernel(const EnergyArgs p, uint64_t* colsum) {
    const int64_t panel = blockIdx.x;
    const int64_t c = static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x;
    if (c >= p.K) return;
    const uint16_t* w = p.W + panel * p.V * p.ld_w + c;
    uint64_t s = 0;
    for (int r = 0; r < p.V; ++r) s += mag_units(w[r * p.ld_w]);
    colsum[panel * p.K + c] = s;
}

// Per panel, the sum of its k largest column norms: the k-th largest key by
// an 8-pass radix select (8 bits a pass, from the top), then keys above it
// in full and the k-th key for the remainder. One CTA per panel.
__global__ void __launch_bounds__(kEnThreads) energy_topk_kernel(const uint64_t* colsum, int64_t K, int64_t k,
                                                                 uint64_t* out) {
    __shared__ unsigned long long bins[256];
    __shared__ uint64_t s_prefix;
    __shared__ unsigned long long s_need;
    __shared__ u128 red[kEnThreads / 32];
    const uint64_t* keys = colsum + static_cast<int64_t>(blockIdx.x) * K;
    uint64_t prefix = 0;             // the high bits fixed so far
    unsigned long long need = static_cast<unsigned long long>(k);  // rank still to find among matching keys
    for (int pass = 0; pass < 8; ++pass) {
        const int shift = 56 - 8 * pass;
        const uint64_t mask = pass == 0 ? 0ull : ~0ull << (shift + 8);
        for (int b = threadIdx.x; b < 256; b += blockDim.x) bins[b] = 0ull;
        __syncthreads();
        for (int64_t c = threadIdx.x; c < K; c += blockDim.x) {
            const uint64_t v = keys[c];
            if ((v & mask) == prefix) atomicAdd(&bins[(v >> shift) & 0xFFu], 1ull);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long run = 0;
            int d = 255;
            for (; d > 0; --d) {
                if (run + bins[d] >= need) break;
                run += bins[d];
            }
            s_prefix = prefix | (static_cast<uint64_t>(d) << shift);
            s_need = need - run;
        }
        __syncthreads();
        prefix = s_prefix;
        need = s_need;
        __syncthreads();
    }
    // prefix = the k-th largest key T; need = how many of the keys equal to T are kept
    u128 acc = 0;
    for (int64_t c = threadIdx.x; c < K; c += blockDim.x) {
        const uint64_t v = keys[c];
        if (v > prefix) acc += v;
    }
    u128 s = block_sum_u128(acc, red);
    if (threadIdx.x == 0) {
        s += static_cast<u128>(need) * prefix;
        out[2 * blockIdx.x] = static_cast<uint64_t>(s);
        out[2 * blockIdx.x + 1] = static_cast<uint64_t>(s >> 64);
    }
}

constexpr int kTotalCtas = kEnergyKeptPair;

}  // namespace

size_t energy_workspace_bytes(int64_t R, int64_t K, int V) {
    // flags (256 B), total partials, kept partials (up to one per panel), and the larger of
    // the histogram and the column norms
    const size_t panels = V > 0 ? static_cast<size_t>(R / V) : 0;
    const size_t kept = std::max<size_t>(kTotalCtas, std::max<size_t>(panels, 1));
    const size_t big = std::max(sizeof(unsigned long long) * kHistBins, sizeof(uint64_t) * panels * K);
    return 256 + 16 * kTotalCtas + 16 * kept + big;
}

cudaError_t launch_energy(const vnm_matrix_s& A, const void* W, int64_t ld_w, int pattern, void* workspace,
                          int sm_count, int* n_total_partials, int* n_kept_partials, cudaStream_t stream) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    EnergyArgs p;
    p.W = static_cast<const uint16_t*>(W);
    p.ld_w = ld_w;
    p.R = A.R;
    p.K = A.K;
    p.V = A.V;
    p.flags = reinterpret_cast<int*>(ws);
    const size_t panels = static_cast<size_t>(A.R / A.V);
    uint64_t* total = reinterpret_cast<uint64_t*>(ws + 256);
    uint64_t* kept = total + 2 * kTotalCtas;
    const size_t kept_slots = std::max<size_t>(kTotalCtas, std::max<size_t>(panels, 1));
    uint8_t* big = reinterpret_cast<uint8_t*>(kept + 2 * kept_slots);
    cudaError_t e = cudaMemsetAsync(ws, 0, 256, stream);
    if (e != cudaSuccess) return e;
    const int total_ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kTotalCtas, A.R)));
    energy_total_kernel<<<total_ctas, kEnThreads, 0, stream>>>(p, total);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *n_total_partials = total_ctas;
    if (pattern == VNM_PATTERN_VNM) {
        const int64_t n = A.R * values_per_row(A.K, A.M);
        const int ctas = static_cast<int>(std::max<int64_t>(
            1, std::min<int64_t>(kTotalCtas, (n + kEnThreads * 64 - 1) / (kEnThreads * 64))));
        energy_values_kernel<<<ctas, kEnThreads, 0, stream>>>(static_cast<const uint16_t*>(A.values), n, kept);
        *n_kept_partials = ctas;
    } else if (pattern == VNM_PATTERN_UNSTRUCTURED) {
        unsigned long long* hist = reinterpret_cast<unsigned long long*>(big);
        e = cudaMemsetAsync(hist, 0, sizeof(unsigned long long) * kHistBins, stream);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(energy_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kHistBins * static_cast<int>(sizeof(uint32_t)));
        if (e != cudaSuccess) return e;
        energy_hist_kernel<<<std::max(1, sm_count), kEnThreads, kHistBins * sizeof(uint32_t), stream>>>(p, hist);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const uint64_t nnz = static_cast<uint64_t>(A.R) * static_cast<uint64_t>(values_per_row(A.K, A.M));
        energy_select_kernel<<<1, kSelThreads, 0, stream>>>(hist, nnz, kept);
        *n_kept_partials = 1;
    } else {
        uint64_t* colsum = reinterpret_cast<uint64_t*>(big);
        const dim3 grid(static_cast<unsigned>(panels), static_cast<unsigned>((A.K + kEnThreads - 1) / kEnThreads));
        energy_colsum_kernel<<<grid, kEnThreads, 0, stream>>>(p, colsum);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        energy_topk_kernel<<<static_cast<unsigned>(panels), kEnThreads, 0, stream>>>(colsum, A.K,
                                                                                     values_per_row(A.K, A.M), kept);
        *n_kept_partials = static_cast<int>(panels);
    }
    return cudaGetLastError();
}

}  // namespace vnm
