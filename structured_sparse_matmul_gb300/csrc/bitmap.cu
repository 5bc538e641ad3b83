// Bitmap format for unstructured sparsity and its small-N SpMM.
//
// Coruscant: Co-Designing GPU Kernel and Sparse Tensor Core to Advocate
// Unstructured Sparsity in Efficient LLM Inference, section 3.1 (Figure 7):
// the matrix is cut into column tiles of 64 elements; a tile is its 64-bit
// bitmap of non-zero positions and its non-zero values, padded to a multiple
// of 8 (one 16-byte load per 8 values), found through a per-tile offset.
// Section 3.2: decode-time products are memory-bound, and K is split across
// thread blocks to spread the work over the SMs.
//
// Layout here (R % 64 == 0): tile (i, k) holds rows 64i .. 64i+63 of column
// k; bit r of bitmaps[i][k] is set when W[64i + r][k] is not +-0; its values
// are those rows' values in row order, then +0.0 up to a multiple of 8, from
// values[bases[i] + offsets[i][k]] (offsets relative to the row block's base,
// so that they stay 32-bit; bases[R/64] is the total length).
//
// GB300 design. Encoding: one thread per tile (a warp reads 32 consecutive
// columns of a row at once: coalesced); a CTA per row block scans its tiles'
// padded counts; one CTA scans the row-block totals. The SpMM (N small): a
// CTA per (row block, K split), no more CTAs than are resident at once; its
// four warps each all 64 rows and a quarter of the split. The values of 32
// consecutive column tiles are one contiguous run (the padding keeps it
// 16-byte aligned), so a warp streams them into shared memory with cp.async
// one chunk ahead of decoding them; lane l owns rows l and l + 32 and reads
// its own two values of a tile where its bits are set, and B's row k from
// shared memory. The CTA adds its warps' sums in shared memory; K splits go
// to fp32 partials and the split-K reduction.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>

#include "vnm_internal.h"
#include "vnm_ptx.cuh"

namespace vnm {
namespace {

constexpr int kBmRows = 64;
constexpr int kBmScanThreads = 1024;

__device__ __forceinline__ bool nonzero_f16(uint16_t h) { return (h & 0x7FFFu) != 0; }

// Per tile: its bitmap and its padded count (the count goes to offsets[] for
// the scan that follows).
__global__ void __launch_bounds__(256) bitmap_count_kernel(const uint16_t* __restrict__ W, int64_t ld_w, int64_t K,
                                                           uint64_t* __restrict__ bitmaps,
                                                           uint32_t* __restrict__ offsets) {
    const int64_t i = blockIdx.y;
    const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (k >= K) return;
    const uint16_t* w = W + i * kBmRows * ld_w + k;
    uint64_t bm = 0;
#pragma unroll 8
    for (int r = 0; r < kBmRows; ++r) bm |= static_cast<uint64_t>(nonzero_f16(w[r * ld_w])) << r;
    bitmaps[i * K + k] = bm;
    offsets[i * K + k] = (static_cast<uint32_t>(__popcll(bm)) + 7u) & ~7u;
}

// Row block i: exclusive scan of its tiles' padded counts (in place), its
// total into bases[i + 1].
__global__ void __launch_bounds__(kBmScanThreads) bitmap_scan_kernel(uint32_t* __restrict__ offsets, int64_t K,
                                                                     int64_t* __restrict__ bases) {
    __shared__ uint32_t part[kBmScanThreads];
    uint32_t* o = offsets + static_cast<int64_t>(blockIdx.x) * K;
    // each thread a contiguous chunk of columns
    const int64_t per = (K + kBmScanThreads - 1) / kBmScanThreads;
    const int64_t c0 = threadIdx.x * per, c1 = c0 + per < K ? c0 + per : K;
    uint32_t sum = 0;
    for (int64_t c = c0; c < c1; ++c) sum += o[c];
    part[threadIdx.x] = sum;
    __syncthreads();
    for (int off = 1; off < kBmScanThreads; off <<= 1) {
        const uint32_t v = threadIdx.x >= static_cast<unsigned>(off) ? part[threadIdx.x - off] : 0u;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    uint32_t run = threadIdx.x > 0 ? part[threadIdx.x - 1] : 0u;
    for (int64_t c = c0; c < c1; ++c) {
        const uint32_t n = o[c];
        o[c] = run;
        run += n;
    }
    if (threadIdx.x == kBmScanThreads - 1) bases[blockIdx.x + 1] = part[kBmScanThreads - 1];
}

// bases[0] = 0, bases[i + 1] = bases[i] + total of row block i (in place; one CTA).
__global__ void __launch_bounds__(kBmScanThreads) bitmap_bases_kernel(int64_t* __restrict__ bases, int64_t blocks) {
    __shared__ int64_t part[kBmScanThreads];
    const int64_t per = (blocks + kBmScanThreads - 1) / kBmScanThreads;
    const int64_t b0 = threadIdx.x * per, b1 = b0 + per < blocks ? b0 + per : blocks;
    int64_t sum = 0;
    for (int64_t b = b0; b < b1; ++b) sum += bases[b + 1];
    part[threadIdx.x] = sum;
    __syncthreads();
    for (int off = 1; off < kBmScanThreads; off <<= 1) {
        const int64_t v = threadIdx.x >= static_cast<unsigned>(off) ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int64_t run = threadIdx.x > 0 ? part[threadIdx.x - 1] : 0;
    for (int64_t b = b0; b < b1; ++b) {
        const int64_t n = bases[b + 1];
        bases[b + 1] = run + n;
        run += n;
    }
    if (threadIdx.x == 0) bases[0] = 0;
}

// Values of every tile in row order, then zeros up to the padded count.
__global__ void __launch_bounds__(256) bitmap_fill_kernel(const uint16_t* __restrict__ W, int64_t ld_w, int64_t K,
                                                          const uint64_t* __restrict__ bitmaps,
                                                          const uint32_t* __restrict__ offsets,
                                                          const int64_t* __restrict__ bases,
                                                          uint16_t* __restrict__ values) {
    const int64_t i = blockIdx.y;
    const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (k >= K) return;
    const uint16_t* w = W + i * kBmRows * ld_w + k;
    uint16_t* v = values + bases[i] + offsets[i * K + k];
    const uint64_t bm = bitmaps[i * K + k];
    int n = 0;
    for (int r = 0; r < kBmRows; ++r)
        if ((bm >> r) & 1ull) v[n++] = w[r * ld_w];
    const int padded = (n + 7) & ~7;
    for (; n < padded; ++n) v[n] = 0;
}

struct BmArgs {
    const uint64_t* bitmaps;
    const uint32_t* offsets;
    const int64_t* bases;
    const __half* values;
    const __half* B;
    int64_t ld_b;
    int64_t R, K, N;
    int splits;
    int64_t kps;          // columns per split
    OutSpec out;          // C (splits == 1)
    float* partial;       // [splits][R][N] fp32 (splits > 1)
};

constexpr int kBmWarps = 4;                    // each warp all 64 rows of the block and a quarter of the K range
constexpr int kBmChunk = 32;                   // column tiles per chunk (one per lane for their metadata)
constexpr int kBmSlot = kBmChunk * kBmRows;    // values of a chunk at most (fp16): 4 KB
constexpr int kBmRing = 2 * kBmSlot;           // a warp's ring of values (a power of 2), by position mod kBmRing
constexpr int kBmStageFloats = 2048;           // B's staged slice: 8 KB of fp32

__host__ __device__ constexpr int bm_stage_cols(int nb) { return kBmStageFloats / nb; }
// CTAs per SM the register budget is set for (40 KB of shared memory each);
// 16 columns of B take 128 registers a thread
__host__ __device__ constexpr int bm_resident(int nb) { return nb <= 8 ? 5 : 4; }
// value tiles decoded together (their shared-memory loads in flight); fewer
// for wide B, whose accumulators take the registers
__host__ __device__ constexpr int bm_unroll(int nb) { return nb <= 4 ? 8 : 4; }

// One lane's metadata of the tile it covers in a chunk (zero past the range).
__device__ __forceinline__ void bm_load_meta(const uint64_t* bm_row, const uint32_t* off_row, int64_t k, int64_t k1,
                                             uint64_t& bm, uint32_t& of) {
    bm = 0;
    of = 0;
    if (k < k1) {
        bm = __ldg(bm_row + k);
        of = __ldg(off_row + k);
    }
}

// First value and end (both multiples of 8) of a chunk of cnt >= 1 tiles
// (64-bit: a row block's last tile may end at 2^32).
__device__ __forceinline__ void bm_chunk_span(uint64_t bm, uint32_t of, int cnt, uint64_t& st, uint64_t& en) {
    st = __shfl_sync(0xFFFFFFFFu, of, 0);
    const uint32_t of_l = __shfl_sync(0xFFFFFFFFu, of, cnt - 1);
    const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(bm), cnt - 1);
    const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(bm >> 32), cnt - 1);
    en = static_cast<uint64_t>(of_l) + ((static_cast<uint32_t>(__popc(lo) + __popc(hi)) + 7u) & ~7u);
}

// The chunk's values (a 16-byte aligned run of at most kBmSlot) -> the ring,
// value v at ring[v mod kBmRing] (a 16-byte granule never wraps). Two
// consecutive chunks span at most kBmRing values, so the next chunk's copy
// never lands on the values of the chunk being decoded.
__device__ __forceinline__ void bm_copy_values(const __half* vals, uint64_t st, uint64_t en, __half* ring, int lane) {
    for (uint64_t v = st + 8 * lane; v < en; v += 8 * 32)
        cp_async_16(smem_u32(ring + (v & (kBmRing - 1))), vals + v, 16);
}

// C[64 rows][N] for one row block and one K split; NB columns of B per pass.
// The split is walked in slices of bm_stage_cols(NB) columns whose rows of B
// are staged in shared memory (as fp32) first; each warp takes a contiguous
// quarter of a slice, in chunks of 32 column tiles. Lane j loads tile j's
// bitmap and offset (coalesced) two chunks ahead; a chunk's values, one
// contiguous 16-byte aligned run, are copied into the warp's shared-memory
// ring (cp.async) one chunk ahead, while the chunk before is decoded. Lane l
// owns rows l and l + 32: in a tile their values sit at popc(lo & below) and
// popc(lo) + popc(hi & below) of the tile's packed values (lo, hi the
// bitmap's halves, broadcast by shuffles from the lane that loaded them).
template <int NB>
__global__ void __launch_bounds__(32 * kBmWarps, bm_resident(NB)) bitmap_spmm_kernel(const BmArgs p) {
    __shared__ __align__(16) __half ring[kBmWarps][kBmRing];  // then the warps' partial sums
    __shared__ __align__(16) float bsh[kBmStageFloats];
    static_assert(kBmWarps * kBmRows * NB * sizeof(float) <= sizeof(ring), "partial sums fit the ring");
    constexpr int kStage = bm_stage_cols(NB);
    constexpr int kUnroll = bm_unroll(NB);
    const int64_t i = blockIdx.x / p.splits;
    const int s = static_cast<int>(blockIdx.x % p.splits);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t s0 = s * p.kps, s1 = s0 + p.kps < p.K ? s0 + p.kps : p.K;
    const uint32_t bit = 1u << lane, below = bit - 1u;
    const uint64_t* bm_row = p.bitmaps + i * p.K;
    const uint32_t* off_row = p.offsets + i * p.K;
    const __half* vals = p.values + p.bases[i];
    for (int64_t n0 = 0; n0 < p.N; n0 += NB) {
        float acc0[NB], acc1[NB];  // rows l and l + 32
#pragma unroll
        for (int n = 0; n < NB; ++n) acc0[n] = acc1[n] = 0.f;
        for (int64_t ks = s0; ks < s1; ks += kStage) {
            const int64_t ke = ks + kStage < s1 ? ks + kStage : s1;
            // this warp's quarter of the slice, its first two chunks' metadata
            const int64_t qn = (ke - ks + kBmWarps - 1) / kBmWarps;
            const int64_t k0 = ks + warp * qn < ke ? ks + warp * qn : ke;
            const int64_t k1 = k0 + qn < ke ? k0 + qn : ke;
            const int nchunks = static_cast<int>((k1 - k0 + kBmChunk - 1) / kBmChunk);
            uint64_t bm_c, bm_n;
            uint32_t of_c, of_n;
            bm_load_meta(bm_row, off_row, k0 + lane, k1, bm_c, of_c);
            bm_load_meta(bm_row, off_row, k0 + kBmChunk + lane, k1, bm_n, of_n);
            // B[ks .. ke)[n0 .. n0 + NB) -> shared memory (zeros past N); the previous slice's reads are done
            __syncthreads();
            for (int64_t e = threadIdx.x; e < (ke - ks) * NB; e += blockDim.x) {
                const int64_t kk = e / NB;
                const int n = static_cast<int>(e - kk * NB);
                bsh[e] = n0 + n < p.N ? __half2float(p.B[(ks + kk) * p.ld_b + n0 + n]) : 0.f;
            }
            if (nchunks > 0) {
                uint64_t st, en;
                bm_chunk_span(bm_c, of_c, static_cast<int>(k1 - k0 < kBmChunk ? k1 - k0 : kBmChunk), st, en);
                bm_copy_values(vals, st, en, ring[warp], lane);
            }
            cp_async_commit();
            __syncthreads();
            for (int c = 0; c < nchunks; ++c) {
                const int64_t kc = k0 + static_cast<int64_t>(c) * kBmChunk;
                const int cnt = static_cast<int>(k1 - kc < kBmChunk ? k1 - kc : kBmChunk);
                // metadata two chunks ahead; the next chunk's values into the other slot
                uint64_t bm_n2;
                uint32_t of_n2;
                bm_load_meta(bm_row, off_row, kc + 2 * kBmChunk + lane, k1, bm_n2, of_n2);
                if (c + 1 < nchunks) {
                    const int64_t cnt_n = k1 - kc - kBmChunk;
                    uint64_t st, en;
                    bm_chunk_span(bm_n, of_n, static_cast<int>(cnt_n < kBmChunk ? cnt_n : kBmChunk), st, en);
                    bm_copy_values(vals, st, en, ring[warp], lane);
                }
                cp_async_commit();
                cp_async_wait<1>();  // this chunk's copies (this lane's)
                __syncwarp();            // ... and every lane's
                const __half* rw = ring[warp];
#pragma unroll
                for (int u0 = 0; u0 < kBmChunk; u0 += kUnroll) {
                    if (u0 >= cnt) break;
                    float a0[kUnroll], a1[kUnroll];
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        // tiles past the range have a zero bitmap (nothing read)
                        const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(bm_c), u0 + u);
                        const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(bm_c >> 32), u0 + u);
                        const uint32_t of = __shfl_sync(0xFFFFFFFFu, of_c, u0 + u);
                        const uint32_t p0 = (of + __popc(lo & below)) & (kBmRing - 1);
                        const uint32_t p1 = (of + __popc(lo) + __popc(hi & below)) & (kBmRing - 1);
                        a0[u] = (lo & bit) ? __half2float(rw[p0]) : 0.f;
                        a1[u] = (hi & bit) ? __half2float(rw[p1]) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        if (u0 + u >= cnt) break;
                        const float* b = bsh + (kc + u0 + u - ks) * NB;
#pragma unroll
                        for (int n = 0; n < NB; ++n) {
                            const float bv = b[n];
                            acc0[n] = fmaf(a0[u], bv, acc0[n]);
                            acc1[n] = fmaf(a1[u], bv, acc1[n]);
                        }
                    }
                }
                __syncwarp();  // this chunk is read before the chunk after next is copied over it
                bm_c = bm_n;
                of_c = of_n;
                bm_n = bm_n2;
                of_n = of_n2;
            }
        }
        // the warps' sums, in warp order (the ring's space, every copy landed and read)
        cp_async_wait_all();
        __syncthreads();
        float* red = reinterpret_cast<float*>(&ring[0][0]);
#pragma unroll
        for (int n = 0; n < NB; ++n) {
            red[(warp * NB + n) * kBmRows + lane] = acc0[n];
            red[(warp * NB + n) * kBmRows + 32 + lane] = acc1[n];
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kBmRows * NB; e += blockDim.x) {
            const int n = e / kBmRows, rr = e % kBmRows;
            if (n0 + n >= p.N) continue;
            float v = red[n * kBmRows + rr];
#pragma unroll
            for (int w = 1; w < kBmWarps; ++w) v += red[(w * NB + n) * kBmRows + rr];
            const int64_t row = i * kBmRows + rr;
            if (p.partial != nullptr)
                p.partial[(static_cast<int64_t>(s) * p.R + row) * p.N + n0 + n] = v;
            else
                out_store(p.out, row, n0 + n, v);
        }
        __syncthreads();  // the partial sums are read before the ring is reused
    }
}

}  // namespace

cudaError_t launch_bitmap_encode_counts(const void* W, int64_t ld_w, int64_t R, int64_t K, void* bitmaps,
                                        void* offsets, int64_t* bases, cudaStream_t stream) {
    const int64_t blocks = R / kBmRows;
    if (blocks == 0 || K == 0) return cudaMemsetAsync(bases, 0, sizeof(int64_t) * (blocks + 1), stream);
    const dim3 grid(static_cast<unsigned>((K + 255) / 256), static_cast<unsigned>(blocks));
    bitmap_count_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(W), ld_w, K,
                                                  static_cast<uint64_t*>(bitmaps), static_cast<uint32_t*>(offsets));
    bitmap_scan_kernel<<<static_cast<unsigned>(blocks), kBmScanThreads, 0, stream>>>(static_cast<uint32_t*>(offsets),
                                                                                   K, bases);
    bitmap_bases_kernel<<<1, kBmScanThreads, 0, stream>>>(bases, blocks);
    return cudaGetLastError();
}

cudaError_t launch_bitmap_encode_fill(const void* W, int64_t ld_w, int64_t R, int64_t K, const void* bitmaps,
                                      const void* offsets, const int64_t* bases, void* values, cudaStream_t stream) {
    const int64_t blocks = R / kBmRows;
    if (blocks == 0 || K == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((K + 255) / 256), static_cast<unsigned>(blocks));
    bitmap_fill_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(W), ld_w, K,
                                                 static_cast<const uint64_t*>(bitmaps),
                                                 static_cast<const uint32_t*>(offsets), bases,
                                                 static_cast<uint16_t*>(values));
    return cudaGetLastError();
}

int bitmap_spmm_splits(int64_t R, int64_t K, int64_t N, int sm_count) {
    // at most the CTAs that are resident at once, each split at least 256
    // columns
    const int64_t blocks = std::max<int64_t>(1, R / kBmRows);
    int64_t s = bm_resident(N <= 8 ? 8 : 16) * static_cast<int64_t>(sm_count) / blocks;
    s = std::min<int64_t>(s, std::max<int64_t>(1, K / 256));
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(s, 64)));
}

cudaError_t launch_bitmap_spmm(int64_t R, int64_t K, const void* bitmaps, const void* offsets, const int64_t* bases,
                               const void* values, const void* B, int64_t ld_b, int64_t N, const OutSpec& out,
                               int splits, float* partial, cudaStream_t stream) {
    BmArgs p;
    p.bitmaps = static_cast<const uint64_t*>(bitmaps);
    p.offsets = static_cast<const uint32_t*>(offsets);
    p.bases = bases;
    p.values = static_cast<const __half*>(values);
    p.B = static_cast<const __half*>(B);
    p.ld_b = ld_b;
    p.R = R;
    p.K = K;
    p.N = N;
    p.splits = std::max(1, splits);
    p.kps = (K + p.splits - 1) / p.splits;
    p.out = out;
    p.partial = p.splits > 1 ? partial : nullptr;
    if (p.splits > 1 && partial == nullptr) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>((R / kBmRows) * p.splits);
    if (grid == 0 || N == 0) return cudaSuccess;
    if (N <= 1)
        bitmap_spmm_kernel<1><<<grid, 32 * kBmWarps, 0, stream>>>(p);
    else if (N <= 2)
        bitmap_spmm_kernel<2><<<grid, 32 * kBmWarps, 0, stream>>>(p);
    else if (N <= 4)
        bitmap_spmm_kernel<4><<<grid, 32 * kBmWarps, 0, stream>>>(p);
    else if (N <= 8)
        bitmap_spmm_kernel<8><<<grid, 32 * kBmWarps, 0, stream>>>(p);
    else
        bitmap_spmm_kernel<16><<<grid, 32 * kBmWarps, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.splits == 1) return e;
    return launch_splitk_reduce(partial, p.splits, R, N, out, stream);
}

}  // namespace vnm
