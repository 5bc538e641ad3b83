// CUDA-core V:N:M SpMM for small N (decode-like products, where the weight
// bytes dominate), and the split-K reduction used by the tensor-core path.
//
// VENOM section 4, Figure 4: each stored value of row r in block j meets the
// row j*M + colidx[r/V][j][slot] of B; the 2-bit m-index picks the slot
// among the block's 4 kept columns (lecture notes "2:4 sparsity on sparse
// tensor cores": the tags act on the activations, selecting K/2 of K).
// One warp owns one row of A: lanes stream the row's values, m-indices and
// the block-row's column-loc with coalesced loads, gather the matching B
// rows (small, cache-resident), accumulate in fp32 and reduce across lanes.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "vnm_internal.h"
#include "vnm_ptx.cuh"

namespace vnm {
namespace {

constexpr int kSimtWarps = 8;

struct SimtArgs {
    const uint32_t* values;  // [R][nblk] words: the 2 fp16 values of one block
    const uint8_t* meta;     // [R][mpitch]
    const uint32_t* colidx;  // [R/V][nblk] words: 4 column bytes
    const __half* B;
    int64_t bk, bn;          // B element (k, n) at B + k * bk + n * bn
    OutSpec out;
    int64_t R, N;
    int V, M;
    int64_t nblk, mpitch;
};

template <int NB>
__device__ __forceinline__ void accumulate_block(const SimtArgs& p, int64_t row, int64_t j, int64_t n0,
                                                 uint32_t vv, uint32_t code, uint32_t sel, float (&acc)[NB]) {
    const int64_t k0 = j * p.M + ((sel >> (8u * (code & 3u))) & 0xFFu);
    const int64_t k1 = j * p.M + ((sel >> (8u * (code >> 2))) & 0xFFu);
    const float a0 = __half2float(__ushort_as_half(static_cast<unsigned short>(vv & 0xFFFFu)));
    const float a1 = __half2float(__ushort_as_half(static_cast<unsigned short>(vv >> 16)));
    const __half* b0 = p.B + k0 * p.bk + n0 * p.bn;
    const __half* b1 = p.B + k1 * p.bk + n0 * p.bn;
#pragma unroll
    for (int q = 0; q < NB; ++q) {
        if (n0 + q < p.N) {
            acc[q] = fmaf(a0, __half2float(b0[q * p.bn]), acc[q]);
            acc[q] = fmaf(a1, __half2float(b1[q * p.bn]), acc[q]);
        }
    }
}

template <int NB>
__global__ void __launch_bounds__(32 * kSimtWarps) spmm_simt_kernel(const SimtArgs p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kSimtWarps + warp;
    if (row >= p.R) return;
    const uint32_t* vrow = p.values + row * p.nblk;
    const uint8_t* mrow = p.meta + row * p.mpitch;
    const uint32_t* crow = p.colidx + (row / p.V) * p.nblk;
    for (int64_t n0 = 0; n0 < p.N; n0 += NB) {
        float acc[NB];
#pragma unroll
        for (int q = 0; q < NB; ++q) acc[q] = 0.f;
        int64_t j = lane;
        // four blocks per lane in flight
        for (; j + 96 < p.nblk; j += 128) {
            uint32_t vv[4], mb[4], sel[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t jj = j + 32 * u;
                vv[u] = __ldg(vrow + jj);
                mb[u] = __ldg(mrow + (jj >> 1));
                sel[u] = __ldg(crow + jj);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t jj = j + 32 * u;
                accumulate_block<NB>(p, row, jj, n0, vv[u], (mb[u] >> (4 * (jj & 1))) & 0xFu, sel[u], acc);
            }
        }
        for (; j < p.nblk; j += 32) {
            const uint32_t vv = __ldg(vrow + j);
            const uint32_t code = (__ldg(mrow + (j >> 1)) >> (4 * (j & 1))) & 0xFu;
            accumulate_block<NB>(p, row, j, n0, vv, code, __ldg(crow + j), acc);
        }
#pragma unroll
        for (int q = 0; q < NB; ++q) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[q] += __shfl_xor_sync(0xFFFFFFFFu, acc[q], off);
        }
        if (lane < NB && n0 + lane < p.N) {
            float v = acc[0];
#pragma unroll
            for (int q = 1; q < NB; ++q)
                if (lane == q) v = acc[q];
            out_store(p.out, row, n0 + lane, v);
        }
    }
}

// C[r][n] = sum over s = 0 .. splits-1 (in order) of partial[s][r][n].
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, int splits, int64_t R, int64_t N,
                                     const OutSpec out) {
    const int64_t total = R * N;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < total;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // a transposed C: consecutive threads take consecutive rows of one column
        const int64_t r = out.ns == 1 ? q / N : q % R, n = out.ns == 1 ? q % N : q / R;
        const int64_t e = r * N + n;
        float s = 0.f;
        for (int z = 0; z < splits; ++z) s += __ldg(partial + z * total + e);
        out_store(out, r, n, s);
    }
}

// ---------------------------------------------------------------------------
// Streaming path for N <= 8 (decode-like): one CTA per (V-block row, K split).
// The rows of a V-block row share column-loc, so per chunk of 32*U blocks
// the CTA first stages the 4 selected rows of B of every block (N <= 8
// values each) in shared memory; each of the 16 warps owns RW rows and
// issues all its loads of the chunk at once (lane = block, RW*U = 16 loads
// per lane), so a chunk costs one round trip to memory; the multiply-adds
// then read B from shared memory. With K split over s CTAs (s = 2, 4 or 8),
// the s CTAs of a V-block row form a thread-block cluster: each leaves its
// fp32 partial sums in its shared memory, and after a cluster barrier CTA q
// sums rows q, q + s, ... over the cluster in split order (distributed
// shared memory), so C is written once by one kernel, deterministically.
constexpr int kStreamWarps = 16;

struct StreamArgs {
    const uint32_t* values;  // [R][nblk] words: the 2 fp16 values of one block
    const uint8_t* meta;     // [R][mpitch]
    const uint32_t* colidx;  // [R/V][nblk] words: 4 column bytes
    const __half* B;
    int64_t bk, bn;          // B element (k, n) at B + k * bk + n * bn
    OutSpec out;
    int64_t R, N;
    int V, M;
    int64_t nblk, mpitch;
    int splits;
    int64_t bps;             // blocks per split
};

// acc + (float)a * (float)b for the fp16 a, b in the low 16 bits (exact
// products, one rounding: the same value as converting then fmaf).
__device__ __forceinline__ float fma_f16(uint32_t a, uint32_t b, float acc) {
    const unsigned short ha = static_cast<unsigned short>(a & 0xFFFFu), hb = static_cast<unsigned short>(b & 0xFFFFu);
    asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(ha), "h"(hb));
    return acc;
}

// The streaming kernel for row-major B and C without bias or activation
// (vnm_spmm). Its strided form below serves the Linear-layer form.
struct StreamArgsRM {  // the row-major, plain form (vnm_spmm)
    const uint32_t* values;  // [R][nblk] words: the 2 fp16 values of one block
    const uint8_t* meta;     // [R][mpitch]
    const uint32_t* colidx;  // [R/V][nblk] words: 4 column bytes
    const __half* B;
    int64_t ld_b;
    void* C;
    int64_t ld_c;
    int64_t R, N;
    int V, M;
    int64_t nblk, mpitch;
    int splits;
    int64_t bps;             // blocks per split
    bool c_f32;
};

template <int NB, int RW, int U>
__global__ void __launch_bounds__(32 * kStreamWarps) spmm_stream_rm_kernel(const StreamArgsRM p) {
    constexpr int kChunk = 32 * U;                       // blocks per chunk
    // staged block: [NB columns][4 slots] halves (a column's 4 slots in 8
    // bytes), padded for NB >= 4 to spread the banks
    constexpr int kStride = 4 * NB + (NB >= 4 ? 4 : 0);
    __shared__ __align__(16) __half Bc[kChunk * kStride];
    __shared__ float red[kStreamWarps * RW][NB];  // this CTA's sums of the pass's rows (split K)
    const int64_t i = blockIdx.x / p.splits;
    const int s = static_cast<int>(blockIdx.x % p.splits);
    const int64_t jb = s * p.bps;
    const int64_t je = jb + p.bps < p.nblk ? jb + p.bps : p.nblk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t* crow = p.colidx + i * p.nblk;

    // the same trip count for every warp (the loop holds CTA barriers); rows
    // past V are masked
    for (int rbase = 0; rbase < p.V; rbase += kStreamWarps * RW) {
        const int r0 = rbase + warp;
        float acc[RW][NB];
#pragma unroll
        for (int t = 0; t < RW; ++t)
#pragma unroll
            for (int n = 0; n < NB; ++n) acc[t][n] = 0.f;
        for (int64_t j0 = jb; j0 < je; j0 += kChunk) {
            // this warp's rows of the chunk: all loads in flight at once
            uint32_t vv[RW][U], mb[RW][U];
#pragma unroll
            for (int t = 0; t < RW; ++t) {
                const int r = r0 + kStreamWarps * t;
                const int64_t row = i * p.V + r;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t jj = j0 + lane + 32 * u;
                    vv[t][u] = 0u;
                    mb[t][u] = 0u;
                    if (r < p.V && jj < je) {
                        vv[t][u] = __ldg(p.values + row * p.nblk + jj);
                        mb[t][u] = __ldg(p.meta + row * p.mpitch + (jj >> 1));
                    }
                }
            }
            // stage the chunk's selected rows of B (the previous chunk's reads are done)
            __syncthreads();
            const int nb = static_cast<int>(je - j0 < kChunk ? je - j0 : kChunk);
            for (int q = threadIdx.x; q < nb * 4; q += blockDim.x) {
                const int jl = q >> 2, slot = q & 3;
                const uint32_t w = __ldg(crow + j0 + jl);
                // column-loc byte, clamped so that a corrupt array cannot address past K
                const uint32_t cb = min((w >> (8 * slot)) & 0xFFu, static_cast<uint32_t>(p.M - 1));
                const __half* src = p.B + ((j0 + jl) * p.M + cb) * p.ld_b;
                __half* dst = Bc + jl * kStride + slot;
#pragma unroll
                for (int n = 0; n < NB; ++n) dst[4 * n] = n < p.N ? src[n] : __float2half_rn(0.f);
            }
            __syncthreads();
#pragma unroll
            for (int t = 0; t < RW; ++t) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t jj = j0 + lane + 32 * u;
                    if (jj >= je) continue;
                    const uint32_t code = (mb[t][u] >> (4 * (jj & 1))) & 0xFu;
                    // byte-permute selector of slots s0 = code & 3 (low half) and s1 = code >> 2
                    const uint32_t sel = ((code & 3u) * 0x22u + 0x10u) | (((code >> 2) * 0x22u + 0x10u) << 8);
                    const uint32_t a = vv[t][u];
                    const uint2* b = reinterpret_cast<const uint2*>(Bc + (lane + 32 * u) * kStride);
#pragma unroll
                    for (int n = 0; n < NB; ++n) {
                        const uint2 w = b[n];  // the 4 slots of column n
                        const uint32_t pr = __byte_perm(w.x, w.y, sel);
                        acc[t][n] = fma_f16(a, pr, acc[t][n]);
                        acc[t][n] = fma_f16(a >> 16, pr >> 16, acc[t][n]);
                    }
                }
            }
        }
        auto store = [&](int r, int n, float v) {
            const int64_t row = i * p.V + r;
            if (p.c_f32)
                static_cast<float*>(p.C)[row * p.ld_c + n] = v;
            else
                static_cast<__half*>(p.C)[row * p.ld_c + n] = __float2half_rn(v);
        };
#pragma unroll
        for (int t = 0; t < RW; ++t) {
            const int r = r0 + kStreamWarps * t;
            float out = 0.f;
#pragma unroll
            for (int n = 0; n < NB; ++n) {
                float v = acc[t][n];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
                if (lane == n) out = v;
            }
            if (p.splits > 1) {
                if (lane < NB) red[warp + kStreamWarps * t][lane] = out;
            } else if (r < p.V && lane < p.N && lane < NB) {
                store(r, lane, out);
            }
        }
        if (p.splits > 1) {
            // every CTA of the cluster holds its partial sums of the pass's rows
            cluster_sync_all();
            const uint32_t red0 = smem_u32(&red[0][0]);
            for (int e = threadIdx.x; e < kStreamWarps * RW * NB; e += blockDim.x) {
                const int l = e / NB, n = e % NB;  // row of the pass (warp + 16 t), column
                const int r = rbase + l;
                if (l % p.splits != s || r >= p.V || n >= p.N) continue;
                float v = 0.f;
                for (int q = 0; q < p.splits; ++q)
                    v += dsmem_ld_f32(dsmem_map(red0 + static_cast<uint32_t>(e) * 4u, static_cast<uint32_t>(q)));
                store(r, n, v);
            }
            // no CTA reuses or leaves its partial sums while another may still read them
            cluster_sync_all();
        }
    }
}

// The strided form: B element (k, n) at B + k * bk + n * bn, C written
// through an OutSpec (PLAIN: row-major B and C, no bias or activation).
template <int NB, int RW, int U, bool PLAIN>
__global__ void __launch_bounds__(32 * kStreamWarps) spmm_stream_kernel(const StreamArgs p) {
    constexpr int kChunk = 32 * U;                       // blocks per chunk
    // staged block: [NB columns][4 slots] halves (a column's 4 slots in 8
    // bytes), padded for NB >= 4 to spread the banks
    constexpr int kStride = 4 * NB + (NB >= 4 ? 4 : 0);
    __shared__ __align__(16) __half Bc[kChunk * kStride];
    __shared__ float red[kStreamWarps * RW][NB];  // this CTA's sums of the pass's rows (split K)
    const int64_t i = blockIdx.x / p.splits;
    const int s = static_cast<int>(blockIdx.x % p.splits);
    const int64_t jb = s * p.bps;
    const int64_t je = jb + p.bps < p.nblk ? jb + p.bps : p.nblk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t* crow = p.colidx + i * p.nblk;

    // the same trip count for every warp (the loop holds CTA barriers); rows
    // past V are masked
    for (int rbase = 0; rbase < p.V; rbase += kStreamWarps * RW) {
        const int r0 = rbase + warp;
        float acc[RW][NB];
#pragma unroll
        for (int t = 0; t < RW; ++t)
#pragma unroll
            for (int n = 0; n < NB; ++n) acc[t][n] = 0.f;
        for (int64_t j0 = jb; j0 < je; j0 += kChunk) {
            // this warp's rows of the chunk: all loads in flight at once
            uint32_t vv[RW][U], mb[RW][U];
#pragma unroll
            for (int t = 0; t < RW; ++t) {
                const int r = r0 + kStreamWarps * t;
                const int64_t row = i * p.V + r;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t jj = j0 + lane + 32 * u;
                    vv[t][u] = 0u;
                    mb[t][u] = 0u;
                    if (r < p.V && jj < je) {
                        vv[t][u] = __ldg(p.values + row * p.nblk + jj);
                        mb[t][u] = __ldg(p.meta + row * p.mpitch + (jj >> 1));
                    }
                }
            }
            // stage the chunk's selected rows of B (the previous chunk's reads are done)
            __syncthreads();
            const int nb = static_cast<int>(je - j0 < kChunk ? je - j0 : kChunk);
            for (int q = threadIdx.x; q < nb * 4; q += blockDim.x) {
                const int jl = q >> 2, slot = q & 3;
                const uint32_t w = __ldg(crow + j0 + jl);
                // column-loc byte, clamped so that a corrupt array cannot address past K
                const uint32_t cb = min((w >> (8 * slot)) & 0xFFu, static_cast<uint32_t>(p.M - 1));
                const __half* src = p.B + ((j0 + jl) * p.M + cb) * p.bk;
                __half* dst = Bc + jl * kStride + slot;
#pragma unroll
                for (int n = 0; n < NB; ++n) dst[4 * n] = n < p.N ? src[PLAIN ? n : n * p.bn] : __float2half_rn(0.f);
            }
            __syncthreads();
#pragma unroll
            for (int t = 0; t < RW; ++t) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t jj = j0 + lane + 32 * u;
                    if (jj >= je) continue;
                    const uint32_t code = (mb[t][u] >> (4 * (jj & 1))) & 0xFu;
                    // byte-permute selector of slots s0 = code & 3 (low half) and s1 = code >> 2
                    const uint32_t sel = ((code & 3u) * 0x22u + 0x10u) | (((code >> 2) * 0x22u + 0x10u) << 8);
                    const uint32_t a = vv[t][u];
                    const uint2* b = reinterpret_cast<const uint2*>(Bc + (lane + 32 * u) * kStride);
#pragma unroll
                    for (int n = 0; n < NB; ++n) {
                        const uint2 w = b[n];  // the 4 slots of column n
                        const uint32_t pr = __byte_perm(w.x, w.y, sel);
                        acc[t][n] = fma_f16(a, pr, acc[t][n]);
                        acc[t][n] = fma_f16(a >> 16, pr >> 16, acc[t][n]);
                    }
                }
            }
        }
        auto store = [&](int r, int n, float v) {
            const int64_t row = i * p.V + r;
            if (!PLAIN)
                out_store(p.out, row, n, v);
            else if (p.out.f32)
                static_cast<float*>(p.out.C)[row * p.out.rs + n] = v;
            else
                static_cast<__half*>(p.out.C)[row * p.out.rs + n] = __float2half_rn(v);
        };
#pragma unroll
        for (int t = 0; t < RW; ++t) {
            const int r = r0 + kStreamWarps * t;
            float out = 0.f;
#pragma unroll
            for (int n = 0; n < NB; ++n) {
                float v = acc[t][n];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
                if (lane == n) out = v;
            }
            if (p.splits > 1) {
                if (lane < NB) red[warp + kStreamWarps * t][lane] = out;
            } else if (r < p.V && lane < p.N && lane < NB) {
                store(r, lane, out);
            }
        }
        if (p.splits > 1) {
            // every CTA of the cluster holds its partial sums of the pass's rows
            cluster_sync_all();
            const uint32_t red0 = smem_u32(&red[0][0]);
            for (int e = threadIdx.x; e < kStreamWarps * RW * NB; e += blockDim.x) {
                const int l = e / NB, n = e % NB;  // row of the pass (warp + 16 t), column
                const int r = rbase + l;
                if (l % p.splits != s || r >= p.V || n >= p.N) continue;
                float v = 0.f;
                for (int q = 0; q < p.splits; ++q)
                    v += dsmem_ld_f32(dsmem_map(red0 + static_cast<uint32_t>(e) * 4u, static_cast<uint32_t>(q)));
                store(r, n, v);
            }
            // no CTA reuses or leaves its partial sums while another may still read them
            cluster_sync_all();
        }
    }
}

template <int NB, int RW, int U, bool PLAIN>
cudaError_t launch_stream4(const StreamArgs& p, cudaStream_t stream) {
    const int64_t ctas = (p.R / p.V) * p.splits;
    if (p.splits == 1) {
        spmm_stream_kernel<NB, RW, U, PLAIN><<<static_cast<unsigned>(ctas), 32 * kStreamWarps, 0, stream>>>(p);
        return cudaGetLastError();
    }
    // the splits of a V-block row are consecutive CTAs: one cluster
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(32 * kStreamWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, spmm_stream_kernel<NB, RW, U, PLAIN>, p);
}

// ---------------------------------------------------------------------------
// Pipelined streaming path (row-major B and C, N <= 8, V a multiple of 64,
// K/M a multiple of 32): the same CTA work as above, 64 rows a pass, but
// each warp owns 8 consecutive rows and streams them on its own: a chunk is
// 32 blocks (lane = block), and the warp's values, m-indices and the
// V-block row's column-loc words of a chunk (16-byte aligned runs) are
// copied into the warp's ring of kPipeStages shared-memory stages with
// cp.async, up to kPipeStages - 1 chunks ahead of the one being multiplied.
// The CTA's rows of B (its K range, at most kPipeBHalves values) are loaded
// into shared memory once; each lane gathers its own block's 4 selected rows
// of B from there. No CTA barrier sits in the chunk loop: a warp waits only
// for its own copies.
constexpr int kPipeWarps = 8;
constexpr int kPipeRows = 64;         // rows per pass: 8 warps x 8
constexpr int kPipeWarpRows = kPipeRows / kPipeWarps;
constexpr int kPipeChunk = 32;        // blocks per chunk
constexpr int kPipeStages = 4;        // 40 KB for the CTA: three chunks in flight per warp
constexpr int kPipeBHalves = 12288;   // 24 KB: the CTA's rows of B
// CTAs per SM the registers are budgeted for (shared memory allows three);
// eight columns of B keep 64 accumulators a thread
__host__ __device__ constexpr int pipe_resident(int nb) { return nb <= 4 ? 3 : 2; }
constexpr int kPipeMaxDevices = 64;

struct PipeStage {  // one warp's chunk
    uint32_t vals[kPipeWarpRows][kPipeChunk];     // 1 KB: the rows' value words
    uint8_t meta[kPipeWarpRows][kPipeChunk / 2];  // their m-index bytes
    uint32_t col[kPipeChunk];                     // the V-block row's column-loc words
};

template <int NB>
__global__ void __launch_bounds__(32 * kPipeWarps, pipe_resident(NB)) spmm_stream_pipe_kernel(const StreamArgsRM p) {
    static_assert(kPipeWarpRows * kPipeWarps == kPipeRows && kPipeStages >= 2, "pipeline shape");
    extern __shared__ __align__(16) uint8_t pipe_smem[];
    __half* Bs = reinterpret_cast<__half*>(pipe_smem);  // [K range][NB]
    __shared__ float red[kPipeRows][NB];
    const int64_t i = blockIdx.x / p.splits;
    const int s = static_cast<int>(blockIdx.x % p.splits);
    const int64_t jb = s * p.bps < p.nblk ? s * p.bps : p.nblk;
    const int64_t je = jb + p.bps < p.nblk ? jb + p.bps : p.nblk;
    const int nch = static_cast<int>((je - jb) / kPipeChunk);  // split bounds are multiples of 32 blocks
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    PipeStage* ring = reinterpret_cast<PipeStage*>(pipe_smem + kPipeBHalves * sizeof(__half)) + warp * kPipeStages;
    const uint32_t* crow = p.colidx + i * p.nblk;

    // the CTA's rows of B (zeros past N), once for every pass
    const int64_t kcols = (je - jb) * p.M;
    for (int64_t e = tid; e < kcols * NB; e += blockDim.x) {
        const int64_t k = e / NB;
        const int n = static_cast<int>(e - k * NB);
        Bs[e] = n < p.N ? p.B[(jb * p.M + k) * p.ld_b + n] : __float2half_rn(0.f);
    }
    __syncthreads();

    for (int rbase = 0; rbase < p.V; rbase += kPipeRows) {
        const int64_t row0 = i * p.V + rbase + kPipeWarpRows * warp;  // this warp's first row
        // chunk c -> stage c % kPipeStages of this warp: values (8 granules a row),
        // m-indices (1 a row), column-loc (8)
        auto issue = [&](int c) {
            PipeStage& g = ring[c % kPipeStages];
            const int64_t j0 = jb + static_cast<int64_t>(c) * kPipeChunk;
#pragma unroll
            for (int h = 0; h < kPipeWarpRows * 8 / 32; ++h) {
                const int x = lane + 32 * h, r = x >> 3, q = x & 7;
                cp_async_16(smem_u32(&g.vals[r][4 * q]), p.values + (row0 + r) * p.nblk + j0 + 4 * q, 16);
            }
            if (lane < kPipeWarpRows)
                cp_async_16(smem_u32(&g.meta[lane][0]), p.meta + (row0 + lane) * p.mpitch + j0 / 2, 16);
            else if (lane < kPipeWarpRows + 8)
                cp_async_16(smem_u32(&g.col[4 * (lane - kPipeWarpRows)]), crow + j0 + 4 * (lane - kPipeWarpRows), 16);
        };

        float acc[kPipeWarpRows][NB];
#pragma unroll
        for (int t = 0; t < kPipeWarpRows; ++t)
#pragma unroll
            for (int n = 0; n < NB; ++n) acc[t][n] = 0.f;
#pragma unroll
        for (int c = 0; c < kPipeStages - 1; ++c) {
            if (c < nch) issue(c);
            cp_async_commit();
        }
        for (int c = 0; c < nch; ++c) {
            cp_async_wait<kPipeStages - 2>();  // chunk c (this lane's copies)
            __syncwarp();                      // ... every lane's; chunk c - 1 read by every lane
            if (c + kPipeStages - 1 < nch) issue(c + kPipeStages - 1);  // over chunk c - 1's stage
            cp_async_commit();
            const PipeStage& g = ring[c % kPipeStages];
            // this lane's block: its 4 selected rows of B, column n's 4 slots as one uint2
            const uint32_t w = g.col[lane];
            const int64_t kb = (static_cast<int64_t>(c) * kPipeChunk + lane) * p.M;  // in the CTA's K range
            uint2 bq[NB];
            {
                uint32_t h[4][NB];
#pragma unroll
                for (int slot = 0; slot < 4; ++slot) {
                    // column-loc byte, clamped so that a corrupt array cannot address past K
                    const uint32_t cb = min((w >> (8 * slot)) & 0xFFu, static_cast<uint32_t>(p.M - 1));
                    const __half* src = Bs + (kb + cb) * NB;
#pragma unroll
                    for (int n = 0; n < NB; ++n) h[slot][n] = __half_as_ushort(src[n]);
                }
#pragma unroll
                for (int n = 0; n < NB; ++n)
                    bq[n] = make_uint2(h[0][n] | (h[1][n] << 16), h[2][n] | (h[3][n] << 16));
            }
#pragma unroll
            for (int t = 0; t < kPipeWarpRows; ++t) {
                const uint32_t a = g.vals[t][lane];
                // this block's 4 bits: slots s0 (bits 0-1, low half) and s1 (bits 2-3)
                const uint32_t code = static_cast<uint32_t>(g.meta[t][lane >> 1]) >> (4 * (lane & 1));
                // byte-permute selector of the two slots' halves: byte s of 0x76543210 is the
                // selector pair (2s, 2s + 1), picked for s0 and s1 by a byte permute of its own
                const uint32_t sel = __byte_perm(0x76543210u, 0u, (code & 3u) | ((code & 0xCu) << 2));
#pragma unroll
                for (int n = 0; n < NB; ++n) {
                    const uint32_t pr = __byte_perm(bq[n].x, bq[n].y, sel);
                    acc[t][n] = fma_f16(a, pr, acc[t][n]);
                    acc[t][n] = fma_f16(a >> 16, pr >> 16, acc[t][n]);
                }
            }
        }
        cp_async_wait_all();
        __syncwarp();  // the warp's ring is free for the next pass

        auto store = [&](int r, int n, float v) {  // r: row of the pass
            const int64_t row = i * p.V + rbase + r;
            if (p.c_f32)
                static_cast<float*>(p.C)[row * p.ld_c + n] = v;
            else
                static_cast<__half*>(p.C)[row * p.ld_c + n] = __float2half_rn(v);
        };
#pragma unroll
        for (int t = 0; t < kPipeWarpRows; ++t) {
            const int r = kPipeWarpRows * warp + t;
            float out = 0.f;
#pragma unroll
            for (int n = 0; n < NB; ++n) {
                float v = acc[t][n];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
                if (lane == n) out = v;
            }
            if (p.splits > 1) {
                if (lane < NB) red[r][lane] = out;
            } else if (lane < p.N && lane < NB) {
                store(r, lane, out);
            }
        }
        if (p.splits > 1) {
            // every CTA of the cluster holds its partial sums of the pass's rows
            cluster_sync_all();
            const uint32_t red0 = smem_u32(&red[0][0]);
            for (int e = tid; e < kPipeRows * NB; e += blockDim.x) {
                const int r = e / NB, n = e % NB;
                if (r % p.splits != s || n >= p.N) continue;
                float v = 0.f;
                for (int q = 0; q < p.splits; ++q)
                    v += dsmem_ld_f32(dsmem_map(red0 + static_cast<uint32_t>(e) * 4u, static_cast<uint32_t>(q)));
                store(r, n, v);
            }
            // no CTA reuses or leaves its partial sums while another may still read them
            cluster_sync_all();
        }
    }
}

// Blocks of a split of the pipelined kernel: on chunk bounds (a split may
// be empty: its CTA adds zeros).
inline int64_t pipe_split_blocks(int64_t nblk, int splits) {
    const int64_t per = (nblk + splits - 1) / splits;
    return (per + kPipeChunk - 1) / kPipeChunk * kPipeChunk;
}

inline bool pipe_aligned(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }

inline int pipe_nb(int64_t N) { return N <= 1 ? 1 : N <= 2 ? 2 : N <= 4 ? 4 : 8; }

template <int NB>
cudaError_t launch_stream_pipe(const StreamArgsRM& q, cudaStream_t stream) {
    StreamArgsRM p = q;
    p.bps = pipe_split_blocks(p.nblk, p.splits);
    const int64_t ctas = (p.R / p.V) * p.splits;
    constexpr size_t smem = kPipeBHalves * sizeof(__half) + sizeof(PipeStage) * kPipeStages * kPipeWarps;
    // the shared-memory opt-in, once per device
    static std::atomic<bool> attr_set[kPipeMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kPipeMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(spmm_stream_pipe_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    if (p.splits == 1) {
        spmm_stream_pipe_kernel<NB><<<static_cast<unsigned>(ctas), 32 * kPipeWarps, smem, stream>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(32 * kPipeWarps);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, spmm_stream_pipe_kernel<NB>, p);
}

template <int NB, int RW, int U>
cudaError_t launch_stream_rm(const StreamArgs& q, cudaStream_t stream) {
    StreamArgsRM p;
    p.values = q.values;
    p.meta = q.meta;
    p.colidx = q.colidx;
    p.B = q.B;
    p.ld_b = q.bk;
    p.C = q.out.C;
    p.ld_c = q.out.rs;
    p.R = q.R;
    p.N = q.N;
    p.V = q.V;
    p.M = q.M;
    p.nblk = q.nblk;
    p.mpitch = q.mpitch;
    p.splits = q.splits;
    p.bps = q.bps;
    p.c_f32 = q.out.f32;
    // the pipelined kernel where every copy is a 16-byte aligned run
    if (p.V % kPipeRows == 0 && p.nblk % kPipeChunk == 0 && pipe_aligned(p.values) && pipe_aligned(p.meta) &&
        pipe_aligned(p.colidx) && pipe_split_blocks(p.nblk, p.splits) * p.M * NB <= kPipeBHalves)
        return launch_stream_pipe<NB>(p, stream);
    const int64_t ctas = (p.R / p.V) * p.splits;
    if (p.splits == 1) {
        spmm_stream_rm_kernel<NB, RW, U><<<static_cast<unsigned>(ctas), 32 * kStreamWarps, 0, stream>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(32 * kStreamWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, spmm_stream_rm_kernel<NB, RW, U>, p);
}

template <int NB, int RW, int U>
cudaError_t launch_stream3(const StreamArgs& p, cudaStream_t stream) {
    const bool plain = p.bn == 1 && p.out.ns == 1 && p.out.bias == nullptr && p.out.act == VNM_ACT_NONE;
    return plain ? launch_stream_rm<NB, RW, U>(p, stream) : launch_stream4<NB, RW, U, false>(p, stream);
}

template <int NB>
cudaError_t launch_stream_nb(const StreamArgs& p, cudaStream_t stream) {
    // RW rows per warp (V <= 16 * RW in one pass), U = 16 / RW blocks per lane
    if (p.V <= 16) return launch_stream3<NB, 1, 8>(p, stream);
    if (p.V <= 32) return launch_stream3<NB, 2, 8>(p, stream);
    if (p.V <= 64) return launch_stream3<NB, 4, 4>(p, stream);
    return launch_stream3<NB, 8, 2>(p, stream);
}

template <int NB>
cudaError_t launch_nb(const SimtArgs& p, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>((p.R + kSimtWarps - 1) / kSimtWarps);
    spmm_simt_kernel<NB><<<grid, 32 * kSimtWarps, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_spmm_simt(const vnm_matrix_s& A, const void* B, int64_t bk, int64_t bn, int64_t N,
                             const OutSpec& out, cudaStream_t stream) {
    SimtArgs p;
    p.values = static_cast<const uint32_t*>(A.values);
    p.meta = static_cast<const uint8_t*>(A.meta);
    p.colidx = static_cast<const uint32_t*>(A.colidx);
    p.B = static_cast<const __half*>(B);
    p.bk = bk;
    p.bn = bn;
    p.out = out;
    p.R = A.R;
    p.N = N;
    p.V = A.V;
    p.M = A.M;
    p.nblk = A.K / A.M;
    p.mpitch = meta_pitch(A.K, A.M);
    if (A.R == 0 || N == 0) return cudaSuccess;
    if (N <= 1) return launch_nb<1>(p, stream);
    if (N <= 2) return launch_nb<2>(p, stream);
    if (N <= 4) return launch_nb<4>(p, stream);
    if (N <= 8) return launch_nb<8>(p, stream);
    return launch_nb<16>(p, stream);
}

int stream_chunk_blocks(int V) { return V <= 32 ? 256 : V <= 64 ? 128 : 64; }

int stream_pipe_splits(const vnm_matrix_s& A, int64_t N) {
    const int64_t nblk = A.K / A.M;
    if (N < 1 || N > 8 || A.V % kPipeRows != 0 || nblk % kPipeChunk != 0 || !pipe_aligned(A.values) ||
        !pipe_aligned(A.meta) || !pipe_aligned(A.colidx))
        return 0;
    // the CTAs that are resident at once, the fewest splits whose rows of B fit
    const int64_t rows_blocks = std::max<int64_t>(1, A.R / A.V);
    int need = 1;
    while (need <= 8 && pipe_split_blocks(nblk, need) * A.M * pipe_nb(N) > kPipeBHalves) need *= 2;
    if (need > 8) return 0;
    int s = need;
    while (s * 2 <= 4 && rows_blocks * s * 2 <= pipe_resident(pipe_nb(N)) * static_cast<int64_t>(A.sm_count) &&
           nblk >= static_cast<int64_t>(s) * 2 * kPipeChunk)
        s *= 2;
    return s;
}

cudaError_t launch_spmm_stream(const vnm_matrix_s& A, const void* B, int64_t bk, int64_t bn, int64_t N,
                               const OutSpec& out, int splits, cudaStream_t stream) {
    StreamArgs p;
    p.values = static_cast<const uint32_t*>(A.values);
    p.meta = static_cast<const uint8_t*>(A.meta);
    p.colidx = static_cast<const uint32_t*>(A.colidx);
    p.B = static_cast<const __half*>(B);
    p.bk = bk;
    p.bn = bn;
    p.out = out;
    p.R = A.R;
    p.N = N;
    p.V = A.V;
    p.M = A.M;
    p.nblk = A.K / A.M;
    p.mpitch = meta_pitch(A.K, A.M);
    if (A.R == 0 || N == 0) return cudaSuccess;
    if (N > 8) return cudaErrorInvalidValue;
    // splits: 1, 2, 4 or 8 (a cluster), none of them empty
    if (splits != 1 && splits != 2 && splits != 4 && splits != 8) return cudaErrorInvalidValue;
    if (splits > p.nblk) return cudaErrorInvalidValue;
    p.splits = splits;
    p.bps = (p.nblk + splits - 1) / splits;
    if ((splits - 1) * p.bps >= p.nblk) return cudaErrorInvalidValue;
    if (N <= 1) return launch_stream_nb<1>(p, stream);
    if (N <= 2) return launch_stream_nb<2>(p, stream);
    if (N <= 4) return launch_stream_nb<4>(p, stream);
    return launch_stream_nb<8>(p, stream);
}

cudaError_t launch_splitk_reduce(const float* partial, int splits, int64_t R, int64_t N, const OutSpec& out,
                                 cudaStream_t stream) {
    const int64_t total = R * N;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((total + threads - 1) / threads, 148 * 16);
    splitk_reduce_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(partial, splits, R, N, out);
    return cudaGetLastError();
}

// 32 x 32 tiles through shared memory (padded row: no bank conflicts).
__global__ void transpose_f16_kernel(const __half* __restrict__ src, int64_t ld_src, int64_t R, int64_t C,
                                     __half* __restrict__ dst, int64_t ld_dst) {
    __shared__ __half tile[32][33];
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32, c0 = static_cast<int64_t>(blockIdx.x) * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int64_t r = r0 + i, c = c0 + threadIdx.x;
        if (r < R && c < C) tile[i][threadIdx.x] = src[r * ld_src + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int64_t c = c0 + i, r = r0 + threadIdx.x;
        if (r < R && c < C) dst[c * ld_dst + r] = tile[threadIdx.x][i];
    }
}

cudaError_t launch_transpose_f16(const void* src, int64_t ld_src, int64_t R, int64_t C, void* dst, int64_t ld_dst,
                                 cudaStream_t stream) {
    if (R == 0 || C == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((C + 31) / 32), static_cast<unsigned>((R + 31) / 32));
    transpose_f16_kernel<<<grid, dim3(32, 8), 0, stream>>>(static_cast<const __half*>(src), ld_src, R, C,
                                                          static_cast<__half*>(dst), ld_dst);
    return cudaGetLastError();
}

}  // namespace vnm
