// Internal declarations shared by the host API (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/vnm.h"

constexpr uint32_t kVnmMagic = 0x564E4D31u;  // "VNM1"
constexpr int kStatusBytes = 256;

// Layout of the device status block (int32 words).
enum StatusWord : int {
    kStatusCode = 0,     // first error recorded (0 = none)
    kStatusWhere = 1,    // kernel-specific detail of that error
    kStatusCount = 2,    // number of errors recorded
};

struct vnm_matrix_s {
    uint32_t magic;
    int64_t R, K;
    int32_t V, M;
    void* values;   // fp16 [R][2K/M]
    void* meta;     // uint8 [R][ceil(2K/M/4)]
    void* colidx;   // uint8 [R/V][K/M][4]
    int device;
    int sm_count;
    int cc_major, cc_minor;
    int* status;    // device, kStatusBytes
};

namespace vnm {

inline int64_t values_per_row(int64_t K, int32_t M) { return 2 * (K / M); }
inline int64_t meta_pitch(int64_t K, int32_t M) { return (values_per_row(K, M) + 3) / 4; }

// Kernel-side error recording: keep the first code, count all.
__device__ __forceinline__ void record_error(int* status, int code, int where) {
    if (atomicCAS(status + kStatusCode, 0, code) == 0) status[kStatusWhere] = where;
    atomicAdd(status + kStatusCount, 1);
}

// Where and how an SpMM writes C: element (r, n) at C + r * rs + n * ns
// (in elements: row-major C has rs = ld_c, ns = 1; the Linear-layer form
// Y = X . A^T writes C transposed, rs = 1, ns = ld_y), after adding bias[r]
// (fp16; none when null) and applying an activation (a vnm_activation).
struct OutSpec {
    void* C;
    int64_t rs, ns;
    bool f32;
    const __half* bias;
    int act;
};

inline OutSpec out_rowmajor(void* C, int64_t ld_c, bool f32) { return OutSpec{C, ld_c, 1, f32, nullptr, 0}; }

#ifdef __CUDACC__
// The value stored for accumulator v of row r (before the rounding to C's type).
__device__ __forceinline__ float out_transform(const OutSpec& o, int64_t r, float v) {
    if (o.bias != nullptr) v += __half2float(o.bias[r]);
    if (o.act == VNM_ACT_RELU) {
        v = fmaxf(v, 0.f);
    } else if (o.act == VNM_ACT_GELU) {
        v = 0.5f * v * (1.f + erff(v * 0.70710678118654752f));
    }
    return v;
}

__device__ __forceinline__ void out_store(const OutSpec& o, int64_t r, int64_t n, float v) {
    v = out_transform(o, r, v);
    if (o.f32)
        static_cast<float*>(o.C)[r * o.rs + n * o.ns] = v;
    else
        static_cast<__half*>(o.C)[r * o.rs + n * o.ns] = __float2half_rn(v);
}
#endif

// ---- launchers (each returns the launch's cudaError_t) ----

cudaError_t launch_compress(const vnm_matrix_s& A, const void* W, int64_t ld_w, cudaStream_t stream);
cudaError_t launch_decompress(const vnm_matrix_s& A, void* W, int64_t ld_w, cudaStream_t stream);

// Streaming CUDA-core SpMM for N <= 8: one CTA per (V-block row, K split);
// splits (1, 2, 4 or 8, none empty) form a thread-block cluster and reduce
// in distributed shared memory: no workspace. `stream_chunk_blocks(V)`
// blocks are staged per pass.
// B element (k, n) at B + k * bk + n * bn (row-major B: bk = ld_b, bn = 1;
// the Linear-layer form reads X as B: bk = 1, bn = ld_x).
cudaError_t launch_spmm_stream(const vnm_matrix_s& A, const void* B, int64_t bk, int64_t bn, int64_t N,
                               const OutSpec& out, int splits, cudaStream_t stream);
int stream_chunk_blocks(int V);
// Splits of the pipelined streaming kernel for this matrix and N (1, 2, 4 or
// 8), 0 where it does not apply (then the general streaming kernel runs).
int stream_pipe_splits(const vnm_matrix_s& A, int64_t N);

// CUDA-core SpMM; writes C directly (fp16 or fp32).
cudaError_t launch_spmm_simt(const vnm_matrix_s& A, const void* B, int64_t bk, int64_t bn, int64_t N,
                             const OutSpec& out, cudaStream_t stream);

// Shared-memory rings of the tensor-core kernel, in stages of 128 columns
// of the MMAs' K (4 MMA k-steps). B: 64-column swizzle atoms of 128 rows x
// 128 bytes, or, for 16- and 32-column tiles loaded by TMA ("narrow"), 128
// rows of exactly tile_n columns (32B/64B swizzle); large stages keep many
// gathered bytes in flight per barrier operation. A (tile_m rows x 128
// bytes, 128B swizzle) has its own, shallower ring of at most 32 KB (never
// deeper than B's). The m-indices do not pass through shared memory.
constexpr int kTcStageK = 128;        // MMA-K columns (rows of B) per stage
constexpr int kTcARingBytes = 32 * 1024;
constexpr int kTcMaxStages = 8;

__host__ __device__ constexpr int tc_a_stage_bytes(int tile_m) { return tile_m * 128; }

__host__ __device__ constexpr int tc_b_stage_bytes(int tile_n, bool narrow_b) {
    return narrow_b ? kTcStageK * tile_n * 2 : ((tile_n + 63) / 64) * kTcStageK * 128;
}

// Dynamic shared memory a CTA may use: about all of it for wide tiles (one
// CTA per SM); half for tiles of at most 64 columns, so that two CTAs share
// an SM (more loads in flight per SM on the small, memory-bound products).
__host__ __device__ constexpr int tc_smem_budget(int tile_n) {
    return tile_n <= 64 ? 110 * 1024 : 227 * 1024 - 2 * 1024;  // minus alignment slack and barriers
}

// B stages of the tensor-core kernel for a tile: as many as fit beside the
// A ring, at most kTcMaxStages.
__host__ __device__ constexpr int tc_stages(int tile_m, int tile_n, bool narrow_b) {
    const int s = (tc_smem_budget(tile_n) - kTcARingBytes) / tc_b_stage_bytes(tile_n, narrow_b);
    return s > kTcMaxStages ? kTcMaxStages : s;
}

// A stages: as many as fit in the A ring, never more than the B stages.
__host__ __device__ constexpr int tc_a_stages(int tile_m, int b_stages) {
    const int s = kTcARingBytes / tc_a_stage_bytes(tile_m);
    return s < b_stages ? s : b_stages;
}

// B of a tensor-core launch is loaded narrow (see tc_b_slot_bytes).
__host__ __device__ constexpr bool tc_narrow_b(int tile_n, bool gather) { return !gather && tile_n < 64; }

// How the tensor-core kernel forms its operands.
enum TcMode : int {
    // M == 4: A is plain 2:4; A values by TMA, B in TMA tiles over K
    kTcTiled = 0,
    // M > 4: the MMAs run over the condensed K; A values by TMA, the 4
    // selected rows of B per block gathered through column-loc
    kTcGather = 1,
    // M == 8: the MMAs run over the whole K. A row keeps 2 values in a block
    // of 8 columns, so it never has more than 2 in a group of 4: the kernel
    // re-encodes each block's two values as 2:4 over the block's columns
    // (zeros fill the groups' free slots) and writes A to shared memory
    // itself; B in TMA tiles over K as for M == 4
    kTcLift = 2,
};

// The tensor-core kernel's K runs over units of kTcStageK columns: of the
// condensed K (kTcTiled, kTcGather) or of the whole K (kTcLift); both equal
// K / 128 when M == 4.
inline int64_t tc_k_units(int64_t K, int32_t M, bool lift) { return lift ? K / kTcStageK : (K / M) / 32; }

struct TcLaunch {
    CUtensorMap tm_a;   // values, box {64, tile_m}: one stage (4 MMA k-steps), 128B swizzle (not read by kTcLift)
    CUtensorMap tm_b;   // B, box {64, 128}, 128B swizzle; {tile_n, 128}, 32B/64B swizzle when narrow;
                        // K-major: box {64, tile_n} (64 K x tile_n rows), 128B swizzle
    int tile_m, tile_n, stages, splits;
    int mode;           // a TcMode
    bool b_kmajor;      // B given K-major (X of the Linear-layer form: tm_b boxes {64 K, tile_n}); tiled and lift
    int sm_count;       // persistent grid: at most sm_count x resident CTAs per SM
    int skip_stage;     // tests of the bounded waits only (-1: none)
};

// tcgen05 sparse SpMM; with splits > 1 it writes fp32 partials to
// `partial` ([splits][R][N]) and a second kernel reduces them into C.
cudaError_t launch_spmm_tc(const vnm_matrix_s& A, const TcLaunch& L, const void* B, int64_t ld_b, int64_t N,
                           const OutSpec& out, float* partial, cudaStream_t stream);

cudaError_t launch_splitk_reduce(const float* partial, int splits, int64_t R, int64_t N, const OutSpec& out,
                                 cudaStream_t stream);

// dst[c][r] = src[r][c] for an R x C fp16 matrix (leading dimensions in elements).
cudaError_t launch_transpose_f16(const void* src, int64_t ld_src, int64_t R, int64_t C, void* dst, int64_t ld_dst,
                                 cudaStream_t stream);

// Fused dense GEMM + prune-and-encode (W = X . Y^T compressed into A in the
// GEMM's epilogue): tm_x / tm_y are X (R x D) and Y (K x D) as 2-D fp16
// maps with boxes of 64 D-columns x 128 rows, 128B swizzle. Shapes it
// serves: V divides 128, M in {4, 8, 16, 32, 64}.
bool gemm_compress_shape_ok(int V, int M);
cudaError_t launch_gemm_compress(const vnm_matrix_s& A, const CUtensorMap& tm_x, const CUtensorMap& tm_y, int64_t D,
                                 void* w_out, int64_t ld_w, cudaStream_t stream);

// Energy of a pruning pattern (a vnm_pattern): partial sums in units of
// 2^-24 as pairs of uint64 (low, high) in the workspace, from byte 256 on:
// n_total pairs of sum |W|, then (from pair kEnergyKeptPair) n_kept pairs of
// the kept |w|; word 0 of the workspace is set when W holds Inf or NaN.
constexpr int kEnergyKeptPair = 1024;
size_t energy_workspace_bytes(int64_t R, int64_t K, int V);
cudaError_t launch_energy(const vnm_matrix_s& A, const void* W, int64_t ld_w, int pattern, void* workspace,
                          int sm_count, int* n_total_partials, int* n_kept_partials, cudaStream_t stream);

// The workspace form of the M = 8 re-encoding: writes A as a plain 2:4
// matrix over the whole K (values2: fp16 [R][K/2], meta2: [R][K/8] bytes,
// both 16-byte aligned), which the 2:4 tensor-core path then reads by TMA.
cudaError_t launch_lift_expand(const vnm_matrix_s& A, void* values2, void* meta2, cudaStream_t stream);

// The plan vnm_spmm makes with an unlimited workspace, but never the
// written-out 2:4 form of M = 8 (lift = 2): what a caller whose workspace
// holds only split-K partials can run.
vnm_spmm_plan plan_without_expansion(const vnm_matrix_s& A, const void* B, int64_t ld_b, int64_t N);

// Bitmap format for unstructured sparsity (R % 64 == 0): bitmaps uint64
// [R/64][K], offsets uint32 [R/64][K] (relative to the row block's base),
// bases int64 [R/64 + 1], values fp16 [bases[R/64]].
cudaError_t launch_bitmap_encode_counts(const void* W, int64_t ld_w, int64_t R, int64_t K, void* bitmaps,
                                        void* offsets, int64_t* bases, cudaStream_t stream);
cudaError_t launch_bitmap_encode_fill(const void* W, int64_t ld_w, int64_t R, int64_t K, const void* bitmaps,
                                      const void* offsets, const int64_t* bases, void* values, cudaStream_t stream);
int bitmap_spmm_splits(int64_t R, int64_t K, int64_t N, int sm_count);
cudaError_t launch_bitmap_spmm(int64_t R, int64_t K, const void* bitmaps, const void* offsets, const int64_t* bases,
                               const void* values, const void* B, int64_t ld_b, int64_t N, const OutSpec& out,
                               int splits, float* partial, cudaStream_t stream);

// Pipeline stages the tensor-core kernel is built with for a tile (0: no such tile).
int tc_default_stages(int tile_m, int tile_n, bool gather);


}  // namespace vnm
