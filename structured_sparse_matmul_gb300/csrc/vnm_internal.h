// Internal declarations shared by the host API (api.cu) and the kernels.
#pragma once

#include <cuda.h>
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

// ---- launchers (each returns the launch's cudaError_t) ----

cudaError_t launch_compress(const vnm_matrix_s& A, const void* W, int64_t ld_w, cudaStream_t stream);
cudaError_t launch_decompress(const vnm_matrix_s& A, void* W, int64_t ld_w, cudaStream_t stream);

// Streaming CUDA-core SpMM for N <= 8: one CTA per (V-block row, K split);
// splits (1, 2, 4 or 8, none empty) form a thread-block cluster and reduce
// in distributed shared memory: no workspace. `stream_chunk_blocks(V)`
// blocks are staged per pass.
cudaError_t launch_spmm_stream(const vnm_matrix_s& A, const void* B, int64_t ld_b, int64_t N, void* C,
                               int64_t ld_c, bool c_f32, int splits, cudaStream_t stream);
int stream_chunk_blocks(int V);

// CUDA-core SpMM; writes C directly (fp16 or fp32).
cudaError_t launch_spmm_simt(const vnm_matrix_s& A, const void* B, int64_t ld_b, int64_t N, void* C,
                             int64_t ld_c, bool c_f32, cudaStream_t stream);

// Shared-memory pipeline depth of the tensor-core kernel for a tile: as many
// 128-column stages (B rows, A values, m-indices) as fit next to the staged
// column-loc words, at most 8.
// `narrow_b`: B rows loaded by TMA into a tile exactly tile_n wide (tile_n
// 16 or 32, 32B/64B swizzle) instead of whole 64-column atoms.
__host__ __device__ constexpr int tc_stages_for(int tile_m, int tile_n, bool narrow_b = false) {
    const int b_bytes = narrow_b ? 128 * tile_n * 2 : ((tile_n + 63) / 64) * 128 * 128;
    const int stage = b_bytes + tile_m * 128 + tile_m * 16;
    const int budget = 227 * 1024 - 2 * 1024;  // minus 1 KB alignment slack and 1 KB for barriers
    const int s = budget / stage;
    return s > 8 ? 8 : s;
}

// B of a tensor-core launch is loaded narrow (see tc_stages_for).
__host__ __device__ constexpr bool tc_narrow_b(int tile_n, bool gather) { return !gather && tile_n < 64; }

struct TcLaunch {
    CUtensorMap tm_a;   // values, box {64, tile_m}: one stage (4 MMA k-steps), 128B swizzle
    CUtensorMap tm_e;   // m-indices as u32 words, box {4, tile_m}, no swizzle
    CUtensorMap tm_b;   // B, box {64, 128}, 128B swizzle; {tile_n, 128}, 32B/64B swizzle when narrow
    int tile_m, tile_n, stages, splits;
    bool gather;        // M > 4: rows of B selected through colidx
    int sm_count;       // persistent grid: at most sm_count x resident CTAs per SM
    int skip_stage;     // tests of the bounded waits only (-1: none)
};

// tcgen05 sparse SpMM; with splits > 1 it writes fp32 partials to
// `partial` ([splits][R][N]) and a second kernel reduces them into C.
cudaError_t launch_spmm_tc(const vnm_matrix_s& A, const TcLaunch& L, const void* B, int64_t ld_b, int64_t N,
                           void* C, int64_t ld_c, bool c_f32, float* partial, cudaStream_t stream);

cudaError_t launch_splitk_reduce(const float* partial, int splits, int64_t R, int64_t N, void* C,
                                 int64_t ld_c, bool c_f32, cudaStream_t stream);

// Pipeline depth the tensor-core kernel is built with for a tile (0: no such tile).
int tc_default_stages(int tile_m, int tile_n, bool gather);


}  // namespace vnm
