// Host side of the libvnm C ABI (include/vnm.h): argument checks, size
// queries, launch planning, TMA descriptor encoding and kernel dispatch.
// Every check runs before anything is enqueued; kernels report what they
// find through the matrix's device status block.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "vnm_internal.h"
#include "vnm_testing.h"

namespace {

using vnm::meta_pitch;
using vnm::values_per_row;

constexpr int32_t kMaxV = 4096;
constexpr int32_t kMinM = 4;
constexpr int32_t kMaxM = 256;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_shape(int64_t R, int64_t K, int32_t V, int32_t M) {
    if (R < 0 || K < 0) return false;
    if (V < 1 || V > kMaxV) return false;
    if (M < kMinM || M > kMaxM) return false;
    if (R % V != 0 || K % M != 0) return false;
    if (R > (int64_t(1) << 31) || K > (int64_t(1) << 31)) return false;  // TMA coordinates are int32
    return true;
}

bool valid_handle(vnm_matrix A) { return A != nullptr && A->magic == kVnmMagic; }

vnm_status check_device(vnm_matrix A) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return VNM_ERR_CUDA;
    return dev == A->device ? VNM_OK : VNM_ERR_INVALID_ARG;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D row-major tensor: dim0 contiguous elements per row, dim1 rows,
// row_bytes apart; box0 x box1 box.
bool encode_2d(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, uint64_t dim0, uint64_t dim1,
               uint64_t row_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t gdim[2] = {dim0, dim1};
    const cuuint64_t gstride[1] = {row_bytes};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t estride[2] = {1, 1};
    return enc(tm, dt, 2, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core path serves: condensed K a whole number of 128-column
// stages (K/M % 32 == 0), every row tile inside one V-block row when
// column-loc matters (M > 4 needs V % 64 == 0: 128-row tiles when
// V % 128 == 0, else 64-row tiles; M == 4 takes any V since column-loc is
// then the identity), B rows 16-byte aligned, N >= 8.
bool tc_geometry_ok(const vnm_matrix_s& A) {
    if (A.K == 0 || (A.K / A.M) % 32 != 0) return false;
    return A.M == 4 || A.V % 64 == 0;
}

// The re-encoded path (M == 8 as 2:4 over the whole K) serves any V that
// is a multiple of 16 (the 16 rows of a half-warp share column-loc words)
// with K a whole number of 128-column stages; tiles of 128 rows.
bool lift_ok(const vnm_matrix_s& A) { return A.M == 8 && A.V % 16 == 0 && A.K > 0 && A.K % vnm::kTcStageK == 0; }

bool tc_tile_m_ok(const vnm_matrix_s& A, int tile_m) {
    if (tile_m == 128) return A.M == 4 || A.V % 128 == 0;
    if (tile_m == 64) return A.M == 4 || A.V % 64 == 0;
    return false;
}

bool tc_operands_ok(const void* B, int64_t ld_b, int64_t N) {
    return N >= 8 && aligned(B, 16) && (ld_b % 8) == 0;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The split the streaming kernel will actually use: 1, 2, 4 or 8 (the CTAs
// of a V-block row form one cluster and reduce in distributed shared
// memory), at most `requested`, no split empty.
int effective_stream_splits(const vnm_matrix_s& A, int requested) {
    const int64_t nblk = A.K / A.M;
    int s = 1;
    while (s * 2 <= std::min(requested, 8)) s *= 2;
    while (s > 1 && (s - 1) * ceil_div(nblk, s) >= nblk) s /= 2;
    return s;
}

// K splits of the streaming CUDA-core path (N <= 8): the pipelined kernel's
// choice where it applies; else up to four CTAs per SM, at most 4 splits (8
// measured slower on every decode shape), every split at least one staged
// chunk of blocks. No workspace: the splits of a V-block row reduce within
// their cluster.
int64_t stream_splits(const vnm_matrix_s& A, int64_t N) {
    if (N > 8 || N < 1) return 1;
    if (const int ps = vnm::stream_pipe_splits(A, N)) return ps;
    const int64_t nblk = A.K / A.M;
    const int64_t rows_blocks = std::max<int64_t>(1, A.R / A.V);
    int64_t s = ceil_div(4 * static_cast<int64_t>(A.sm_count), rows_blocks);
    s = std::min<int64_t>(s, std::max<int64_t>(1, nblk / vnm::stream_chunk_blocks(A.V)));
    return effective_stream_splits(A, static_cast<int>(std::min<int64_t>(s, 4)));
}

// Workspace bytes of the written-out 2:4 form of an M = 8 matrix (lift = 2):
// values [R][K/2] fp16, then m-indices [R][K/8], each 256-byte aligned.
size_t expand_values_bytes(const vnm_matrix_s& A) { return (static_cast<size_t>(A.R) * A.K + 255) & ~size_t(255); }
size_t expand_bytes(const vnm_matrix_s& A) {
    return expand_values_bytes(A) + ((static_cast<size_t>(A.R) * (A.K / 8) + 255) & ~size_t(255));
}

vnm_spmm_plan make_plan(const vnm_matrix_s& A, const void* B, int64_t ld_b, int64_t N, size_t workspace_bytes,
                        bool allow_expand = true) {
    vnm_spmm_plan pl;
    std::memset(&pl, 0, sizeof(pl));
    pl.splits = 1;
    if (A.R == 0 || N == 0 || A.K == 0) {
        pl.path = VNM_PATH_NONE;
        return pl;
    }
    if (!((tc_geometry_ok(A) || lift_ok(A)) && tc_operands_ok(B, ld_b, N))) {
        pl.path = VNM_PATH_SIMT;
        pl.splits = static_cast<int32_t>(stream_splits(A, N));
        return pl;
    }
    pl.path = VNM_PATH_TC;
    // M == 8 where the gather cannot run (V % 64 != 0): the MMAs over the
    // whole K with A re-encoded on chip. Where both run the gather is kept:
    // measured as fast or faster (the re-encoded A's shared-memory stores
    // contend with the MMAs' operand reads)
    pl.lift = !tc_geometry_ok(A) && lift_ok(A) ? 1 : 0;
    // M == 8 whose gather would run 64-row tiles (half-rate M = 64 MMAs), with
    // wide B and a workspace that holds it: A written out as 2:4 by a first
    // kernel, then the 2:4 path (twice the MMA work of the gather, all at the
    // M = 128 rate, operands by TMA)
    if (allow_expand && lift_ok(A) && A.V % 128 != 0 && N >= 512 && workspace_bytes >= expand_bytes(A)) pl.lift = 2;
    pl.tile_m = pl.lift || tc_tile_m_ok(A, 128) ? 128 : 64;
    // 256-column tiles for wide B (measured fastest on every shape: the
    // per-stage costs are spread over the most MMA work and the fewest A
    // re-reads); else 128, or N rounded up to a supported width
    pl.tile_n = N >= 256 ? 256 : N >= 128 ? 128 : static_cast<int32_t>(ceil_div(N, 16) * 16);
    if (pl.tile_n > 64 && pl.tile_n < 128) pl.tile_n = 128;
    if (pl.tile_n > 32 && pl.tile_n < 64) pl.tile_n = 64;
    if (pl.tile_n > 16 && pl.tile_n < 32) pl.tile_n = 32;
    pl.stages = vnm::tc_default_stages(pl.tile_m, pl.tile_n, A.M > 4 && !pl.lift);
    // split K when the tiles alone cannot fill the GPU
    const int64_t tiles = ceil_div(A.R, pl.tile_m) * ceil_div(N, pl.tile_n);
    const int64_t num_kt = vnm::tc_k_units(A.K, A.M, pl.lift != 0);
    int64_t splits = 1;
    if (tiles < A.sm_count) splits = std::min<int64_t>(num_kt, std::max<int64_t>(1, A.sm_count / tiles));
    const int64_t per_split = A.R * N * static_cast<int64_t>(sizeof(float));
    const size_t room = pl.lift == 2 ? workspace_bytes - expand_bytes(A) : workspace_bytes;
    if (splits > 1) splits = std::min<int64_t>(splits, static_cast<int64_t>(room) / per_split);
    splits = std::max<int64_t>(1, splits);
    pl.splits = static_cast<int32_t>(std::max<int64_t>(1, splits));
    return pl;
}

// The split the kernels will actually use (no empty split).
int effective_splits(const vnm_matrix_s& A, int requested, bool lift) {
    const int num_kt = static_cast<int>(vnm::tc_k_units(A.K, A.M, lift));
    const int req = std::max(1, std::min(requested, num_kt));
    const int per = (num_kt + req - 1) / req;
    return (num_kt + per - 1) / per;
}

vnm_status check_plan(const vnm_matrix_s& A, const vnm_spmm_plan& pl, const void* B, int64_t ld_b, int64_t N,
                      size_t workspace_bytes, const void* workspace) {
    for (int32_t r : pl.reserved)
        if (r != 0) return VNM_ERR_INVALID_ARG;
    if (pl.lift < 0 || pl.lift > 2) return VNM_ERR_INVALID_ARG;  // read by the TC path only
    if (pl.path == VNM_PATH_SIMT) return pl.splits < 1 ? VNM_ERR_INVALID_ARG : VNM_OK;  // no workspace
    if (pl.path != VNM_PATH_TC) return VNM_ERR_UNSUPPORTED;
    if (!tc_operands_ok(B, ld_b, N)) return VNM_ERR_UNSUPPORTED;
    if (pl.lift) {
        if (!lift_ok(A) || pl.tile_m != 128) return VNM_ERR_UNSUPPORTED;
    } else if (!tc_geometry_ok(A) || !tc_tile_m_ok(A, pl.tile_m)) {
        return VNM_ERR_UNSUPPORTED;
    }
    const int depth = vnm::tc_default_stages(pl.tile_m, pl.tile_n, A.M > 4 && !pl.lift);
    if (depth == 0 || (pl.stages != 0 && pl.stages != depth)) return VNM_ERR_UNSUPPORTED;
    if (pl.splits < 1) return VNM_ERR_INVALID_ARG;
    const int s = effective_splits(A, pl.splits, pl.lift != 0);
    const size_t need = (pl.lift == 2 ? expand_bytes(A) : 0) + (s > 1 ? static_cast<size_t>(s) * A.R * N * sizeof(float) : 0);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, pl.lift == 2 ? 256 : 16)))
        return VNM_ERR_INVALID_ARG;
    return VNM_OK;
}

// The B operand of a product: element (k, n) at ptr + k * bk + n * bn.
// Row-major B (vnm_spmm): bk = ld_b, bn = 1. The Linear-layer form reads X
// (N x K, row-major) as a K-major B: bk = 1, bn = ld_x.
struct BOperand {
    const void* ptr;
    int64_t bk, bn;
    bool kmajor() const { return bk == 1 && bn != 1; }
};

vnm_status run_product(vnm_matrix A, const vnm_spmm_plan& pl, const BOperand& B, int64_t N, const vnm::OutSpec& out,
                       void* workspace, cudaStream_t stream, int skip_stage = -1) {
    cudaError_t e = cudaSuccess;
    if (pl.path == VNM_PATH_SIMT) {
        if (N <= 8)
            e = vnm::launch_spmm_stream(*A, B.ptr, B.bk, B.bn, N, out, effective_stream_splits(*A, pl.splits), stream);
        else
            e = vnm::launch_spmm_simt(*A, B.ptr, B.bk, B.bn, N, out, stream);
    } else if (pl.path == VNM_PATH_TC && pl.lift == 2) {
        // A written out as a plain 2:4 matrix over the whole K, then the 2:4 path on it
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        if (vnm::launch_lift_expand(*A, ws, ws + expand_values_bytes(*A), stream) != cudaSuccess) return VNM_ERR_CUDA;
        vnm_matrix_s A2 = *A;
        A2.M = 4;
        A2.values = ws;
        A2.meta = ws + expand_values_bytes(*A);
        vnm_spmm_plan pl2 = pl;
        pl2.lift = 0;
        return run_product(&A2, pl2, B, N, out, ws + expand_bytes(*A), stream, skip_stage);
    } else if (pl.path == VNM_PATH_TC) {
        vnm::TcLaunch L;
        std::memset(&L, 0, sizeof(L));
        L.tile_m = pl.tile_m;
        L.tile_n = pl.tile_n;
        L.mode = A->M == 4 ? vnm::kTcTiled : pl.lift ? vnm::kTcLift : vnm::kTcGather;
        const bool gather = L.mode == vnm::kTcGather;
        L.b_kmajor = B.kmajor();
        if (L.b_kmajor && gather) return VNM_ERR_INTERNAL;
        L.stages = vnm::tc_default_stages(pl.tile_m, pl.tile_n, gather);
        L.splits = effective_splits(*A, pl.splits, pl.lift != 0);
        L.sm_count = A->sm_count;
        L.skip_stage = skip_stage;
        const uint64_t vpr = static_cast<uint64_t>(values_per_row(A->K, A->M));
        // A values: one stage (64 values per row, 4 MMA k-steps) per box, 128B swizzle
        bool ok = encode_2d(&L.tm_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A->values, vpr, A->R, vpr * 2, 64,
                            static_cast<uint32_t>(pl.tile_m), CU_TENSOR_MAP_SWIZZLE_128B);
        if (L.b_kmajor) {
            // K-major B: boxes of 64 K (128 bytes) x tile_n rows, 128B swizzle
            ok = ok && encode_2d(&L.tm_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B.ptr, A->K, N, B.bn * 2, 64,
                                 static_cast<uint32_t>(pl.tile_n), CU_TENSOR_MAP_SWIZZLE_128B);
        } else {
            // B tiles by TMA (M == 4, lift): 64-column atoms, or exactly tile_n columns with the
            // matching swizzle for 16- and 32-column tiles; the gather reads B itself
            const bool narrow = vnm::tc_narrow_b(pl.tile_n, gather);
            ok = ok && encode_2d(&L.tm_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B.ptr, N, A->K, B.bk * 2,
                                 narrow ? static_cast<uint32_t>(pl.tile_n) : 64,
                                 gather ? 1 : static_cast<uint32_t>(vnm::kTcStageK),
                                 !narrow ? CU_TENSOR_MAP_SWIZZLE_128B
                                         : pl.tile_n == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
        }
        if (!ok) return VNM_ERR_CUDA;
        e = vnm::launch_spmm_tc(*A, L, B.ptr, B.bk, N, out, static_cast<float*>(workspace), stream);
    }
    return e == cudaSuccess ? VNM_OK : VNM_ERR_CUDA;
}

vnm_status run_spmm(vnm_matrix A, const vnm_spmm_plan& pl, const void* B, int64_t ld_b, int64_t N, void* C,
                    int64_t ld_c, vnm_dtype c_type, void* workspace, cudaStream_t stream, int skip_stage = -1) {
    return run_product(A, pl, BOperand{B, ld_b, 1}, N, vnm::out_rowmajor(C, ld_c, c_type == VNM_F32), workspace,
                       stream, skip_stage);
}

vnm_status check_spmm_args(vnm_matrix A, const void* B, int64_t ld_b, int64_t N, const void* C, int64_t ld_c,
                           vnm_dtype c_type) {
    if (!valid_handle(A)) return VNM_ERR_INVALID_ARG;
    if (c_type != VNM_F16 && c_type != VNM_F32) return VNM_ERR_INVALID_ARG;
    if (N < 0 || ld_b < std::max<int64_t>(N, 1) || ld_c < std::max<int64_t>(N, 1)) return VNM_ERR_INVALID_ARG;
    if (N > (int64_t(1) << 31)) return VNM_ERR_INVALID_ARG;
    const bool work = A->R > 0 && N > 0;
    if (work && (C == nullptr || !aligned(C, c_type == VNM_F32 ? 4 : 2))) return VNM_ERR_INVALID_ARG;
    if (work && A->K > 0 && (B == nullptr || !aligned(B, 2))) return VNM_ERR_INVALID_ARG;
    return VNM_OK;
}

}  // namespace

namespace vnm {

vnm_spmm_plan plan_without_expansion(const vnm_matrix_s& A, const void* B, int64_t ld_b, int64_t N) {
    return make_plan(A, B, ld_b, N, SIZE_MAX / 2, /*allow_expand=*/false);
}

}  // namespace vnm

extern "C" {

const char* vnm_status_string(vnm_status s) {
    switch (s) {
        case VNM_OK: return "VNM_OK";
        case VNM_ERR_INVALID_ARG: return "VNM_ERR_INVALID_ARG";
        case VNM_ERR_UNSUPPORTED: return "VNM_ERR_UNSUPPORTED";
        case VNM_ERR_CUDA: return "VNM_ERR_CUDA";
        case VNM_ERR_NONFINITE: return "VNM_ERR_NONFINITE";
        case VNM_ERR_TIMEOUT: return "VNM_ERR_TIMEOUT";
        case VNM_ERR_INTERNAL: return "VNM_ERR_INTERNAL";
    }
    return "VNM_ERR_UNKNOWN";
}

int32_t vnm_version(void) { return VNM_VERSION; }

vnm_status vnm_sizes(int64_t R, int64_t K, int32_t V, int32_t M, size_t* values_bytes, size_t* meta_bytes,
                     size_t* colidx_bytes) {
    if (!valid_shape(R, K, V, M)) return VNM_ERR_INVALID_ARG;
    if (values_bytes) *values_bytes = static_cast<size_t>(R * values_per_row(K, M)) * 2;
    if (meta_bytes) *meta_bytes = static_cast<size_t>(R * meta_pitch(K, M));
    if (colidx_bytes) *colidx_bytes = static_cast<size_t>((R / V) * (K / M) * 4);
    return VNM_OK;
}

vnm_status vnm_matrix_create(int64_t R, int64_t K, int32_t V, int32_t M, void* values, void* meta, void* colidx,
                             vnm_matrix* out) {
    if (out == nullptr) return VNM_ERR_INVALID_ARG;
    *out = nullptr;
    size_t vb, mb, cb;
    if (vnm_sizes(R, K, V, M, &vb, &mb, &cb) != VNM_OK) return VNM_ERR_INVALID_ARG;
    if ((vb && (values == nullptr || !aligned(values, 16))) || (mb && (meta == nullptr || !aligned(meta, 16))) ||
        (cb && (colidx == nullptr || !aligned(colidx, 16))))
        return VNM_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return VNM_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return VNM_ERR_CUDA;
    vnm_matrix A = new (std::nothrow) vnm_matrix_s;
    if (A == nullptr) return VNM_ERR_INTERNAL;
    A->magic = kVnmMagic;
    A->R = R;
    A->K = K;
    A->V = V;
    A->M = M;
    A->values = values;
    A->meta = meta;
    A->colidx = colidx;
    A->device = dev;
    A->sm_count = prop.multiProcessorCount;
    A->cc_major = prop.major;
    A->cc_minor = prop.minor;
    A->status = nullptr;
    if (cudaMalloc(&A->status, kStatusBytes) != cudaSuccess || cudaMemset(A->status, 0, kStatusBytes) != cudaSuccess) {
        if (A->status) cudaFree(A->status);
        A->magic = 0;
        delete A;
        return VNM_ERR_CUDA;
    }
    *out = A;
    return VNM_OK;
}

vnm_status vnm_matrix_destroy(vnm_matrix A) {
    if (A == nullptr) return VNM_OK;
    if (!valid_handle(A)) return VNM_ERR_INVALID_ARG;
    A->magic = 0;
    vnm_status st = VNM_OK;
    if (A->status != nullptr && cudaFree(A->status) != cudaSuccess) st = VNM_ERR_CUDA;  // cudaFree synchronises
    delete A;
    return st;
}

vnm_status vnm_compress(vnm_matrix A, const void* W, int64_t ld_w, vnm_stream_t stream) {
    if (!valid_handle(A)) return VNM_ERR_INVALID_ARG;
    if (ld_w < std::max<int64_t>(A->K, 1)) return VNM_ERR_INVALID_ARG;
    if (A->R == 0 || A->K == 0) return VNM_OK;
    if (W == nullptr || !aligned(W, 16) || (ld_w % 8) != 0) return VNM_ERR_INVALID_ARG;
    vnm_status st = check_device(A);
    if (st != VNM_OK) return st;
    return vnm::launch_compress(*A, W, ld_w, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? VNM_OK
                                                                                                   : VNM_ERR_CUDA;
}

vnm_status vnm_decompress(vnm_matrix A, void* W_out, int64_t ld_w, vnm_stream_t stream) {
    if (!valid_handle(A)) return VNM_ERR_INVALID_ARG;
    if (ld_w < std::max<int64_t>(A->K, 1)) return VNM_ERR_INVALID_ARG;
    if (A->R == 0 || A->K == 0) return VNM_OK;
    if (W_out == nullptr || !aligned(W_out, 2)) return VNM_ERR_INVALID_ARG;
    vnm_status st = check_device(A);
    if (st != VNM_OK) return st;
    return vnm::launch_decompress(*A, W_out, ld_w, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? VNM_OK
               : VNM_ERR_CUDA;
}

// ---- the Linear-layer form Y = act(X . A^T + bias) ----

// How vnm_linear runs a product: the plan, whether X is first transposed into
// the workspace (the gather needs a row-major B), and the workspace layout.
struct LinearPlan {
    vnm_spmm_plan pl;
    bool transpose;       // X^T (K x T, leading dimension ldt) at the workspace start
    int64_t ldt;
    size_t t_bytes;       // bytes of X^T, 256-byte aligned
    size_t bytes;         // total workspace: X^T, then the split-K partials
};

LinearPlan make_linear_plan(const vnm_matrix_s& A, bool x_aligned, int64_t T, size_t workspace_bytes) {
    LinearPlan lp;
    std::memset(&lp, 0, sizeof(lp));
    lp.ldt = ((std::max<int64_t>(T, 1) + 7) / 8) * 8;
    // the plan vnm_spmm makes for a row-major B of T columns (alignment assumed)
    const void* aligned_b = reinterpret_cast<const void*>(uintptr_t(256));
    lp.pl = make_plan(A, aligned_b, lp.ldt, T, SIZE_MAX / 2, /*allow_expand=*/false);
    if (lp.pl.path == VNM_PATH_TC) {
        // K-major B is read in place by TMA where the B tiles are not gathered: M == 4, or
        // M == 8 re-encoded (lift); the gather needs X^T in the workspace, as does an X that
        // TMA cannot read (not 16-byte aligned rows)
        if (A.M == 8 && lift_ok(A) && !lp.pl.lift) {
            lp.pl.lift = 1;
            lp.pl.tile_m = 128;
            lp.pl.stages = vnm::tc_default_stages(128, lp.pl.tile_n, false);
            const int64_t tiles = ceil_div(A.R, 128) * ceil_div(T, lp.pl.tile_n);
            const int64_t num_kt = vnm::tc_k_units(A.K, A.M, true);
            lp.pl.splits = tiles < A.sm_count
                               ? static_cast<int32_t>(std::min<int64_t>(num_kt, std::max<int64_t>(1, A.sm_count / tiles)))
                               : 1;
        }
        const bool gather = A.M > 4 && !lp.pl.lift;
        lp.transpose = gather || !x_aligned;
    }
    if (lp.transpose) lp.t_bytes = (static_cast<size_t>(A.K) * lp.ldt * 2 + 255) & ~static_cast<size_t>(255);
    // split K only within the workspace given
    if (lp.pl.path == VNM_PATH_TC && lp.pl.splits > 1) {
        const size_t per_split = static_cast<size_t>(A.R) * T * sizeof(float);
        const size_t room = workspace_bytes > lp.t_bytes ? workspace_bytes - lp.t_bytes : 0;
        lp.pl.splits = static_cast<int32_t>(std::max<int64_t>(
            1, std::min<int64_t>(lp.pl.splits, static_cast<int64_t>(room / std::max<size_t>(per_split, 1)))));
    }
    const int s = lp.pl.path == VNM_PATH_TC ? effective_splits(A, lp.pl.splits, lp.pl.lift != 0) : 1;
    lp.bytes = lp.t_bytes + (s > 1 ? static_cast<size_t>(s) * A.R * T * sizeof(float) : 0);
    return lp;
}

vnm_status vnm_linear_workspace_size(vnm_matrix A, int64_t T, size_t* bytes) {
    if (!valid_handle(A) || bytes == nullptr || T < 0) return VNM_ERR_INVALID_ARG;
    // the largest need: an unaligned X (transposed) and an unlimited split
    *bytes = make_linear_plan(*A, false, T, SIZE_MAX / 2).bytes;
    return VNM_OK;
}

vnm_status vnm_linear(vnm_matrix A, const void* X, int64_t ld_x, int64_t T, const void* bias, vnm_activation act,
                      void* Y, int64_t ld_y, vnm_dtype y_type, void* workspace, size_t workspace_bytes,
                      vnm_stream_t stream) {
    if (!valid_handle(A)) return VNM_ERR_INVALID_ARG;
    if (y_type != VNM_F16 && y_type != VNM_F32) return VNM_ERR_INVALID_ARG;
    if (act != VNM_ACT_NONE && act != VNM_ACT_RELU && act != VNM_ACT_GELU) return VNM_ERR_INVALID_ARG;
    if (T < 0 || T > (int64_t(1) << 31) || ld_x < std::max<int64_t>(A->K, 1) || ld_y < std::max<int64_t>(A->R, 1))
        return VNM_ERR_INVALID_ARG;
    if (A->R == 0 || T == 0) return VNM_OK;
    if (Y == nullptr || !aligned(Y, y_type == VNM_F32 ? 4 : 2)) return VNM_ERR_INVALID_ARG;
    if (bias != nullptr && !aligned(bias, 2)) return VNM_ERR_INVALID_ARG;
    if (A->K > 0 && (X == nullptr || !aligned(X, 2))) return VNM_ERR_INVALID_ARG;
    if (workspace == nullptr) workspace_bytes = 0;
    vnm_status st = check_device(A);
    if (st != VNM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // C = A . X^T is R x T; it is Y^T: element (r, t) at Y + t * ld_y + r
    vnm::OutSpec out{Y, 1, ld_y, y_type == VNM_F32, static_cast<const __half*>(bias), static_cast<int>(act)};
    if (A->K == 0) {
        // Y = act(bias): the split-K reduction over no partial sums
        return vnm::launch_splitk_reduce(nullptr, 0, A->R, T, out, s) == cudaSuccess ? VNM_OK : VNM_ERR_CUDA;
    }
    const bool x_aligned = aligned(X, 16) && ld_x % 8 == 0;
    const LinearPlan lp = make_linear_plan(*A, x_aligned, T, workspace_bytes);
    if (workspace_bytes < lp.bytes || (lp.bytes > 0 && !aligned(workspace, 256))) return VNM_ERR_INVALID_ARG;
    BOperand B{X, 1, ld_x};
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (lp.transpose) {
        if (vnm::launch_transpose_f16(X, ld_x, T, A->K, ws, lp.ldt, s) != cudaSuccess) return VNM_ERR_CUDA;
        B = BOperand{ws, lp.ldt, 1};
    }
    return run_product(A, lp.pl, B, T, out, ws + lp.t_bytes, s);
}

// ---- the bitmap format (unstructured sparsity) ----

vnm_status vnm_bitmap_sizes(int64_t R, int64_t K, size_t* bitmaps_bytes, size_t* offsets_bytes, size_t* bases_bytes,
                            size_t* values_max_bytes) {
    if (R < 0 || K < 0 || R % 64 != 0 || R > (int64_t(1) << 31) || K > (int64_t(1) << 26)) return VNM_ERR_INVALID_ARG;
    const size_t tiles = static_cast<size_t>(R / 64) * static_cast<size_t>(K);
    if (bitmaps_bytes) *bitmaps_bytes = tiles * 8;
    if (offsets_bytes) *offsets_bytes = tiles * 4;
    if (bases_bytes) *bases_bytes = (static_cast<size_t>(R / 64) + 1) * 8;
    if (values_max_bytes) *values_max_bytes = static_cast<size_t>(R) * K * 2;
    return VNM_OK;
}

vnm_status vnm_bitmap_encode(const void* W, int64_t ld_w, int64_t R, int64_t K, void* bitmaps, void* offsets,
                             int64_t* bases, void* values, int64_t values_capacity, int64_t* values_len,
                             vnm_stream_t stream) {
    if (vnm_bitmap_sizes(R, K, nullptr, nullptr, nullptr, nullptr) != VNM_OK || values_len == nullptr)
        return VNM_ERR_INVALID_ARG;
    if (ld_w < std::max<int64_t>(K, 1) || bases == nullptr || !aligned(bases, 8)) return VNM_ERR_INVALID_ARG;
    const bool work = R > 0 && K > 0;
    if (work && (W == nullptr || !aligned(W, 2) || bitmaps == nullptr || !aligned(bitmaps, 8) || offsets == nullptr ||
                 !aligned(offsets, 4)))
        return VNM_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (vnm::launch_bitmap_encode_counts(W, ld_w, R, K, bitmaps, offsets, bases, s) != cudaSuccess) return VNM_ERR_CUDA;
    int64_t len = 0;
    if (cudaMemcpyAsync(&len, bases + R / 64, sizeof(int64_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return VNM_ERR_CUDA;
    *values_len = len;
    if (len > values_capacity || (len > 0 && (values == nullptr || !aligned(values, 16)))) return VNM_ERR_INVALID_ARG;
    return vnm::launch_bitmap_encode_fill(W, ld_w, R, K, bitmaps, offsets, bases, values, s) == cudaSuccess
               ? VNM_OK
               : VNM_ERR_CUDA;
}

int bitmap_device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    return std::max(1, sms);
}

vnm_status vnm_bitmap_spmm_workspace_size(int64_t R, int64_t K, int64_t N, size_t* bytes) {
    if (bytes == nullptr || N < 0 || vnm_bitmap_sizes(R, K, nullptr, nullptr, nullptr, nullptr) != VNM_OK)
        return VNM_ERR_INVALID_ARG;
    const int s = vnm::bitmap_spmm_splits(R, K, N, bitmap_device_sms());
    *bytes = s > 1 ? static_cast<size_t>(s) * R * N * sizeof(float) : 0;
    return VNM_OK;
}

vnm_status vnm_bitmap_spmm(int64_t R, int64_t K, const void* bitmaps, const void* offsets, const int64_t* bases,
                           const void* values, const void* B, int64_t ld_b, int64_t N, void* C, int64_t ld_c,
                           vnm_dtype c_type, void* workspace, size_t workspace_bytes, vnm_stream_t stream) {
    if (vnm_bitmap_sizes(R, K, nullptr, nullptr, nullptr, nullptr) != VNM_OK) return VNM_ERR_INVALID_ARG;
    if (c_type != VNM_F16 && c_type != VNM_F32) return VNM_ERR_INVALID_ARG;
    if (N < 0 || N > (int64_t(1) << 31) || ld_b < std::max<int64_t>(N, 1) || ld_c < std::max<int64_t>(N, 1))
        return VNM_ERR_INVALID_ARG;
    if (R == 0 || N == 0) return VNM_OK;
    if (C == nullptr || !aligned(C, c_type == VNM_F32 ? 4 : 2)) return VNM_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const vnm::OutSpec out = vnm::out_rowmajor(C, ld_c, c_type == VNM_F32);
    if (K == 0) return vnm::launch_splitk_reduce(nullptr, 0, R, N, out, s) == cudaSuccess ? VNM_OK : VNM_ERR_CUDA;
    if (bitmaps == nullptr || offsets == nullptr || bases == nullptr || values == nullptr || B == nullptr ||
        !aligned(bitmaps, 8) || !aligned(offsets, 4) || !aligned(bases, 8) || !aligned(values, 16) || !aligned(B, 2))
        return VNM_ERR_INVALID_ARG;
    int splits = vnm::bitmap_spmm_splits(R, K, N, bitmap_device_sms());
    const size_t per = static_cast<size_t>(R) * N * sizeof(float);
    if (workspace == nullptr || !aligned(workspace, 16)) workspace_bytes = 0;
    splits = static_cast<int>(std::max<size_t>(1, std::min<size_t>(splits, workspace_bytes / per)));
    return vnm::launch_bitmap_spmm(R, K, bitmaps, offsets, bases, values, B, ld_b, N, out, splits,
                                   splits > 1 ? static_cast<float*>(workspace) : nullptr, s) == cudaSuccess
               ? VNM_OK
               : VNM_ERR_CUDA;
}

vnm_status vnm_energy_workspace_size(vnm_matrix A, size_t* bytes) {
    if (!valid_handle(A) || bytes == nullptr) return VNM_ERR_INVALID_ARG;
    *bytes = vnm::energy_workspace_bytes(A->R, A->K, A->V);
    return VNM_OK;
}

vnm_status vnm_energy(vnm_matrix A, const void* W, int64_t ld_w, vnm_pattern pattern, void* workspace,
                      size_t workspace_bytes, uint64_t kept_units[2], uint64_t total_units[2], double* energy,
                      vnm_stream_t stream) {
    if (!valid_handle(A)) return VNM_ERR_INVALID_ARG;
    if (pattern != VNM_PATTERN_VNM && pattern != VNM_PATTERN_UNSTRUCTURED && pattern != VNM_PATTERN_VECTORWISE)
        return VNM_ERR_INVALID_ARG;
    if (ld_w < std::max<int64_t>(A->K, 1)) return VNM_ERR_INVALID_ARG;
    auto put = [&](unsigned __int128 kept, unsigned __int128 total) {
        if (kept_units) {
            kept_units[0] = static_cast<uint64_t>(kept);
            kept_units[1] = static_cast<uint64_t>(kept >> 64);
        }
        if (total_units) {
            total_units[0] = static_cast<uint64_t>(total);
            total_units[1] = static_cast<uint64_t>(total >> 64);
        }
        if (energy) *energy = total == 0 ? 1.0 : static_cast<double>(static_cast<long double>(kept) /
                                                                     static_cast<long double>(total));
    };
    if (A->R == 0 || A->K == 0) {
        put(0, 0);
        return VNM_OK;
    }
    if (W == nullptr || !aligned(W, 2)) return VNM_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned(workspace, 16) ||
        workspace_bytes < vnm::energy_workspace_bytes(A->R, A->K, A->V))
        return VNM_ERR_INVALID_ARG;
    vnm_status st = check_device(A);
    if (st != VNM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int n_total = 0, n_kept = 0;
    if (vnm::launch_energy(*A, W, ld_w, static_cast<int>(pattern), workspace, A->sm_count, &n_total, &n_kept, s) !=
        cudaSuccess)
        return VNM_ERR_CUDA;
    std::vector<uint64_t> host(2 * (vnm::kEnergyKeptPair + std::max(n_kept, 1)));
    int flags = 0;
    const uint8_t* ws = static_cast<const uint8_t*>(workspace);
    if (cudaMemcpyAsync(&flags, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(host.data(), ws + 256, sizeof(uint64_t) * 2 * n_total, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(host.data() + 2 * vnm::kEnergyKeptPair, ws + 256 + 16 * vnm::kEnergyKeptPair,
                        sizeof(uint64_t) * 2 * n_kept, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return VNM_ERR_CUDA;
    if (flags) return VNM_ERR_NONFINITE;
    unsigned __int128 total = 0, kept = 0;
    for (int i = 0; i < n_total; ++i)
        total += (static_cast<unsigned __int128>(host[2 * i + 1]) << 64) | host[2 * i];
    for (int i = 0; i < n_kept; ++i) {
        const size_t j = 2 * (vnm::kEnergyKeptPair + i);
        kept += (static_cast<unsigned __int128>(host[j + 1]) << 64) | host[j];
    }
    put(kept, total);
    return VNM_OK;
}

vnm_status vnm_gemm_compress(vnm_matrix A, const void* X, int64_t ld_x, const void* Y, int64_t ld_y, int64_t D,
                             void* W_out, int64_t ld_w, vnm_stream_t stream) {
    if (!valid_handle(A)) return VNM_ERR_INVALID_ARG;
    if (D < 0 || D > (int64_t(1) << 31)) return VNM_ERR_INVALID_ARG;
    if (ld_x < std::max<int64_t>(D, 1) || ld_y < std::max<int64_t>(D, 1)) return VNM_ERR_INVALID_ARG;
    if (W_out != nullptr && (ld_w < std::max<int64_t>(A->K, 1) || !aligned(W_out, 2))) return VNM_ERR_INVALID_ARG;
    if (!vnm::gemm_compress_shape_ok(A->V, A->M)) return VNM_ERR_UNSUPPORTED;
    if (A->R == 0 || A->K == 0) return VNM_OK;
    if (D > 0 && (X == nullptr || Y == nullptr || !aligned(X, 16) || !aligned(Y, 16) || ld_x % 8 != 0 ||
                  ld_y % 8 != 0))
        return VNM_ERR_INVALID_ARG;
    vnm_status st = check_device(A);
    if (st != VNM_OK) return st;
    CUtensorMap tm_x, tm_y;
    std::memset(&tm_x, 0, sizeof(tm_x));
    std::memset(&tm_y, 0, sizeof(tm_y));
    if (D > 0) {
        // boxes of 64 D-columns (128 bytes) x 128 rows, 128B swizzle; rows and columns past
        // the matrix read as zeros
        const bool ok = encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, D, A->R, ld_x * 2, 64, 128,
                                  CU_TENSOR_MAP_SWIZZLE_128B) &&
                        encode_2d(&tm_y, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Y, D, A->K, ld_y * 2, 64, 128,
                                  CU_TENSOR_MAP_SWIZZLE_128B);
        if (!ok) return VNM_ERR_CUDA;
    }
    return vnm::launch_gemm_compress(*A, tm_x, tm_y, D, W_out, ld_w, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? VNM_OK
               : VNM_ERR_CUDA;
}

vnm_status vnm_spmm_plan_query(vnm_matrix A, const void* B, int64_t ld_b, int64_t N, vnm_dtype c_type,
                               size_t workspace_bytes, vnm_spmm_plan* plan) {
    if (!valid_handle(A) || plan == nullptr) return VNM_ERR_INVALID_ARG;
    if (c_type != VNM_F16 && c_type != VNM_F32) return VNM_ERR_INVALID_ARG;
    if (N < 0 || ld_b < std::max<int64_t>(N, 1)) return VNM_ERR_INVALID_ARG;
    *plan = make_plan(*A, B, ld_b, N, workspace_bytes);
    return VNM_OK;
}

vnm_status vnm_spmm_workspace_size(vnm_matrix A, int64_t N, size_t* bytes) {
    if (!valid_handle(A) || bytes == nullptr || N < 0) return VNM_ERR_INVALID_ARG;
    // assume a B that the tensor-core path accepts; an unlimited workspace
    const void* aligned_b = reinterpret_cast<const void*>(uintptr_t(256));
    vnm_spmm_plan pl = make_plan(*A, aligned_b, ((std::max<int64_t>(N, 1) + 7) / 8) * 8, N, SIZE_MAX / 2);
    *bytes = 0;
    int s = 1;
    if (pl.path == VNM_PATH_TC) s = effective_splits(*A, pl.splits, pl.lift != 0);
    if (s > 1) *bytes = static_cast<size_t>(s) * A->R * N * sizeof(float);
    if (pl.path == VNM_PATH_TC && pl.lift == 2) *bytes += expand_bytes(*A);
    return VNM_OK;
}

vnm_status vnm_spmm_with_plan(vnm_matrix A, const vnm_spmm_plan* plan, const void* B, int64_t ld_b, int64_t N,
                              void* C, int64_t ld_c, vnm_dtype c_type, void* workspace, size_t workspace_bytes,
                              vnm_stream_t stream) {
    vnm_status st = check_spmm_args(A, B, ld_b, N, C, ld_c, c_type);
    if (st != VNM_OK) return st;
    if (plan == nullptr) return VNM_ERR_INVALID_ARG;
    if (A->R == 0 || N == 0) return VNM_OK;
    st = check_device(A);
    if (st != VNM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (A->K == 0) {
        const size_t esz = c_type == VNM_F32 ? 4 : 2;
        return cudaMemset2DAsync(C, ld_c * esz, 0, N * esz, A->R, s) == cudaSuccess ? VNM_OK : VNM_ERR_CUDA;
    }
    st = check_plan(*A, *plan, B, ld_b, N, workspace_bytes, workspace);
    if (st != VNM_OK) return st;
    return run_spmm(A, *plan, B, ld_b, N, C, ld_c, c_type, workspace, s);
}

vnm_status vnm_spmm(vnm_matrix A, const void* B, int64_t ld_b, int64_t N, void* C, int64_t ld_c, vnm_dtype c_type,
                    void* workspace, size_t workspace_bytes, vnm_stream_t stream) {
    vnm_status st = check_spmm_args(A, B, ld_b, N, C, ld_c, c_type);
    if (st != VNM_OK) return st;
    if (workspace == nullptr) workspace_bytes = 0;
    vnm_spmm_plan pl = make_plan(*A, B, ld_b, N, workspace_bytes);
    return vnm_spmm_with_plan(A, &pl, B, ld_b, N, C, ld_c, c_type, workspace, workspace_bytes, stream);
}

vnm_status vnm_testing_spmm_skip_stage(vnm_matrix A, const void* B, int64_t ld_b, int64_t N, void* C, int64_t ld_c,
                                       vnm_dtype c_type, void* workspace, size_t workspace_bytes, int32_t skip_stage,
                                       vnm_stream_t stream) {
    vnm_status st = check_spmm_args(A, B, ld_b, N, C, ld_c, c_type);
    if (st != VNM_OK) return st;
    if (workspace == nullptr) workspace_bytes = 0;
    const vnm_spmm_plan pl = make_plan(*A, B, ld_b, N, workspace_bytes);
    if (pl.path != VNM_PATH_TC || A->K == 0 || skip_stage < 0) return VNM_ERR_UNSUPPORTED;
    st = check_device(A);
    if (st != VNM_OK) return st;
    st = check_plan(*A, pl, B, ld_b, N, workspace_bytes, workspace);
    if (st != VNM_OK) return st;
    return run_spmm(A, pl, B, ld_b, N, C, ld_c, c_type, workspace, reinterpret_cast<cudaStream_t>(stream),
                    skip_stage);
}

vnm_status vnm_get_status(vnm_matrix A, vnm_stream_t stream) {
    if (!valid_handle(A)) return VNM_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return VNM_ERR_CUDA;
    int words[3] = {0, 0, 0};
    if (cudaMemcpy(words, A->status, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess) return VNM_ERR_CUDA;
    if (words[kStatusCode] != 0 && cudaMemset(A->status, 0, sizeof(words)) != cudaSuccess) return VNM_ERR_CUDA;
    return static_cast<vnm_status>(words[kStatusCode]);
}

}  // extern "C"
