// vnm_spmm_noalloc: the SpMM for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc where they need this product: a
// serving loop whose device memory is already held in full by another
// caching allocator, or a latency-critical path that must not take the
// implicit device synchronisation that cudaMalloc and cudaFree can cause.
// Such a caller cannot create a vnm_matrix either (vnm_matrix_create
// allocates a status block), so this entry point takes the compressed
// arrays directly and keeps its split-K scratch, and its internal status
// words, in a fixed static device array of this library.
//
// The array's device address is resolved with cudaGetSymbolAddress once per
// CUDA context, on the first call made with that context current (the
// device's primary context, or a context the caller created and made
// current); that first call should come before any stream capture. The
// cache is keyed by the context's unique id, so a context that was
// destroyed or reset (cudaDeviceReset) and created again resolves the
// address anew instead of reusing a stale one. In host code the array's name
// is only a host stand-in, so the kernels are given the resolved address.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "vnm_internal.h"

namespace {

constexpr size_t kStatusRegionBytes = 256;             // status words (first kStatusBytes of it used)
constexpr size_t kScratchBytes = size_t(8) << 20;      // 8 MiB of fp32 split-K partial sums
constexpr int kMaxContexts = 64;

// Holds the status region followed by the split-K scratch. Every call shares
// it and it keeps the last call's contents; calls that overlap on the GPU
// (for example on two streams) race on it.
static __device__ __align__(256) unsigned char g_noalloc_area[kStatusRegionBytes + kScratchBytes];

struct ResolvedArea {
    unsigned long long ctx_id;
    unsigned char* address;
};

std::mutex g_mutex;
ResolvedArea g_resolved[kMaxContexts] = {};
int g_resolved_count = 0;
int g_resolved_next = 0;  // slot reused once the table is full (oldest first)

// Driver entry points for the current context and its id (CUDA 12.0+).
struct ContextQueries {
    PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const ContextQueries& context_queries() {
    static ContextQueries q;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &r) == cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            q.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &r) == cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            q.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    return q;
}

// Unique id of the calling thread's current CUDA context (false if none).
bool current_context_id(unsigned long long* id) {
    const ContextQueries& q = context_queries();
    if (q.get_current == nullptr || q.get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (q.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return q.get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_noalloc_area in the current context (null on failure).
unsigned char* area_address() {
    unsigned long long id = 0;
    if (!current_context_id(&id)) {
        // no context is current yet: resolving the symbol makes the device's
        // primary context current (the runtime's usual set-up); ask again
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_area) != cudaSuccess) return nullptr;
        if (!current_context_id(&id)) return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    for (int i = 0; i < g_resolved_count; ++i)
        if (g_resolved[i].ctx_id == id) return g_resolved[i].address;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_area) != cudaSuccess) return nullptr;
    int slot = g_resolved_count < kMaxContexts ? g_resolved_count++ : g_resolved_next++ % kMaxContexts;
    g_resolved[slot].ctx_id = id;
    g_resolved[slot].address = static_cast<unsigned char*>(p);
    return g_resolved[slot].address;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" vnm_status vnm_spmm_noalloc(int64_t R, int64_t K, int32_t V, int32_t M, const void* values,
                                       const void* meta, const void* colidx, const void* B, int64_t ld_b,
                                       int64_t N, void* C, int64_t ld_c, vnm_dtype c_type, int32_t* status,
                                       vnm_stream_t stream) {
    size_t vb = 0, mb = 0, cb = 0;
    if (vnm_sizes(R, K, V, M, &vb, &mb, &cb) != VNM_OK) return VNM_ERR_INVALID_ARG;
    if ((vb && (values == nullptr || !aligned16(values))) || (mb && (meta == nullptr || !aligned16(meta))) ||
        (cb && (colidx == nullptr || !aligned16(colidx))))
        return VNM_ERR_INVALID_ARG;
    if (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u) != 0) return VNM_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return VNM_ERR_CUDA;
    unsigned char* area = area_address();
    if (area == nullptr) return VNM_ERR_CUDA;
    int sms = 0, major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return VNM_ERR_CUDA;

    // a handle on the stack: it describes the caller's arrays and owns nothing
    vnm_matrix_s A;
    A.magic = kVnmMagic;
    A.R = R;
    A.K = K;
    A.V = V;
    A.M = M;
    A.values = const_cast<void*>(values);
    A.meta = const_cast<void*>(meta);
    A.colidx = const_cast<void*>(colidx);
    A.device = dev;
    A.sm_count = sms;
    A.cc_major = major;
    A.cc_minor = minor;
    A.status = status != nullptr ? status : reinterpret_cast<int*>(area);

    // the plan vnm_spmm makes with unlimited workspace (without the written-out
    // 2:4 form of M = 8, which the scratch does not hold); its split-K
    // partials must fit the static scratch
    vnm_spmm_plan plan;
    vnm_status st = vnm_spmm_plan_query(&A, B, ld_b, N, c_type, 0, &plan);  // argument checks
    if (st != VNM_OK) return st;
    plan = vnm::plan_without_expansion(A, B, ld_b, N);
    size_t need = 0;
    if (plan.path == VNM_PATH_TC && plan.splits > 1)
        need = static_cast<size_t>(plan.splits) * static_cast<size_t>(R) * static_cast<size_t>(N) * sizeof(float);
    if (need > kScratchBytes) return VNM_ERR_INVALID_ARG;  // partials would exceed the 8 MiB static scratch

    // the internal status words must start at zero for this call
    if (status == nullptr && cudaMemsetAsync(area, 0, kStatusBytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return VNM_ERR_CUDA;
    return vnm_spmm_with_plan(&A, &plan, B, ld_b, N, C, ld_c, c_type, need ? area + kStatusRegionBytes : nullptr, need,
                              stream);
}
