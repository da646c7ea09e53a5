// layout_noalloc.cu -- moe_layout_noalloc: the sort-free layout for callers that
// cannot allocate device memory, with its scratch in a fixed device array.
//
// Who needs it: code that runs where cudaMalloc is not an option -- a serving
// process that reserves all of its device memory up front and forbids allocation
// afterwards, or a plug-in whose host owns the allocator and hands out no scratch.  moe_layout needs a caller-supplied workspace for its
// per-chunk counts; this variant needs none, because that scratch lives in a
// file-scope __device__ array that is part of the library's image.
//
// The array is LAYOUT_NOALLOC_SCRATCH_BYTES (1 MiB) on every GPU that loads the
// library and stays allocated until the process exits.  It holds the per-chunk
// expert counts and their scan, 2 * ceil(N*k/256) * E int32 values, which caps the
// shape at ceil(N*k/256) * E <= 131072 (for example N*k = 131072 with E = 256).
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;

// The scratch.  In host code this name is only a stand-in for the device symbol:
// its device address must be fetched with cudaGetSymbolAddress before a kernel
// may be given it.
static __device__ __align__(256) unsigned char g_layout_scratch[kNoAllocScratchBytes];

// Id of the calling thread's current CUDA context (unique for the life of the
// process), or 0 when there is none or the driver query is unavailable.  The
// driver entry points are fetched through the runtime, so the library does not
// link libcuda.  Called with the cache's mutex held.
unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    }
    if (!get_current || !get_id) return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_layout_scratch on the current device, looked up with that
// device current and cached with the id of the context it belongs to.  A device
// reset (or any teardown of the context) reloads the library's device image, and
// the array may then live elsewhere: when the current context's id differs from
// the cached one, or cannot be read, the address is looked up again.  Returns
// nullptr on failure.
void* scratch_on_current_device(cudaError_t* err) {
    static std::mutex mu;
    static void* addr[256] = {};
    static unsigned long long ctx[256] = {};
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= 256) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (!addr[dev] || id == 0 || id != ctx[dev]) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_layout_scratch);   // makes the primary context current
        if (*err != cudaSuccess || p == nullptr) return nullptr;
        addr[dev] = p;
        ctx[dev] = current_context_id();
    }
    return addr[dev];
}

}  // namespace
}  // namespace moe

extern "C" int moe_layout_noalloc(const int32_t* idx, const moe_shape_t* shape, int32_t* counts,
                                  int32_t* offsets, int32_t* sched, int32_t* inv, void* stream) {
    using namespace moe;
    const int rc = validate_shape(shape);     // the same checks, and statuses, as moe_layout
    if (rc != MOE_OK) return rc;
    const moe_shape_t& s = *shape;
    if (!counts || !offsets || (s.N > 0 && (!idx || !sched || !inv))) return MOE_ERR_INVALID_ARG;
    const int T = s.N * s.k;
    const size_t per_array = sizeof(int32_t) * (size_t)layout_chunks(T) * (size_t)s.E;
    const size_t per_array_padded = (per_array + 255) & ~(size_t)255;
    if (2 * per_array_padded > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;  // shape too large
    cudaError_t err = cudaSuccess;
    uint8_t* scratch = static_cast<uint8_t*>(scratch_on_current_device(&err));
    if (!scratch) return MOE_ERR_CUDA;
    // Both arrays are written in full before they are read, so stale contents
    // from an earlier call need no clearing.
    int32_t* cnt = reinterpret_cast<int32_t*>(scratch);
    int32_t* base = reinterpret_cast<int32_t*>(scratch + per_array_padded);
    err = launch_layout(idx, s.N, s.k, s.E, s.S, counts, offsets, sched, inv, cnt, base,
                        /*ws=*/nullptr, (cudaStream_t)stream);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
