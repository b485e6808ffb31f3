// moe_noalloc.cu -- moe_layout_noalloc: the layout entry point for callers
// that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: a plugin inside an
// inference engine whose device memory is planned ahead of time and owned by
// the engine, or a plain C caller with no device allocator of its own
// (cudaMalloc also synchronises the whole device, which a hot path cannot
// afford).  For them this variant keeps the layout scratch in a fixed array
// of the library's own device memory, declared below.  Every GPU that loads
// the library holds this array until the process exits.

#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace {

// The scratch itself.  In host code this name is only a host-side stand-in:
// its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_layout_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch in the current device's context.  It is
// looked up on every call rather than cached: the lookup allocates nothing
// and costs far less than a launch, and a cached address would go stale when
// the module is loaded again at another address (after cudaDeviceReset, or
// in another context on the same device).  The first lookup on a device
// loads the library's device code there.
cudaError_t scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_layout_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" int moe_layout_noalloc(const moe_problem* problem, const int32_t* ids,
                                  const moe_layout_t* layout, moe_stream_t stream) {
    MOE_NVTX("moe_layout_noalloc");
    size_t need = 0;
    const int rc = moe_workspace_bytes(problem, &need);
    if (rc != MOE_OK) return rc;
    if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_CAPACITY;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    // The ordinary layout path clears the counters it needs at the start of
    // every call, so leftovers of an earlier call never leak into this one.
    return moe_layout(problem, ids, scratch, layout, stream);
}
