// build_map_noalloc.cu -- bevpool_build_map_noalloc: the scatter-map build for
// callers that may not allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they build the map: an inference-engine plugin whose enqueue
// step is not allowed to allocate, real-time or safety-certified code that
// forbids allocation after start-up, or a host program that runs inside
// another framework which owns every device allocation.  For them this entry
// point runs the same kernels as bevpool_build_map, but its scratch lives in a
// fixed-size array compiled into the library (g_build_map_scratch below)
// instead of a caller-provided workspace.
//
// Properties of that array:
//   - it is a file-scope __device__ array, so every GPU on which the library's
//     kernels are loaded holds its BEVPOOL_NOALLOC_SCRATCH_BYTES until the
//     process exits;
//   - all calls on a device share it, and it keeps whatever the last call left
//     in it.  Nothing in it needs to start at zero: every kernel of the build
//     writes the scratch words it later reads within the same call;
//   - two calls whose work overlaps on the GPU (different streams, or the same
//     array reached through two host threads) race on it; callers must order
//     such calls themselves.
//
// In host code the array's name only stands for the host-side shadow of the
// symbol, not a device address, so it is never passed to a kernel.  The
// device address is looked up with cudaGetSymbolAddress, with the device
// current, on the first call on each device, and again whenever the device's
// context has changed since (after cudaDeviceReset the module is loaded anew
// and the old address is void); calls in between reuse it.  That look-up is
// not allowed while a stream is being captured, so the first call on a
// device (and the first after a reset) must come before any stream capture
// that contains this entry point.
//
// With lazy module loading (the CUDA default) the array's memory is committed
// by that first look-up, not when the library is loaded; if the device is
// short of memory then, the call returns BEVPOOL_ERR_CUDA.  Callers that must
// not fail later make one call during start-up.
#include <mutex>

#include <cuda.h>   // driver types only; the two driver calls below are reached through the runtime

#include "bevpool_internal.cuh"

namespace bevpool {
namespace {

constexpr size_t kNoallocScratchBytes = BEVPOOL_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_build_map_scratch[kNoallocScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Process-unique id of the calling thread's current context, or 0 when there
// is none (or the driver cannot say).
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
        cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_build_map_scratch on the current device: looked up
// with that device current, and again when the device's context has changed
// (a reset) since the last look-up.
cudaError_t scratch_address(void **out) {
    static std::mutex mu;
    static void *addr[64] = {};
    static unsigned long long ctx_of[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_build_map_scratch);   // makes the primary context current if needed
        if (e != cudaSuccess) return e;
        addr[dev] = p;
        ctx_of[dev] = current_context_id();
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace bevpool

extern "C" bevpool_status bevpool_build_map_noalloc(const int32_t *cell_ids, int32_t NC, int32_t D, int32_t H,
                                                    int32_t W, int32_t n_cells, int32_t *ranks_depth,
                                                    int32_t *ranks_feat, int32_t *ranks_bev,
                                                    int32_t *interval_starts, int32_t *interval_lengths,
                                                    int32_t *d_counts, int32_t *h_counts, void *stream) {
    using namespace bevpool;
    int64_t nf = 0;
    if (!frustum_points(NC, D, H, W, &nf) || n_cells < 1) return BEVPOOL_ERR_INVALID_ARG;
    if (nf > BEVPOOL_NOALLOC_MAX_FRUSTUM) return BEVPOOL_ERR_WORKSPACE;   // larger than the built-in scratch
    // bevpool_build_map takes the counting-sort path when its workspace fits in
    // the scratch and the radix path otherwise; the radix path always fits for
    // frusta up to the limit.
    if (radix_workspace_bytes(nf) > kNoallocScratchBytes) return BEVPOOL_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) {
        cudaGetLastError();
        return BEVPOOL_ERR_CUDA;
    }
    return bevpool_build_map(cell_ids, NC, D, H, W, n_cells, ranks_depth, ranks_feat, ranks_bev, interval_starts,
                             interval_lengths, d_counts, h_counts, scratch, kNoallocScratchBytes, stream);
}
