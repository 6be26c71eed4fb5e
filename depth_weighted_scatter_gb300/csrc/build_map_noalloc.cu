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
// first call on each device looks up the device address with
// cudaGetSymbolAddress (with that device current) and caches it; that
// look-up is not allowed while a stream is being captured, so the first call
// on a device must come before any stream capture that contains this entry
// point.
#include <mutex>

#include "bevpool_internal.cuh"

namespace bevpool {
namespace {

constexpr size_t kNoallocScratchBytes = BEVPOOL_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_build_map_scratch[kNoallocScratchBytes];

// Device address of g_build_map_scratch on the current device (looked up once
// per device, with that device current).
cudaError_t scratch_address(void **out) {
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_build_map_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
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
    if (NC < 1 || D < 1 || H < 1 || W < 1 || n_cells < 1) return BEVPOOL_ERR_INVALID_ARG;
    const int64_t nf = static_cast<int64_t>(NC) * D * H * W;
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
