// bevpool_internal.cuh -- shared device helpers and host-side launch plumbing
// for libbevpool (sm_103a).  Not part of the public ABI (include/bevpool.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <climits>

#include "../../include/bevpool.h"
#include "fastdiv.h"

namespace bevpool {

constexpr int kThreads = 256;            // every kernel in the library runs 256-thread CTAs
constexpr int kWarps = kThreads / 32;

// Launch accounting: every kernel launch made by the library bumps this.
extern std::atomic<int64_t> g_kernel_launches;

inline void count_launch() { g_kernel_launches.fetch_add(1, std::memory_order_relaxed); }

// Per-device properties the host code needs (cached).
struct DeviceInfo {
    int sm_count = 0;
    int l2_bytes = 0;
    int max_smem_optin = 0;
};
bool device_info(DeviceInfo *out);

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Number of frustum points NC*D*H*W into *nf, or false if a factor is below 1
// or the product exceeds INT32_MAX (checked one multiply at a time, so the
// product never overflows).
inline bool frustum_points(int32_t NC, int32_t D, int32_t H, int32_t W, int64_t *nf) {
    if (NC < 1 || D < 1 || H < 1 || W < 1) return false;
    int64_t n = NC;
    for (const int32_t f : {D, H, W}) {
        if (n > INT32_MAX / f) return false;
        n *= f;
    }
    *nf = n;
    return true;
}

// Programmatic dependent launch.  A kernel launched with launch_dependent()
// may be scheduled while the previous kernel of the stream is still running
// (once every CTA of that kernel has called grid_dep_allow() or exited); its
// grid_dep_wait() then blocks until the previous kernel has completed and its
// writes are visible.  In a kernel launched normally grid_dep_wait() returns
// at once.  Every kernel here waits before touching data an earlier kernel
// of the call writes; the map build's counting and scatter passes read their
// block of the caller's cell ids first (written before the call began, so
// complete and visible once the first kernel of the call has passed its own
// wait, which comes before that kernel lets its dependants start).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_allow() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- device helpers

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive sum over the 256 threads of a CTA.  `scratch` needs kWarps+1 ints.
// Returns this thread's exclusive prefix; *total receives the CTA sum.
__device__ __forceinline__ int cta_exclusive_sum(int v, int *scratch, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kWarps ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < kWarps; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kWarps) scratch[lane] = w;   // inclusive warp totals
    }
    __syncthreads();
    int warp_excl = warp ? scratch[warp - 1] : 0;
    int tot = scratch[kWarps - 1];
    __syncthreads();                            // scratch may be reused right after
    *total = tot;
    return warp_excl + x - v;
}

// Sum over the CTA (result valid in every thread).  `scratch` needs kWarps ints.
__device__ __forceinline__ long long cta_sum_ll(long long v, long long *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    long long t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += scratch[w];
    __syncthreads();
    return t;
}

// Max over the CTA (result valid in every thread).  `scratch` needs kWarps ints.
__device__ __forceinline__ int cta_max(int v, int *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    int t = scratch[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) t = max(t, scratch[w]);
    __syncthreads();
    return t;
}

// ---------------------------------------------------------------- launchers

// Build-map pipeline (build_map.cu).  All pointers device; sizes validated.
struct BuildMapArgs {
    const int32_t *cell_ids;
    int32_t NC, D, H, W, n_cells;
    int32_t *ranks_depth, *ranks_feat, *ranks_bev;
    int32_t *interval_starts, *interval_lengths;
    int32_t *d_counts;
    void *workspace;
    size_t workspace_bytes;
    bool counting;            // counting-sort path (n_cells <= kCountingMaxCells) or radix path
    cudaStream_t stream;
};
// Grids up to this many cells use the counting-sort map build; larger ones the radix sort.
constexpr int32_t kCountingMaxCells = 1 << 24;
size_t build_map_workspace_bytes(int64_t n_frustum, int32_t n_cells);   // preferred path
size_t radix_workspace_bytes(int64_t n_frustum);
size_t count_workspace_bytes(int64_t n_frustum, int32_t n_cells);
cudaError_t launch_build_map(const BuildMapArgs &a);
cudaError_t launch_build_map_radix(const BuildMapArgs &a);
cudaError_t launch_build_map_counting(const BuildMapArgs &a);

// The launch plan of one forward call, chosen on the host from the sizes and
// the device (forward_impl.cuh: plan_variant, launch_forward_t).
struct ForwardPlan {
    int32_t variant;          // kernel variant: 0 default, 1 lean, 2 short, 3 lean-short
    int32_t ctas_per_sm;      // compute CTAs per SM in one wave
    int32_t owners;           // owners per compute CTA
    int32_t batch;            // points in flight per owner
    int32_t round;            // points per staged round of a compute CTA
    int32_t n_compute;        // compute CTAs
    int32_t fill_cells;       // cells per fill CTA
    int32_t n_fill;           // fill CTAs
};

// Forward (forward_f16.cu / forward_e4m3.cu).
struct ForwardArgs {
    const void *depth, *feat;
    const void *feat_block;   // NVFP4 block scales (else unused)
    const int32_t *ranks_depth, *ranks_feat, *ranks_bev;
    const int32_t *interval_starts, *interval_lengths;
    const int32_t *d_counts;
    int32_t n_points, n_intervals, n_cells, C;
    int64_t n_depth;          // NC*D*H*W
    int32_t n_feat_rows;      // NC*H*W
    float scale;              // depth_scale * feat_scale (/ out_scale for an E4M3 output)
    int out_e4m3;             // 1: E4M3 output codes, 0: fp16 output
    int streaming_stores;     // 1: evict-first output stores (HBM regime)
    int loose_capacity;       // 1: n_points is the whole frustum, not a bound close to the device count
    int sm_count;             // SMs of the current device (launch sizing)
    void *out;
    cudaStream_t stream;
    ForwardPlan *plan_out;    // non-null: write the launch plan here and launch nothing
};
bool forward_supported(int dtype, int C);
cudaError_t launch_forward_f16(const ForwardArgs &a);             // fp16 output
cudaError_t launch_forward_e4m3(const ForwardArgs &a);
cudaError_t launch_forward_f16_e4m3out(const ForwardArgs &a);     // E4M3 output (C % 16 == 0)
cudaError_t launch_forward_e4m3_e4m3out(const ForwardArgs &a);
cudaError_t launch_forward_nvfp4(const ForwardArgs &a);           // NVFP4 features, fp16 output
cudaError_t launch_forward_nvfp4_e4m3out(const ForwardArgs &a);   // NVFP4 features, E4M3 output

// Map validation (abi.cu).
cudaError_t launch_validate_map(const int32_t *ranks_depth, const int32_t *ranks_feat,
                                const int32_t *ranks_bev, const int32_t *starts,
                                const int32_t *lengths, int32_t n_points, int32_t n_intervals,
                                int64_t n_depth, int32_t n_feat_rows, int32_t n_cells,
                                int32_t *d_result, cudaStream_t stream);

}  // namespace bevpool
