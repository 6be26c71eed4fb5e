// abi.cu -- the extern "C" entry points of libbevpool (declared in
// include/bevpool.h): host-side argument checks, dispatch, status codes, and
// the scatter-map validation kernel.
#include <cmath>
#include <mutex>

#include "bevpool_internal.cuh"

namespace bevpool {

std::atomic<int64_t> g_kernel_launches{0};

bool device_info(DeviceInfo *out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo d;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return false;
        cache[dev] = d;
        have[dev] = true;
    }
    *out = cache[dev];
    return true;
}

bool forward_supported(int dtype, int C) {
    if (dtype == BEVPOOL_NVFP4) {
        switch (C) {
            case 64: case 80: case 96: case 128: case 160: case 192: case 256:
                return true;
            default:
                return false;
        }
    }
    if (dtype != BEVPOOL_F16 && dtype != BEVPOOL_E4M3) return false;
    switch (C) {
        case 8: case 16: case 32: case 64: case 80: case 96: case 128: case 160: case 192: case 256:
            return true;
        default:
            return false;
    }
}

namespace {

__global__ void k_zero_word(int32_t *p) { *p = 0; }

__global__ void __launch_bounds__(kThreads)
k_validate(const int32_t *__restrict__ ranks_depth, const int32_t *__restrict__ ranks_feat,
           const int32_t *__restrict__ ranks_bev, const int32_t *__restrict__ starts,
           const int32_t *__restrict__ lengths, int32_t n_points, int32_t n_intervals, int64_t n_depth,
           int32_t n_feat_rows, int32_t n_cells, int32_t *__restrict__ result) {
    int bits = 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t i = tid; i < n_intervals; i += stride) {
        const int64_t s = starts[i], L = lengths[i];
        if (i == 0 && s != 0) bits |= 1;
        if (L < 1) bits |= 2;
        if (i + 1 < n_intervals) {
            if (starts[i + 1] != s + L) bits |= 1;
        } else if (s + L != n_points) {
            bits |= 2;
        }
        if (s >= 0 && L >= 1 && s + L <= n_points) {
            const int b0 = ranks_bev[s], b1 = ranks_bev[s + L - 1];
            if (b0 != b1) bits |= 4;
            if (s > 0 && ranks_bev[s - 1] >= b0) bits |= 4;
        }
    }
    if (tid == 0 && n_intervals == 0 && n_points != 0) bits |= 2;
    for (int64_t t = tid; t < n_points; t += stride) {
        const int b = ranks_bev[t];
        if (b < 0 || b >= n_cells) bits |= 8;
        if (t > 0 && ranks_bev[t - 1] > b) bits |= 4;
        const int d = ranks_depth[t];
        if (d < 0 || d >= n_depth) bits |= 16;
        const int f = ranks_feat[t];
        if (f < 0 || f >= n_feat_rows) bits |= 32;
    }
    if (bits) atomicOr(result, bits);
}

}  // namespace

cudaError_t launch_validate_map(const int32_t *ranks_depth, const int32_t *ranks_feat, const int32_t *ranks_bev,
                                const int32_t *starts, const int32_t *lengths, int32_t n_points,
                                int32_t n_intervals, int64_t n_depth, int32_t n_feat_rows, int32_t n_cells,
                                int32_t *d_result, cudaStream_t stream) {
    DeviceInfo info;
    if (!device_info(&info)) return cudaErrorInvalidDevice;
    k_zero_word<<<1, 1, 0, stream>>>(d_result);
    count_launch();
    const int64_t work = n_points > n_intervals ? n_points : n_intervals;
    int64_t grid = div_up(work > 0 ? work : 1, kThreads);
    const int64_t cap = static_cast<int64_t>(info.sm_count) * 8;
    if (grid > cap) grid = cap;
    k_validate<<<static_cast<int>(grid), kThreads, 0, stream>>>(ranks_depth, ranks_feat, ranks_bev, starts,
                                                                 lengths, n_points, n_intervals, n_depth,
                                                                 n_feat_rows, n_cells, d_result);
    count_launch();
    return cudaGetLastError();
}

}  // namespace bevpool

using namespace bevpool;

namespace {

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline bevpool_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return BEVPOOL_OK;
    cudaGetLastError();   // clear the runtime's last-error slot
    return BEVPOOL_ERR_CUDA;
}

inline bool frustum_ok(int32_t NC, int32_t D, int32_t H, int32_t W) {
    int64_t nf = 0;
    return frustum_points(NC, D, H, W, &nf);
}

}  // namespace

extern "C" {

const char *bevpool_status_string(bevpool_status status) {
    switch (status) {
        case BEVPOOL_OK: return "ok";
        case BEVPOOL_ERR_INVALID_ARG: return "invalid argument";
        case BEVPOOL_ERR_OUT_OF_RANGE: return "index out of range";
        case BEVPOOL_ERR_UNSUPPORTED: return "unsupported channel count or dtype";
        case BEVPOOL_ERR_WORKSPACE: return "workspace missing or too small";
        case BEVPOOL_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

int32_t bevpool_version(void) { return 300; }   // 0.3.0: launch-plan query, gather probe

int64_t bevpool_kernel_launches(void) { return g_kernel_launches.load(std::memory_order_relaxed); }

int32_t bevpool_forward_supported(bevpool_dtype dtype, int32_t C) {
    return forward_supported(static_cast<int>(dtype), C) ? 1 : 0;
}

size_t bevpool_build_map_workspace_size(int64_t n_frustum, int32_t n_cells) {
    if (n_frustum < 1 || n_frustum > INT32_MAX || n_cells < 1) return 0;
    return build_map_workspace_bytes(n_frustum, n_cells);
}

bevpool_status bevpool_build_map(const int32_t *cell_ids, int32_t NC, int32_t D, int32_t H, int32_t W,
                                 int32_t n_cells, int32_t *ranks_depth, int32_t *ranks_feat, int32_t *ranks_bev,
                                 int32_t *interval_starts, int32_t *interval_lengths, int32_t *d_counts,
                                 int32_t *h_counts, void *workspace, size_t workspace_bytes, void *stream) {
    if (!frustum_ok(NC, D, H, W) || n_cells < 1) return BEVPOOL_ERR_INVALID_ARG;
    if (!cell_ids || !ranks_depth || !ranks_feat || !ranks_bev || !interval_starts || !interval_lengths ||
        !d_counts)
        return BEVPOOL_ERR_INVALID_ARG;
    const void *ptrs[] = {cell_ids, ranks_depth, ranks_feat, ranks_bev, interval_starts, interval_lengths,
                          d_counts};
    for (const void *p : ptrs)
        if (!aligned(p, 4)) return BEVPOOL_ERR_INVALID_ARG;
    const int64_t nf = static_cast<int64_t>(NC) * D * H * W;
    if (!workspace || !aligned(workspace, 256)) return BEVPOOL_ERR_WORKSPACE;
    // Counting-sort path when the grid is small enough and the workspace holds
    // it; otherwise the radix path (smaller for huge grids).
    const bool counting = n_cells <= kCountingMaxCells && workspace_bytes >= count_workspace_bytes(nf, n_cells);
    if (!counting && workspace_bytes < radix_workspace_bytes(nf)) return BEVPOOL_ERR_WORKSPACE;

    BuildMapArgs a;
    a.cell_ids = cell_ids;
    a.NC = NC;
    a.D = D;
    a.H = H;
    a.W = W;
    a.n_cells = n_cells;
    a.ranks_depth = ranks_depth;
    a.ranks_feat = ranks_feat;
    a.ranks_bev = ranks_bev;
    a.interval_starts = interval_starts;
    a.interval_lengths = interval_lengths;
    a.d_counts = d_counts;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.counting = counting;
    a.stream = static_cast<cudaStream_t>(stream);
    bevpool_status st = cuda_status(launch_build_map(a));
    if (st != BEVPOOL_OK || !h_counts) return st;
    st = cuda_status(cudaMemcpyAsync(h_counts, d_counts, 3 * sizeof(int32_t), cudaMemcpyDeviceToHost, a.stream));
    if (st != BEVPOOL_OK) return st;
    st = cuda_status(cudaStreamSynchronize(a.stream));
    if (st != BEVPOOL_OK) return st;
    return h_counts[2] > 0 ? BEVPOOL_ERR_OUT_OF_RANGE : BEVPOOL_OK;
}

namespace {

// The size checks of a forward call (no device needed).
bevpool_status forward_sizes_ok(bevpool_dtype dtype, int32_t NC, int32_t D, int32_t H, int32_t W, int32_t C,
                                bool e4m3_out, int32_t n_points, int32_t n_intervals, int32_t n_cells) {
    if (dtype != BEVPOOL_F16 && dtype != BEVPOOL_E4M3 && dtype != BEVPOOL_NVFP4) return BEVPOOL_ERR_UNSUPPORTED;
    if (!forward_supported(static_cast<int>(dtype), C)) return BEVPOOL_ERR_UNSUPPORTED;
    if (e4m3_out && C % 16 != 0) return BEVPOOL_ERR_UNSUPPORTED;
    if (!frustum_ok(NC, D, H, W) || n_cells < 1) return BEVPOOL_ERR_INVALID_ARG;
    if (static_cast<int64_t>(n_cells) * C > INT32_MAX) return BEVPOOL_ERR_INVALID_ARG;
    const int64_t nf = static_cast<int64_t>(NC) * D * H * W;
    if (n_points < 0 || n_intervals < 0 || n_points > nf || n_intervals > n_points) return BEVPOOL_ERR_INVALID_ARG;
    return BEVPOOL_OK;
}

// The size checks and launch-shaping choices of a forward call, without its
// pointers: fills every size field of *a, the memory regime and the SM count.
bevpool_status forward_prepare(bevpool_dtype dtype, int32_t NC, int32_t D, int32_t H, int32_t W, int32_t C,
                               bool e4m3_out, int32_t n_points, int32_t n_intervals, bool counts_on_device,
                               int32_t n_cells, const DeviceInfo &info, ForwardArgs *a) {
    const bevpool_status st = forward_sizes_ok(dtype, NC, D, H, W, C, e4m3_out, n_points, n_intervals, n_cells);
    if (st != BEVPOOL_OK) return st;
    const int64_t nf = static_cast<int64_t>(NC) * D * H * W;
    *a = ForwardArgs{};
    a->n_points = n_points;
    a->n_intervals = n_intervals;
    a->n_cells = n_cells;
    a->C = C;
    a->n_depth = nf;
    a->n_feat_rows = NC * H * W;
    a->out_e4m3 = e4m3_out ? 1 : 0;
    // Memory regime (section "Classify the memory regime"): when the bytes the
    // forward touches do not fit comfortably in L2, stream the output past it.
    const int64_t eb = dtype == BEVPOOL_F16 ? 2 : 1;
    const int64_t ob = e4m3_out ? 1 : 2;
    const int64_t feat_bytes = dtype == BEVPOOL_NVFP4 ? static_cast<int64_t>(a->n_feat_rows) * (C / 2 + C / 16)
                                                      : static_cast<int64_t>(a->n_feat_rows) * C * eb;
    const int64_t footprint = static_cast<int64_t>(n_points) * 12 + static_cast<int64_t>(n_intervals) * 8 +
                              nf * eb + feat_bytes + static_cast<int64_t>(n_cells) * C * ob;
    a->streaming_stores = footprint > static_cast<int64_t>(info.l2_bytes) / 2 ? 1 : 0;
    // Device counts bounded by the whole frustum (what bevpool_pool_frame
    // passes) say nothing about the actual count: size the launch for one
    // resident wave and leave the choice of variant to the memory regime.
    a->loose_capacity = counts_on_device && n_points >= nf ? 1 : 0;
    a->sm_count = info.sm_count;
    return BEVPOOL_OK;
}

cudaError_t forward_dispatch(bevpool_dtype dtype, bool e4m3_out, const ForwardArgs &a) {
    if (dtype == BEVPOOL_NVFP4) return e4m3_out ? launch_forward_nvfp4_e4m3out(a) : launch_forward_nvfp4(a);
    if (e4m3_out) return dtype == BEVPOOL_F16 ? launch_forward_f16_e4m3out(a) : launch_forward_e4m3_e4m3out(a);
    return dtype == BEVPOOL_F16 ? launch_forward_f16(a) : launch_forward_e4m3(a);
}

// Shared body of the forward entry points (fp16 output, or E4M3 output codes
// of value / out_scale).
bevpool_status forward_impl(bevpool_dtype dtype, const void *depth, const void *feat, const void *feat_block,
                            int32_t NC, int32_t D, int32_t H, int32_t W, int32_t C, float depth_scale,
                            float feat_scale, bool e4m3_out,
                            float out_scale, const int32_t *ranks_depth, const int32_t *ranks_feat,
                            const int32_t *ranks_bev, const int32_t *interval_starts,
                            const int32_t *interval_lengths, int32_t n_points, int32_t n_intervals,
                            const int32_t *d_counts, int32_t n_cells, void *out, void *stream) {
    const bevpool_status sz = forward_sizes_ok(dtype, NC, D, H, W, C, e4m3_out, n_points, n_intervals, n_cells);
    if (sz != BEVPOOL_OK) return sz;
    if (dtype == BEVPOOL_NVFP4 && !feat_block) return BEVPOOL_ERR_INVALID_ARG;
    if (!depth || !feat || !out) return BEVPOOL_ERR_INVALID_ARG;
    if (n_points > 0 && (!ranks_depth || !ranks_feat || !ranks_bev)) return BEVPOOL_ERR_INVALID_ARG;
    if (n_intervals > 0 && (!interval_starts || !interval_lengths)) return BEVPOOL_ERR_INVALID_ARG;
    if (!aligned(feat, 16) || !aligned(out, 16)) return BEVPOOL_ERR_INVALID_ARG;
    if (dtype == BEVPOOL_F16 && !aligned(depth, 2)) return BEVPOOL_ERR_INVALID_ARG;
    const void *idx[] = {ranks_depth, ranks_feat, ranks_bev, interval_starts, interval_lengths, d_counts};
    for (const void *p : idx)
        if (p && !aligned(p, 4)) return BEVPOOL_ERR_INVALID_ARG;
    if (e4m3_out && !(std::isfinite(out_scale) && out_scale > 0.0f)) return BEVPOOL_ERR_INVALID_ARG;
    float scale = depth_scale * feat_scale;
    if (e4m3_out) scale /= out_scale;
    if (!std::isfinite(scale)) return BEVPOOL_ERR_INVALID_ARG;

    DeviceInfo info;
    if (!device_info(&info)) return BEVPOOL_ERR_CUDA;
    ForwardArgs a;
    const bevpool_status st = forward_prepare(dtype, NC, D, H, W, C, e4m3_out, n_points, n_intervals,
                                              d_counts != nullptr, n_cells, info, &a);
    if (st != BEVPOOL_OK) return st;
    a.depth = depth;
    a.feat = feat;
    a.feat_block = feat_block;
    a.ranks_depth = ranks_depth;
    a.ranks_feat = ranks_feat;
    a.ranks_bev = ranks_bev;
    a.interval_starts = interval_starts;
    a.interval_lengths = interval_lengths;
    a.d_counts = d_counts;
    a.scale = scale;
    a.out = out;
    a.stream = static_cast<cudaStream_t>(stream);
    a.plan_out = nullptr;
    return cuda_status(forward_dispatch(dtype, e4m3_out, a));
}

}  // namespace

bevpool_status bevpool_forward(bevpool_dtype dtype, const void *depth, const void *feat, int32_t NC, int32_t D,
                               int32_t H, int32_t W, int32_t C, float depth_scale, float feat_scale,
                               const int32_t *ranks_depth, const int32_t *ranks_feat, const int32_t *ranks_bev,
                               const int32_t *interval_starts, const int32_t *interval_lengths,
                               int32_t n_points, int32_t n_intervals, const int32_t *d_counts, int32_t n_cells,
                               void *out, void *stream) {
    if (dtype == BEVPOOL_NVFP4) return BEVPOOL_ERR_UNSUPPORTED;      // needs the block scales
    return forward_impl(dtype, depth, feat, nullptr, NC, D, H, W, C, depth_scale, feat_scale, false, 0.0f, ranks_depth,
                        ranks_feat, ranks_bev, interval_starts, interval_lengths, n_points, n_intervals, d_counts,
                        n_cells, out, stream);
}

bevpool_status bevpool_forward_e4m3_out(bevpool_dtype dtype, const void *depth, const void *feat, int32_t NC,
                                        int32_t D, int32_t H, int32_t W, int32_t C, float depth_scale,
                                        float feat_scale, float out_scale, const int32_t *ranks_depth,
                                        const int32_t *ranks_feat, const int32_t *ranks_bev,
                                        const int32_t *interval_starts, const int32_t *interval_lengths,
                                        int32_t n_points, int32_t n_intervals, const int32_t *d_counts,
                                        int32_t n_cells, void *out, void *stream) {
    if (dtype == BEVPOOL_NVFP4) return BEVPOOL_ERR_UNSUPPORTED;      // needs the block scales
    return forward_impl(dtype, depth, feat, nullptr, NC, D, H, W, C, depth_scale, feat_scale, true, out_scale,
                        ranks_depth,
                        ranks_feat, ranks_bev, interval_starts, interval_lengths, n_points, n_intervals, d_counts,
                        n_cells, out, stream);
}

bevpool_status bevpool_forward_nvfp4(const void *depth, const void *feat, const void *feat_block, int32_t NC,
                                     int32_t D, int32_t H, int32_t W, int32_t C, float depth_scale,
                                     float feat_scale, bevpool_dtype out_dtype, float out_scale,
                                     const int32_t *ranks_depth, const int32_t *ranks_feat,
                                     const int32_t *ranks_bev, const int32_t *interval_starts,
                                     const int32_t *interval_lengths, int32_t n_points, int32_t n_intervals,
                                     const int32_t *d_counts, int32_t n_cells, void *out, void *stream) {
    if (out_dtype != BEVPOOL_F16 && out_dtype != BEVPOOL_E4M3) return BEVPOOL_ERR_UNSUPPORTED;
    return forward_impl(BEVPOOL_NVFP4, depth, feat, feat_block, NC, D, H, W, C, depth_scale, feat_scale,
                        out_dtype == BEVPOOL_E4M3, out_scale, ranks_depth, ranks_feat, ranks_bev, interval_starts,
                        interval_lengths, n_points, n_intervals, d_counts, n_cells, out, stream);
}

bevpool_status bevpool_forward_plan(bevpool_dtype dtype, int32_t C, int32_t e4m3_out, int32_t NC, int32_t D,
                                    int32_t H, int32_t W, int32_t n_points, int32_t n_intervals,
                                    int32_t counts_on_device, int32_t n_cells, int32_t sm_count, int64_t l2_bytes,
                                    int32_t *plan) {
    if (!plan) return BEVPOOL_ERR_INVALID_ARG;
    const bevpool_status sz = forward_sizes_ok(dtype, NC, D, H, W, C, e4m3_out != 0, n_points, n_intervals, n_cells);
    if (sz != BEVPOOL_OK) return sz;
    DeviceInfo info;
    if (sm_count > 0 && l2_bytes > 0) {
        if (l2_bytes > INT32_MAX) return BEVPOOL_ERR_INVALID_ARG;
        info.sm_count = sm_count;
        info.l2_bytes = static_cast<int>(l2_bytes);
    } else if (!device_info(&info)) {
        return BEVPOOL_ERR_CUDA;
    }
    ForwardArgs a;
    const bevpool_status st = forward_prepare(dtype, NC, D, H, W, C, e4m3_out != 0, n_points, n_intervals,
                                              counts_on_device != 0, n_cells, info, &a);
    if (st != BEVPOOL_OK) return st;
    ForwardPlan pl;
    a.plan_out = &pl;
    const bevpool_status ds = cuda_status(forward_dispatch(dtype, e4m3_out != 0, a));
    if (ds != BEVPOOL_OK) return ds;
    const int32_t fields[] = {pl.variant, pl.ctas_per_sm, pl.owners, pl.batch, pl.round, pl.n_compute,
                              pl.fill_cells, pl.n_fill, a.streaming_stores};
    for (int k = 0; k < 9; ++k) plan[k] = fields[k];
    return BEVPOOL_OK;
}

bevpool_status bevpool_pool_frame(const int32_t *cell_ids, int32_t NC, int32_t D, int32_t H, int32_t W,
                                  int32_t n_cells, bevpool_dtype dtype, const void *depth, const void *feat,
                                  int32_t C, float depth_scale, float feat_scale, int32_t *ranks_depth,
                                  int32_t *ranks_feat, int32_t *ranks_bev, int32_t *interval_starts,
                                  int32_t *interval_lengths, int32_t *d_counts, void *workspace,
                                  size_t workspace_bytes, void *out, void *stream) {
    // Everything the two calls would reject is checked before either enqueues work.
    if (dtype != BEVPOOL_F16 && dtype != BEVPOOL_E4M3) return BEVPOOL_ERR_UNSUPPORTED;
    if (!forward_supported(static_cast<int>(dtype), C)) return BEVPOOL_ERR_UNSUPPORTED;
    if (!frustum_ok(NC, D, H, W) || n_cells < 1) return BEVPOOL_ERR_INVALID_ARG;
    if (static_cast<int64_t>(n_cells) * C > INT32_MAX) return BEVPOOL_ERR_INVALID_ARG;
    if (!depth || !feat || !out || !aligned(feat, 16) || !aligned(out, 16)) return BEVPOOL_ERR_INVALID_ARG;
    if (dtype == BEVPOOL_F16 && !aligned(depth, 2)) return BEVPOOL_ERR_INVALID_ARG;
    if (!std::isfinite(depth_scale * feat_scale)) return BEVPOOL_ERR_INVALID_ARG;
    bevpool_status st = bevpool_build_map(cell_ids, NC, D, H, W, n_cells, ranks_depth, ranks_feat, ranks_bev,
                                          interval_starts, interval_lengths, d_counts, nullptr, workspace,
                                          workspace_bytes, stream);
    if (st != BEVPOOL_OK) return st;
    const int64_t nf = static_cast<int64_t>(NC) * D * H * W;
    const int32_t cap_points = static_cast<int32_t>(nf);
    const int32_t cap_intervals = static_cast<int32_t>(nf < n_cells ? nf : n_cells);
    return bevpool_forward(dtype, depth, feat, NC, D, H, W, C, depth_scale, feat_scale, ranks_depth, ranks_feat,
                           ranks_bev, interval_starts, interval_lengths, cap_points, cap_intervals, d_counts,
                           n_cells, out, stream);
}

bevpool_status bevpool_validate_map(const int32_t *ranks_depth, const int32_t *ranks_feat, const int32_t *ranks_bev,
                                    const int32_t *interval_starts, const int32_t *interval_lengths,
                                    int32_t n_points, int32_t n_intervals, int32_t NC, int32_t D, int32_t H,
                                    int32_t W, int32_t n_cells, int32_t *d_result, int32_t *h_result,
                                    void *stream) {
    if (!frustum_ok(NC, D, H, W) || n_cells < 1 || n_points < 0 || n_intervals < 0 || !d_result)
        return BEVPOOL_ERR_INVALID_ARG;
    if (n_points > 0 && (!ranks_depth || !ranks_feat || !ranks_bev)) return BEVPOOL_ERR_INVALID_ARG;
    if (n_intervals > 0 && (!interval_starts || !interval_lengths)) return BEVPOOL_ERR_INVALID_ARG;
    const int64_t nf = static_cast<int64_t>(NC) * D * H * W;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bevpool_status st = cuda_status(launch_validate_map(ranks_depth, ranks_feat, ranks_bev, interval_starts,
                                                        interval_lengths, n_points, n_intervals, nf, NC * H * W,
                                                        n_cells, d_result, s));
    if (st != BEVPOOL_OK || !h_result) return st;
    st = cuda_status(cudaMemcpyAsync(h_result, d_result, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    if (st != BEVPOOL_OK) return st;
    st = cuda_status(cudaStreamSynchronize(s));
    if (st != BEVPOOL_OK) return st;
    return *h_result ? BEVPOOL_ERR_OUT_OF_RANGE : BEVPOOL_OK;
}

}  // extern "C"
