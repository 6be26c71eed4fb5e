/*
 * bevpool.h -- C ABI of libbevpool, GB300 (sm_103a) BEV pooling.
 *
 * BEV pooling is the depth-weighted scatter-reduce of "Accelerating BEV
 * Pooling on NVIDIA GPUs for Physical AI Applications" (NVIDIA technical
 * blog), section "Eliminate redundant scatter traffic":
 *
 *     out[ranks_bev[t], c] += depth[ranks_depth[t]] * feat[ranks_feat[t], c]
 *
 * over every scatter point t of a five-array INT32 scatter map
 * (ranks_depth, ranks_feat, ranks_bev, interval_starts, interval_lengths).
 * The map is prepared ahead of the forward (section "Implement
 * interval-owned scatter-reduce"); each interval is the run of points that
 * share one BEV cell and is reduced by one owner that writes the cell once.
 *
 * Conventions shared by every entry point:
 *   - Pointers marked "device" must point to device memory of the current
 *     CUDA device; pointers marked "host" to host memory.  The library
 *     allocates nothing: the caller owns every buffer, including scratch
 *     ("workspace"), which it sizes with the matching *_workspace_size call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on it and returns, except
 *     where a host output pointer is given: then the call synchronises the
 *     stream before returning.
 *   - Errors are returned as bevpool_status; the library never aborts,
 *     traps or prints.  Arguments are checked on the host before any work
 *     is enqueued; on an error nothing is enqueued.  A CUDA launch error is
 *     returned as BEVPOOL_ERR_CUDA and cleared from the runtime's
 *     last-error slot.
 *   - Layouts (frustum point index p = ((nc*D + d)*H + h)*W + w):
 *       cell_ids [NC*D*H*W] int32, -1 = point dropped, else in [0, n_cells)
 *       depth    [NC, D, H, W]  (element p belongs to frustum point p)
 *       feat     [NC, H, W, C]  (row r = (nc*H + h)*W + w holds C channels;
 *                                NVFP4 rows: see bevpool_forward_nvfp4)
 *       out      [n_cells, C]   fp16 (IEEE binary16), row-major (E4M3 codes
 *                                from the calls with an E4M3 output)
 *   - Sizes: NC*D*H*W < 2^31, n_cells*C < 2^31.
 *   - Calls on different streams may run concurrently only if they share no
 *     output or workspace buffer.
 */
#ifndef BEVPOOL_H
#define BEVPOOL_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BEVPOOL_API __attribute__((visibility("default")))
#else
#define BEVPOOL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bevpool_status {
    BEVPOOL_OK = 0,
    BEVPOOL_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad alignment      */
    BEVPOOL_ERR_OUT_OF_RANGE = 2,  /* a cell id or map entry outside its range   */
    BEVPOOL_ERR_UNSUPPORTED = 3,   /* channel count / dtype with no kernel       */
    BEVPOOL_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required */
    BEVPOOL_ERR_CUDA = 5           /* a CUDA runtime call or launch failed       */
} bevpool_status;

typedef enum bevpool_dtype {
    BEVPOOL_F16 = 0,   /* depth and feat are IEEE binary16                         */
    BEVPOOL_E4M3 = 1,  /* depth and feat are OCP FP8 E4M3 codes, one scale each    */
    BEVPOOL_NVFP4 = 2  /* feat NVFP4 (E2M1 + E4M3 block scales), depth E4M3:
                          bevpool_forward_nvfp4 only                             */
} bevpool_dtype;

/* Human-readable name of a status code (static string, never NULL). */
BEVPOOL_API const char *bevpool_status_string(bevpool_status status);

/* Library version as major*10000 + minor*100 + patch. */
BEVPOOL_API int32_t bevpool_version(void);

/* Number of kernels this library has launched in this process so far
 * (all devices, all streams).  Used to count launches in a timed region. */
BEVPOOL_API int64_t bevpool_kernel_launches(void);

/* Whether channel count C has a compiled forward kernel for dtype (1 / 0);
 * for BEVPOOL_NVFP4 it answers for bevpool_forward_nvfp4. */
BEVPOOL_API int32_t bevpool_forward_supported(bevpool_dtype dtype, int32_t C);

/* The launch plan a forward call with these sizes would use (no kernel is
 * launched and no pointer is needed).  The plan is the library's own launch
 * shaping, not a step of the pages' method; it is exported so that its rules
 * can be checked without a GPU.
 *   dtype, C, e4m3_out  as for bevpool_forward (e4m3_out != 0:
 *                       bevpool_forward_e4m3_out; BEVPOOL_NVFP4 stands for
 *                       bevpool_forward_nvfp4);
 *   NC, D, H, W,
 *   n_points,
 *   n_intervals,
 *   n_cells             as for bevpool_forward;
 *   counts_on_device    non-zero when the call passes d_counts (then n_points
 *                       and n_intervals are capacities);
 *   sm_count, l2_bytes  the GPU to plan for; when either is <= 0, the current
 *                       device (which then needs a GPU);
 *   plan                host int32[9], filled with {variant (0 default,
 *                       1 lean, 2 short intervals, 3 lean with short
 *                       intervals), compute CTAs per SM, owners per compute
 *                       CTA, points in flight per owner, points per staged
 *                       round, compute CTAs, cells per fill CTA, fill CTAs,
 *                       streaming output stores (1: the output is written
 *                       past the L2)}.
 * Returns what bevpool_forward would for the same sizes
 * (BEVPOOL_ERR_UNSUPPORTED / BEVPOOL_ERR_INVALID_ARG), BEVPOOL_ERR_INVALID_ARG
 * for a null plan. */
BEVPOOL_API bevpool_status bevpool_forward_plan(bevpool_dtype dtype, int32_t C, int32_t e4m3_out, int32_t NC,
                                                int32_t D, int32_t H, int32_t W, int32_t n_points,
                                                int32_t n_intervals, int32_t counts_on_device, int32_t n_cells,
                                                int32_t sm_count, int64_t l2_bytes, int32_t *plan);

/*
 * Bytes of device workspace bevpool_build_map needs for a frustum of
 * n_frustum = NC*D*H*W points and a grid of n_cells cells.  Returns 0 for
 * invalid sizes.
 */
BEVPOOL_API size_t bevpool_build_map_workspace_size(int64_t n_frustum, int32_t n_cells);

/*
 * Build the five-array scatter map from per-frustum-point BEV cell ids
 * (the map the section "Implement interval-owned scatter-reduce" says is
 * prepared ahead).  Bit-exact and deterministic: the kept points are sorted
 * by (cell, p) -- a stable sort of frustum order by cell -- and
 *     ranks_bev[t]   = cell of the t-th sorted point
 *     ranks_depth[t] = its frustum index p
 *     ranks_feat[t]  = nc*H*W + h*W + w   (the only integer division, done here)
 * Intervals are the maximal runs of equal ranks_bev, in ascending cell order:
 *     interval_starts[i], interval_lengths[i] (>= 1), contiguous, summing to n.
 *
 *   cell_ids          device, [NC*D*H*W] int32; -1 drops the point.
 *   NC, D, H, W       frustum dimensions (all >= 1).
 *   n_cells           number of BEV cells (>= 1).
 *   ranks_*           device, capacity NC*D*H*W int32 each (n entries written).
 *   interval_*        device, capacity min(NC*D*H*W, n_cells) int32 each.
 *   d_counts          device, int32[3]: {n_points, n_intervals, n_invalid},
 *                     written by the enqueued work.  n_invalid counts ids
 *                     that are neither -1 nor in [0, n_cells); such points are
 *                     treated as dropped.
 *   h_counts          host, int32[3] or NULL.  If non-NULL the call copies
 *                     d_counts here, synchronises `stream`, and returns
 *                     BEVPOOL_ERR_OUT_OF_RANGE when n_invalid > 0.
 *   workspace         device scratch of at least
 *                     bevpool_build_map_workspace_size(NC*D*H*W, n_cells)
 *                     bytes, 256-byte aligned; contents need no initialisation
 *                     and are clobbered.
 */
BEVPOOL_API bevpool_status bevpool_build_map(const int32_t *cell_ids, int32_t NC, int32_t D, int32_t H,
                                 int32_t W, int32_t n_cells, int32_t *ranks_depth,
                                 int32_t *ranks_feat, int32_t *ranks_bev,
                                 int32_t *interval_starts, int32_t *interval_lengths,
                                 int32_t *d_counts, int32_t *h_counts, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * bevpool_build_map without a workspace argument, for callers that may not
 * allocate device memory (for example an inference-engine plugin whose
 * enqueue step must not allocate, or real-time code that forbids allocation
 * after start-up).  The pages have no counterpart to this entry point: it is
 * an interface convenience of this library.
 *
 * It runs the same kernels and gives the same results as bevpool_build_map,
 * with the same arguments and outputs, but its scratch is a fixed array of
 * BEVPOOL_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU
 * that loads the library holds until the process exits.  It calls no
 * allocating routine.
 *   - NC*D*H*W must not exceed BEVPOOL_NOALLOC_MAX_FRUSTUM; larger frusta
 *     return BEVPOOL_ERR_WORKSPACE and enqueue nothing.
 *   - All calls on a device share the array: calls whose work may overlap on
 *     the GPU (other streams, other host threads) race and must be ordered by
 *     the caller.  Nothing in the array needs clearing between calls.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress), which cannot happen during stream capture: make
 *     the first call on a device outside any capture.  A call after
 *     cudaDeviceReset finds the device's context changed and looks the
 *     address up again, so the first call after a reset must also be made
 *     outside any capture.
 *   - Under lazy module loading (the CUDA default) that first look-up is
 *     what commits the array's memory on the device, so it is the one call
 *     that can fail for lack of device memory (BEVPOOL_ERR_CUDA).  Callers
 *     that must not fail later make one call at start-up.
 */
#define BEVPOOL_NOALLOC_MAX_FRUSTUM (1 << 21)
#define BEVPOOL_NOALLOC_SCRATCH_BYTES (37u * 1024u * 1024u)
BEVPOOL_API bevpool_status bevpool_build_map_noalloc(const int32_t *cell_ids, int32_t NC, int32_t D, int32_t H,
                                         int32_t W, int32_t n_cells, int32_t *ranks_depth,
                                         int32_t *ranks_feat, int32_t *ranks_bev,
                                         int32_t *interval_starts, int32_t *interval_lengths,
                                         int32_t *d_counts, int32_t *h_counts, void *stream);

/*
 * Interval-owned forward (sections "Eliminate redundant scatter traffic"
 * and "Implement interval-owned scatter-reduce"): for every interval i,
 *     out[ranks_bev[s], c] = scale * sum_{t in [s, s+len)}
 *                            depth[ranks_depth[t]] * feat[ranks_feat[t], c]
 * with s = interval_starts[i], len = interval_lengths[i] and
 * scale = depth_scale * feat_scale, accumulated in FP32 and rounded once to
 * fp16 (round to nearest even).  Every one of the n_cells rows of `out` is
 * written exactly once; rows no interval names are written as zeros.  No
 * atomics: calls with identical arguments give bit-identical results (the
 * work split, and so the FP32 summation order inside an interval that two
 * lane groups share, depends on n_points and the device's SM count).
 *
 *   dtype             BEVPOOL_F16 or BEVPOOL_E4M3 (depth and feat alike).
 *   depth             device, [NC, D, H, W] elements of dtype.
 *   feat              device, [NC*H*W, C] elements of dtype, 16-byte aligned.
 *   NC, D, H, W       frustum dimensions; bound the indices in the map.
 *   C                 channels; bevpool_forward_supported(dtype, C) must be 1.
 *   depth_scale,
 *   feat_scale        multipliers of the E4M3 code values (use 1 for F16).
 *   ranks_depth,
 *   ranks_feat,
 *   ranks_bev         device, [n_points] int32 (as built by bevpool_build_map).
 *   interval_starts,
 *   interval_lengths  device, [n_intervals] int32.
 *   n_points,
 *   n_intervals       host counts.  If d_counts is non-NULL they are
 *                     capacities instead and the counts are read on the
 *                     device from d_counts[0] and d_counts[1] (clamped to the
 *                     capacities), so a forward can follow bevpool_build_map
 *                     on the same stream without a host synchronisation.
 *   d_counts          device int32[>=2] or NULL.
 *   n_cells           rows of out.
 *   out               device, [n_cells, C] fp16, 16-byte aligned; fully
 *                     overwritten.
 *
 * The map is trusted for its ordering: ranks_bev ascending and the
 * intervals its maximal runs, as bevpool_build_map writes them (the kernel
 * splits work at interval starts and ends an interval where ranks_bev
 * changes).  Indices are still bounds-checked on the device: a point whose
 * ranks_depth / ranks_feat lies outside the tensors contributes nothing, a
 * cell outside [0, n_cells) is not written, and nothing outside
 * [0, n_points) of the map arrays is read.  Use bevpool_validate_map to
 * check a map.
 */
BEVPOOL_API bevpool_status bevpool_forward(bevpool_dtype dtype, const void *depth, const void *feat,
                               int32_t NC, int32_t D, int32_t H, int32_t W, int32_t C,
                               float depth_scale, float feat_scale, const int32_t *ranks_depth,
                               const int32_t *ranks_feat, const int32_t *ranks_bev,
                               const int32_t *interval_starts, const int32_t *interval_lengths,
                               int32_t n_points, int32_t n_intervals, const int32_t *d_counts,
                               int32_t n_cells, void *out, void *stream);

/*
 * The forward with an FP8 output: the pages' FP8 path halves output bytes as
 * well as feature bytes (section "Eliminate redundant scatter traffic",
 * Figure 4; section "Map the algorithm to hardware" keeps depth and output
 * in FP8).  Same arguments and semantics as bevpool_forward, except that
 * every output value v (including the input scales) is stored as the OCP
 * E4M3 code nearest to v / out_scale, computed from the FP32 sum (round to
 * nearest even, magnitudes above 448 saturate to +-448); cells no interval
 * names get the code 0x00.
 *
 *   out_scale         per-tensor output scale, finite and > 0 (e.g. from a
 *                     calibration: max |output| / 448).
 *   out               device, [n_cells, C] uint8 E4M3 codes, 16-byte
 *                     aligned; fully overwritten.
 *
 * Requires C % 16 == 0 (rows of whole 16-byte vectors) besides
 * bevpool_forward_supported(dtype, C); other C give BEVPOOL_ERR_UNSUPPORTED.
 * A non-positive or non-finite out_scale gives BEVPOOL_ERR_INVALID_ARG.
 */
BEVPOOL_API bevpool_status bevpool_forward_e4m3_out(bevpool_dtype dtype, const void *depth, const void *feat,
                                        int32_t NC, int32_t D, int32_t H, int32_t W, int32_t C,
                                        float depth_scale, float feat_scale, float out_scale,
                                        const int32_t *ranks_depth, const int32_t *ranks_feat,
                                        const int32_t *ranks_bev, const int32_t *interval_starts,
                                        const int32_t *interval_lengths, int32_t n_points,
                                        int32_t n_intervals, const int32_t *d_counts, int32_t n_cells,
                                        void *out, void *stream);

/*
 * The forward with NVFP4 features, the experiment of section "Map the
 * algorithm to hardware": camera features stored as OCP E2M1 (4-bit)
 * elements with one E4M3 scale per 16 elements, depth kept in E4M3.  Feature
 * value c of row r:
 *     e2m1(nibble c of feat row r) * e4m3(feat_block[r * C/16 + c/16]) * feat_scale
 * with element 2i in the low nibble of byte i (a row is C/2 bytes); depth
 * value = e4m3(depth[p]) * depth_scale.  The sum and the rest of the
 * semantics are those of bevpool_forward; out_dtype BEVPOOL_F16 stores fp16
 * rows, BEVPOOL_E4M3 stores E4M3 codes of value / out_scale as
 * bevpool_forward_e4m3_out does (out_scale is ignored for fp16).
 *
 *   depth             device, [NC, D, H, W] E4M3 codes.
 *   feat              device, [NC*H*W, C/2] bytes of E2M1 pairs, 16-byte aligned.
 *   feat_block        device, [NC*H*W, C/16] E4M3 block scales.
 *   C                 64, 80, 96, 128, 160, 192 or 256 (one 16-element block
 *                     per lane, at least four lanes per row).
 *
 * Each depth code times each block scale is formed in fp16 (exact for E4M3
 * values), so their product must stay within the fp16 range (|product| <=
 * 65504); it does when the depth codes lie in [-1, 1], as when depth_scale =
 * max|depth|.  The pages report this format slower than FP8 for the
 * scatter-reduce; it is here to confirm that on this GPU.
 */
BEVPOOL_API bevpool_status bevpool_forward_nvfp4(const void *depth, const void *feat, const void *feat_block,
                                     int32_t NC, int32_t D, int32_t H, int32_t W, int32_t C,
                                     float depth_scale, float feat_scale, bevpool_dtype out_dtype,
                                     float out_scale, const int32_t *ranks_depth, const int32_t *ranks_feat,
                                     const int32_t *ranks_bev, const int32_t *interval_starts,
                                     const int32_t *interval_lengths, int32_t n_points, int32_t n_intervals,
                                     const int32_t *d_counts, int32_t n_cells, void *out, void *stream);

/*
 * One frame with its own geometry: bevpool_build_map (no host
 * synchronisation) followed on the same stream by bevpool_forward reading
 * the counts on the device, for pipelines whose cell ids change every frame
 * (the pages prepare the map ahead, section "Implement interval-owned
 * scatter-reduce"; this puts the build next to the forward in one call).
 * Nothing is copied to the host, so the call can be captured in a CUDA graph
 * and replayed with new cell_ids / depth / feat in the same buffers.
 *
 * Arguments are those of bevpool_build_map (the five map arrays with
 * capacity NC*D*H*W, d_counts, the workspace) and of bevpool_forward
 * (dtype, depth, feat, C, the scales, out [n_cells, C] fp16).  The map is
 * left in the arrays for later use; d_counts[2] counts invalid cell ids
 * (treated as dropped).  The result is bit-identical to the two calls made
 * one after the other with the same capacities (NC*D*H*W points and
 * min(NC*D*H*W, n_cells) intervals).
 */
BEVPOOL_API bevpool_status bevpool_pool_frame(const int32_t *cell_ids, int32_t NC, int32_t D, int32_t H,
                                  int32_t W, int32_t n_cells, bevpool_dtype dtype, const void *depth,
                                  const void *feat, int32_t C, float depth_scale, float feat_scale,
                                  int32_t *ranks_depth, int32_t *ranks_feat, int32_t *ranks_bev,
                                  int32_t *interval_starts, int32_t *interval_lengths, int32_t *d_counts,
                                  void *workspace, size_t workspace_bytes, void *out, void *stream);

/*
 * Check a scatter map on the device (debug aid; the five-array map of the
 * section "Eliminate redundant scatter traffic" with the interval structure
 * of the section "Implement interval-owned scatter-reduce").  Writes to
 * d_result (device int32[1]) a bit set of the violations found, 0 if none:
 *     1  interval_starts[0] != 0 or starts not contiguous (start[i+1] != start[i]+len[i])
 *     2  an interval length < 1, or the lengths do not sum to n_points
 *     4  ranks_bev differs inside an interval, or interval cells not strictly
 *        increasing
 *     8  a ranks_bev entry outside [0, n_cells)
 *    16  a ranks_depth entry outside [0, NC*D*H*W)
 *    32  a ranks_feat entry outside [0, NC*H*W)
 * h_result: host int32[1] or NULL; if non-NULL the call synchronises the
 * stream, copies the bit set there and returns BEVPOOL_ERR_OUT_OF_RANGE when
 * it is non-zero.  n_points / n_intervals are host counts.
 */
BEVPOOL_API bevpool_status bevpool_validate_map(const int32_t *ranks_depth, const int32_t *ranks_feat,
                                    const int32_t *ranks_bev, const int32_t *interval_starts,
                                    const int32_t *interval_lengths, int32_t n_points,
                                    int32_t n_intervals, int32_t NC, int32_t D, int32_t H,
                                    int32_t W, int32_t n_cells, int32_t *d_result,
                                    int32_t *h_result, void *stream);

/*
 * L2 streaming probe (a measurement helper, not part of the pooling path):
 * the bandwidth at which the SMs read, write or copy a buffer resident in L2,
 * the denominator of the forward's roofline when its working set fits in L2
 * (the pages' large-L2 regime, section "Optimize for large L2 caches").
 * buf: device, 16-byte aligned; bytes at most 2^32.  One launch on `stream`;
 * time it with events around the call, after one call that brings the
 * buffer into L2.
 *
 * mode = 0 (read): reads the `bytes` of buf (a multiple of 16) `passes` times
 *   with 16-byte L2-only loads and adds the sum of its 32-bit words (mod 2^32,
 *   once per pass) to *d_sink (device uint32 the caller zeroes first), so
 *   every byte is known to have been read.
 * mode = 1 (write): writes buf (a multiple of 16 bytes) `passes` times with
 *   16-byte stores; afterwards 32-bit word k holds k ^ ((passes - 1) * 0x9E3779B9)
 *   (mod 2^32).
 * mode = 2 (copy): bytes a multiple of 32; each pass reads the first half and
 *   writes the second half; afterwards word k of the second half holds word k
 *   of the first half ^ ((passes - 1) * 0x9E3779B9).  A pass moves `bytes`
 *   (half read, half written), the convention of a STREAM copy.
 * d_sink may be NULL for modes 1 and 2.  Returns BEVPOOL_ERR_INVALID_ARG for
 * a bad argument (nothing launched), BEVPOOL_ERR_CUDA if the launch fails.
 */
BEVPOOL_API bevpool_status bevpool_probe_l2(int32_t mode, void *buf, size_t bytes, int32_t passes,
                                uint32_t *d_sink, void *stream);

/*
 * Gather probe (a measurement helper, not part of the pooling path): the
 * forward's feature-row gather alone, over a caller's row list (normally a
 * map's ranks_feat), in the forward's lane layout: owners of row_bytes / 16
 * lanes, one 16-byte vector a lane, eight rows in flight per owner, each
 * owner a contiguous equal share of the points; no depth, no accumulation
 * into output rows, no stores.  It bounds the rate the forward's walk can
 * reach on the same rows (the gather of "Optimize for large L2 caches").
 *   feat         device, 16-byte aligned, n_rows rows of row_bytes bytes;
 *   row_bytes    a multiple of 16 in [16, 512];
 *   rows         device int32[n_points]; rows outside [0, n_rows) are skipped;
 *   ctas_per_sm  256-thread CTAs per SM in the launch, 1..8;
 *   d_sink       device uint32 the caller zeroes first; the launch adds the
 *                sum (mod 2^32) of the 32-bit words of every gathered row.
 *                NULL: the timing mode (the sum is formed but not written, so
 *                no atomic or barrier enters the measured time).
 * One launch on `stream`.  Returns BEVPOOL_ERR_INVALID_ARG for a bad
 * argument (nothing launched), BEVPOOL_ERR_CUDA if the launch fails.
 */
BEVPOOL_API bevpool_status bevpool_probe_gather(const void *feat, int32_t n_rows, int32_t row_bytes,
                                                const int32_t *rows, int32_t n_points, int32_t ctas_per_sm,
                                                uint32_t *d_sink, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BEVPOOL_H */
