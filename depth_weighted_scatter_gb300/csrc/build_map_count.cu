// build_map_count.cu -- scatter-map construction by counting sort, for grids
// of at most kCountingMaxCells cells (every BEV grid in practice).
//
// Produces exactly the map of build_map.cu's radix path (the five INT32
// arrays of "Accelerating BEV Pooling on NVIDIA GPUs for Physical AI
// Applications", section "Eliminate redundant scatter traffic", kept points
// sorted by (cell, p)), with seven launches and far more parallelism:
//
//   1. k_zero        clear the per-cell counters;
//   2. k_count_cells one atomic increment per kept frustum point;
//   3. k_tile_sums   per 1024-cell tile: points and non-empty cells;
//   4. k_offsets     exclusive scan of the counts (each CTA adds up the tile
//                    sums before it), giving every cell's first position; the
//                    non-empty cells are the intervals, so interval_starts /
//                    interval_lengths are written here too;
//   5. k_scatter     each kept point takes the next slot of its cell with an
//                    atomic increment; inside a cell the order is arbitrary;
//   6. k_sort_runs   restore the stable order inside every interval (ascending
//                    frustum index p) and write ranks_depth / ranks_feat /
//                    ranks_bev: one thread sorts an interval of up to 16
//                    points in registers (a bitonic network); longer
//                    intervals go to two work lists;
//   7. k_sort_lists  persistent CTAs drain the lists: a warp ranks one
//                    32-point slice of an interval of up to 8192 points by
//                    counting (rank = number of smaller values in the whole
//                    interval), so the slices of a long interval run on many
//                    warps at once; beyond 8192 points a CTA rebuilds the run
//                    by scanning the frustum in order for that cell.
//
// The result is independent of the order the atomics happened in: counts
// are exact and step 6 puts every interval in ascending p.  No kernel waits
// on another CTA.
#include <climits>

#include "bevpool_internal.cuh"

namespace bevpool {
namespace {

constexpr int kItems = 16;
constexpr int kTile = kThreads * kItems;        // 4096 frustum points per CTA tile
constexpr int kCellItems = 4;
constexpr int kCellTile = kThreads * kCellItems; // 1024 cells per scan tile
constexpr int kThreadSortMax = 16;              // longest interval one thread sorts in registers
constexpr int kSliceSortMax = 8192;             // longest interval ranked in 32-point slices (at most 256 slices)
static_assert(kCountingMaxCells <= (1 << 24), "a slice entry holds the interval index in 24 bits");
// Slices replace a warp ranking a whole interval of up to 128 points and a
// CTA sorting a longer one in shared memory (bitonic; a run of 464 points
// held one CTA for 12 us, the end of the list pass).  Measured, map build
// with L2 flushed: canonical 28.8 -> 26.8 us, BEVDet 42.5 -> 35.0, Table-1
// large 47.9 -> 41.7, very large 86.2 -> 81.8, DRAM batch unchanged (no run
// over 16 points).
#ifndef BEVPOOL_MAP_LIST_CTAS_PER_SM
#define BEVPOOL_MAP_LIST_CTAS_PER_SM 8           // the list pass's residency (32 registers, no shared buffer)
#endif

struct CountWs {
    int32_t *count;       // [n_cells]  points per cell
    int32_t *offset;      // [n_cells]  first position of each cell (then the scatter cursor)
    int32_t *tmp_p;       // [n_frustum] frustum indices grouped by cell, unordered inside a cell
    int32_t *icell;       // [min(n_frustum, n_cells)] cell of each interval
    int32_t *tile_cnt;    // [cell tiles]
    int32_t *tile_nz;     // [cell tiles]
    int32_t *invalid;     // [1]
    int32_t *lists;       // [2]: entries in slice_list, long_list
    int32_t *slice_list;  // [n_frustum / 16 + 1] (interval << 8 | slice) of intervals of 17..kSliceSortMax points
    int32_t *long_list;   // [min(n_frustum, n_cells)] intervals of more than kSliceSortMax points
};

size_t carve(void *base, int64_t nf, int32_t n_cells, CountWs *ws) {
    const int64_t nct = div_up(n_cells, kCellTile);
    const int64_t ni = nf < n_cells ? nf : n_cells;
    size_t off = 0;
    auto take = [&](int64_t count) -> int32_t * {
        int32_t *p = base ? reinterpret_cast<int32_t *>(static_cast<char *>(base) + off) : nullptr;
        off = align_up(off + static_cast<size_t>(count) * sizeof(int32_t), 256);
        return p;
    };
    CountWs w;
    w.count = take(n_cells);
    w.offset = take(n_cells);
    w.tmp_p = take(nf);
    w.icell = take(ni);
    w.tile_cnt = take(nct);
    w.tile_nz = take(nct);
    w.invalid = take(1);
    w.lists = take(2);
    // an interval of L > 16 points has ceil(L / 32) <= L / 16 slices, so all
    // of them together have at most n_frustum / 16
    w.slice_list = take(nf / 16 + 1);
    w.long_list = take(ni);
    if (ws) *ws = w;
    return off;
}

__global__ void __launch_bounds__(kThreads) k_zero(int32_t *__restrict__ count, int32_t n_cells,
                                                   int32_t *__restrict__ invalid, int32_t *__restrict__ lists) {
    grid_dep_wait();
    grid_dep_allow();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n_cells; i += stride)
        count[i] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *invalid = 0;
        lists[0] = 0;
        lists[1] = 0;
    }
}

// The kItems cell ids of thread t of tile b: frustum points
// b*kTile + t*kItems + j (blocked, so one thread's ids are contiguous and can
// be loaded as int4 when the array is 16-byte aligned); -2 past the end.
__device__ __forceinline__ void load_block(const int32_t *__restrict__ cell_ids, int64_t nf, bool vec,
                                           int64_t first, int *c) {
    if (vec && first + kItems <= nf) {
        const int4 *p = reinterpret_cast<const int4 *>(cell_ids + first);
#pragma unroll
        for (int q = 0; q < kItems / 4; ++q) {
            const int4 v = __ldg(p + q);
            c[4 * q] = v.x; c[4 * q + 1] = v.y; c[4 * q + 2] = v.z; c[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < kItems; ++j) c[j] = first + j < nf ? __ldg(cell_ids + first + j) : -2;
    }
}

__global__ void __launch_bounds__(kThreads)
k_count_cells(const int32_t *__restrict__ cell_ids, int64_t nf, int32_t n_cells, bool vec,
              int32_t *__restrict__ count, int32_t *__restrict__ invalid) {
    __shared__ long long red[kWarps];
    const int64_t first = static_cast<int64_t>(blockIdx.x) * kTile + static_cast<int64_t>(threadIdx.x) * kItems;
    int c[kItems];
    load_block(cell_ids, nf, vec, first, c);       // the caller's input: read while k_zero drains
    grid_dep_wait();
    grid_dep_allow();
    int bad = 0;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        if (c[j] >= 0 && c[j] < n_cells)
            atomicAdd(count + c[j], 1);
        else if (c[j] != -1 && c[j] != -2)
            ++bad;
    }
    const long long tot = cta_sum_ll(bad, red);
    if (threadIdx.x == 0 && tot > 0) atomicAdd(invalid, static_cast<int>(tot < INT_MAX ? tot : INT_MAX));
}

__global__ void __launch_bounds__(kThreads)
k_tile_sums(const int32_t *__restrict__ count, int32_t n_cells, int32_t *__restrict__ tile_cnt,
            int32_t *__restrict__ tile_nz) {
    grid_dep_wait();
    grid_dep_allow();
    __shared__ long long red[kWarps];
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kCellTile;
    int cnt = 0, nz = 0;
#pragma unroll
    for (int j = 0; j < kCellItems; ++j) {
        const int64_t c = base + j * kThreads + threadIdx.x;
        if (c < n_cells) {
            const int v = count[c];
            cnt += v;
            nz += v > 0;
        }
    }
    const long long tot = cta_sum_ll(static_cast<long long>(cnt) + (static_cast<long long>(nz) << 32), red);
    if (threadIdx.x == 0) {
        tile_cnt[blockIdx.x] = static_cast<int32_t>(tot & 0xffffffffll);
        tile_nz[blockIdx.x] = static_cast<int32_t>(tot >> 32);
    }
}

// Exclusive scan of the counts of one 1024-cell tile (each thread owns 4
// consecutive cells), plus the interval of every non-empty cell.
__global__ void __launch_bounds__(kThreads)
k_offsets(const int32_t *__restrict__ count, int32_t n_cells, const int32_t *__restrict__ tile_cnt,
          const int32_t *__restrict__ tile_nz, int32_t *__restrict__ offset, int32_t *__restrict__ starts,
          int32_t *__restrict__ lengths, int32_t *__restrict__ icell, const int32_t *__restrict__ invalid,
          int32_t *__restrict__ d_counts) {
    grid_dep_wait();
    grid_dep_allow();
    const int b = blockIdx.x;
    long long pre = 0;
    for (int i = threadIdx.x; i < b; i += kThreads)
        pre += static_cast<long long>(tile_cnt[i]) + (static_cast<long long>(tile_nz[i]) << 32);
    const int64_t c0 = static_cast<int64_t>(b) * kCellTile + static_cast<int64_t>(threadIdx.x) * kCellItems;
    int v[kCellItems];
    int my_cnt = 0, my_nz = 0;
#pragma unroll
    for (int j = 0; j < kCellItems; ++j) {
        v[j] = c0 + j < n_cells ? count[c0 + j] : 0;
        my_cnt += v[j];
        my_nz += v[j] > 0;
    }
    // One scan for both running sums and the sum of the earlier tiles: points
    // in the low 32 bits, non-empty cells in the high 32 (every sum < 2^31,
    // so nothing carries between the halves), one barrier.
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long my = static_cast<long long>(my_cnt) + (static_cast<long long>(my_nz) << 32);
    long long x = my;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, o);
    __shared__ long long s_scan[kWarps], s_pre[kWarps];
    if (lane == 31) s_scan[warp] = x;
    if (lane == 0) s_pre[warp] = pre;
    __syncthreads();
    long long base = 0, tot = 0, pre_all = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const long long t = s_scan[w];
        if (w < warp) base += t;
        tot += t;
        pre_all += s_pre[w];
    }
    const int pre_cnt = static_cast<int>(pre_all & 0xffffffffll);
    const int pre_nz = static_cast<int>(pre_all >> 32);
    const long long ex = base + x - my;
    int run_cnt = static_cast<int>(ex & 0xffffffffll) + pre_cnt;
    int run_nz = static_cast<int>(ex >> 32) + pre_nz;
    const int tot_cnt = static_cast<int>(tot & 0xffffffffll), tot_nz = static_cast<int>(tot >> 32);
#pragma unroll
    for (int j = 0; j < kCellItems; ++j) {
        if (c0 + j < n_cells) {
            offset[c0 + j] = run_cnt;
            if (v[j] > 0) {
                starts[run_nz] = run_cnt;
                lengths[run_nz] = v[j];
                icell[run_nz] = static_cast<int32_t>(c0 + j);
                ++run_nz;
            }
            run_cnt += v[j];
        }
    }
    if (b == static_cast<int>(gridDim.x) - 1 && threadIdx.x == 0) {
        d_counts[0] = pre_cnt + tot_cnt;
        d_counts[1] = pre_nz + tot_nz;
        d_counts[2] = *invalid;
    }
}

__global__ void __launch_bounds__(kThreads)
k_scatter(const int32_t *__restrict__ cell_ids, int64_t nf, int32_t n_cells, bool vec,
          int32_t *__restrict__ cursor, int32_t *__restrict__ tmp_p) {
    const int64_t first = static_cast<int64_t>(blockIdx.x) * kTile + static_cast<int64_t>(threadIdx.x) * kItems;
    int c[kItems];
    load_block(cell_ids, nf, vec, first, c);       // the caller's input: read while k_offsets drains
    grid_dep_wait();
    grid_dep_allow();
    int pos[kItems];
#pragma unroll
    for (int j = 0; j < kItems; ++j) pos[j] = (c[j] >= 0 && c[j] < n_cells) ? atomicAdd(cursor + c[j], 1) : -1;
#pragma unroll
    for (int j = 0; j < kItems; ++j)
        if (pos[j] >= 0) tmp_p[pos[j]] = static_cast<int32_t>(first + j);
}

struct Derive {
    int32_t *ranks_depth, *ranks_feat, *ranks_bev;
    FastDiv dhw, hw;
    __device__ __forceinline__ void put(int pos, int p, int cell) const {
        const uint32_t u = static_cast<uint32_t>(p);
        const uint32_t nc = dhw.div(u);
        ranks_depth[pos] = p;
        ranks_feat[pos] = static_cast<int32_t>(nc * hw.d + (u - hw.div(u) * hw.d));
        ranks_bev[pos] = cell;
    }
};

// One warp ranks slice k of an interval [s, s + L) (its points s + 32k ..
// s + 32k + 31): a value's rank is the number of smaller values in the whole
// interval (p are distinct), counted over the interval 32 values at a time,
// eight chunks of loads in flight.
__device__ __forceinline__ void warp_rank_slice(const int32_t *__restrict__ src, int s, int L, int k, int cell,
                                                const Derive &out) {
    const int lane = threadIdx.x & 31;
    const int idx = k * 32 + lane;
    const int v = idx < L ? __ldg(src + s + idx) : INT_MAX;
    const int nch = (L + 31) >> 5;                       // uniform over the warp
    int rank = 0;
    for (int c0 = 0; c0 < nch; c0 += 8) {
        int x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = (c0 + u) * 32 + lane;
            x[u] = e < L ? __ldg(src + s + e) : INT_MAX;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (c0 + u < nch) {                          // uniform
#pragma unroll
                for (int t = 0; t < 32; ++t) rank += __shfl_sync(0xffffffffu, x[u], t) < v;
            }
        }
    }
    if (idx < L) out.put(s + rank, v, cell);
}

// Longer intervals: rebuild the run in frustum order by a stable compaction of
// the whole frustum restricted to this cell.
__device__ __forceinline__ void cta_scan_frustum(const int32_t *__restrict__ cell_ids, int64_t nf, int s,
                                                 int cell, const Derive &out, int *scratch) {
    int running = s;
    for (int64_t base = 0; base < nf; base += kThreads) {
        const int64_t e = base + threadIdx.x;
        const int hit = (e < nf && __ldg(cell_ids + e) == cell) ? 1 : 0;
        int tot;
        const int ex = cta_exclusive_sum(hit, scratch, &tot);
        if (hit) out.put(running + ex, static_cast<int>(e), cell);
        running += tot;
    }
}

// Ascending sort of N register values (bitonic network; N a power of two).
template <int N>
__device__ __forceinline__ void sort_regs(int *v) {
#pragma unroll
    for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    const int a = v[i], b = v[l];
                    const bool up = (i & k) == 0;
                    v[i] = up ? min(a, b) : max(a, b);
                    v[l] = up ? max(a, b) : min(a, b);
                }
            }
        }
    }
}

// One thread sorts an interval of L <= N points in registers and writes it.
template <int N>
__device__ __forceinline__ void thread_sort(const int32_t *__restrict__ src, int s, int L, int cell,
                                            const Derive &out) {
    int v[N];
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] = k < L ? __ldg(src + s + k) : INT_MAX;
    sort_regs<N>(v);
#pragma unroll
    for (int k = 0; k < N; ++k)
        if (k < L) out.put(s + k, v[k], cell);
}

// One thread per interval: intervals of up to kThreadSortMax points are
// sorted in registers on the spot; longer ones are appended to the slice or
// long work list for k_sort_lists (the list order does not affect the result).
__global__ void __launch_bounds__(kThreads)
k_sort_runs(const int32_t *__restrict__ tmp_p, const int32_t *__restrict__ starts,
            const int32_t *__restrict__ lengths, const int32_t *__restrict__ icell,
            const int32_t *__restrict__ d_counts, int32_t *__restrict__ lists, int32_t *__restrict__ slice_list,
            int32_t *__restrict__ long_list, Derive out) {
    grid_dep_wait();
    grid_dep_allow();
    const int n_int = __ldg(d_counts + 1);
    const int i = blockIdx.x * kThreads + threadIdx.x;
    if (i >= n_int) return;
    const int s = __ldg(starts + i), L = __ldg(lengths + i), cell = __ldg(icell + i);
    if (L <= 4)
        thread_sort<4>(tmp_p, s, L, cell, out);
    else if (L <= 8)
        thread_sort<8>(tmp_p, s, L, cell, out);
    else if (L <= kThreadSortMax)
        thread_sort<kThreadSortMax>(tmp_p, s, L, cell, out);
    else if (L <= kSliceSortMax) {
        const int nsl = (L + 31) >> 5;
        const int base = atomicAdd(lists + 0, nsl);
        for (int k = 0; k < nsl; ++k) slice_list[base + k] = static_cast<int32_t>((static_cast<uint32_t>(i) << 8) | k);
    } else {
        long_list[atomicAdd(lists + 1, 1)] = i;
    }
}

// Persistent CTAs drain the lists: each warp ranks slices (32 points of an
// interval of 17..kSliceSortMax points, so a long interval is spread over
// many warps), then each CTA rebuilds the rare longer intervals by scanning
// the frustum.
__global__ void __launch_bounds__(kThreads)
k_sort_lists(const int32_t *__restrict__ tmp_p, const int32_t *__restrict__ starts,
             const int32_t *__restrict__ lengths, const int32_t *__restrict__ icell,
             const int32_t *__restrict__ lists, const int32_t *__restrict__ slice_list,
             const int32_t *__restrict__ long_list, const int32_t *__restrict__ cell_ids, int64_t nf, Derive out) {
    grid_dep_wait();
    grid_dep_allow();
    __shared__ int scratch[kWarps + 1];
    const int n_slices = __ldg(lists + 0), n_long = __ldg(lists + 1);
    const int warps_total = gridDim.x * kWarps;
    for (int x = blockIdx.x * kWarps + (threadIdx.x >> 5); x < n_slices; x += warps_total) {   // warp-uniform
        const uint32_t e = static_cast<uint32_t>(__ldg(slice_list + x));
        const int j = static_cast<int>(e >> 8), k = static_cast<int>(e & 255u);
        warp_rank_slice(tmp_p, __ldg(starts + j), __ldg(lengths + j), k, __ldg(icell + j), out);
    }
    for (int x = blockIdx.x; x < n_long; x += gridDim.x) {                                   // CTA-uniform
        const int j = __ldg(long_list + x);
        cta_scan_frustum(cell_ids, nf, __ldg(starts + j), __ldg(icell + j), out, scratch);
    }
}

}  // namespace

size_t count_workspace_bytes(int64_t n_frustum, int32_t n_cells) { return carve(nullptr, n_frustum, n_cells, nullptr); }

cudaError_t launch_build_map_counting(const BuildMapArgs &a) {
    const int64_t nf = static_cast<int64_t>(a.NC) * a.D * a.H * a.W;
    CountWs ws;
    carve(a.workspace, nf, a.n_cells, &ws);
    cudaStream_t st = a.stream;
    DeviceInfo info;
    if (!device_info(&info)) return cudaErrorInvalidDevice;
    const int nt = static_cast<int>(div_up(nf, kTile));
    const int nct = static_cast<int>(div_up(a.n_cells, kCellTile));
    const bool vec = (reinterpret_cast<uintptr_t>(a.cell_ids) & 15u) == 0;
    int64_t zgrid = div_up(a.n_cells, kThreads * 4);
    if (zgrid > info.sm_count * 8) zgrid = info.sm_count * 8;
    if (zgrid < 1) zgrid = 1;
    // every kernel may launch while its predecessor drains (programmatic dependent launch)
    cudaError_t e = launch_dependent(k_zero, dim3(static_cast<unsigned>(zgrid)), dim3(kThreads), 0, st, ws.count,
                                     a.n_cells, ws.invalid, ws.lists);
    count_launch();
    if (e == cudaSuccess)
        e = launch_dependent(k_count_cells, dim3(nt), dim3(kThreads), 0, st, a.cell_ids, nf, a.n_cells, vec, ws.count,
                             ws.invalid);
    count_launch();
    if (e == cudaSuccess)
        e = launch_dependent(k_tile_sums, dim3(nct), dim3(kThreads), 0, st, ws.count, a.n_cells, ws.tile_cnt,
                             ws.tile_nz);
    count_launch();
    if (e == cudaSuccess)
        e = launch_dependent(k_offsets, dim3(nct), dim3(kThreads), 0, st, ws.count, a.n_cells, ws.tile_cnt,
                             ws.tile_nz, ws.offset, a.interval_starts, a.interval_lengths, ws.icell, ws.invalid,
                             a.d_counts);
    count_launch();
    if (e == cudaSuccess)
        e = launch_dependent(k_scatter, dim3(nt), dim3(kThreads), 0, st, a.cell_ids, nf, a.n_cells, vec, ws.offset,
                             ws.tmp_p);
    count_launch();
    const int64_t max_int = nf < a.n_cells ? nf : a.n_cells;
    Derive out{a.ranks_depth, a.ranks_feat, a.ranks_bev, FastDiv(static_cast<uint32_t>(a.D) * a.H * a.W),
               FastDiv(static_cast<uint32_t>(a.H) * a.W)};
    if (e == cudaSuccess)
        e = launch_dependent(k_sort_runs, dim3(static_cast<unsigned>(div_up(max_int, kThreads))), dim3(kThreads), 0,
                             st, ws.tmp_p, a.interval_starts, a.interval_lengths, ws.icell, a.d_counts, ws.lists,
                             ws.slice_list, ws.long_list, out);
    count_launch();
    if (e == cudaSuccess)
        e = launch_dependent(k_sort_lists, dim3(info.sm_count * BEVPOOL_MAP_LIST_CTAS_PER_SM), dim3(kThreads), 0, st, ws.tmp_p,
                             a.interval_starts, a.interval_lengths, ws.icell, ws.lists, ws.slice_list, ws.long_list,
                             a.cell_ids, nf, out);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace bevpool
