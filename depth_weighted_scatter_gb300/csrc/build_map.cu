// build_map.cu -- scatter-map construction on the GPU (sm_103a): the radix
// path, used for grids of more than kCountingMaxCells cells (build_map_count.cu
// handles the rest), and the dispatch between the two.
//
// Builds the five-array INT32 scatter map of "Accelerating BEV Pooling on
// NVIDIA GPUs for Physical AI Applications" (section "Eliminate redundant
// scatter traffic": separate ranks_depth / ranks_feat / ranks_bev arrays plus
// interval_starts / interval_lengths, with the feature-row index precomputed
// so the forward does no integer division).  The pages say the map is
// prepared ahead (section "Implement interval-owned scatter-reduce") but not
// how; this file does it as
//
//   1. compaction  : keep (cell, p) for every frustum point with a valid cell,
//                    in frustum order (per-tile counts, then a stable scatter
//                    whose tile offset each CTA sums from the counts before it);
//   2. radix sort  : stable LSD radix sort of the kept pairs by cell, <= 11-bit
//                    digits, reduce-then-scan per pass (tile histograms, a
//                    column scan per digit, stable scatter).  Stability keeps
//                    equal cells in ascending p, which makes the map bit-exact;
//   3. derivation  : the last pass writes ranks_bev = cell, ranks_depth = p and
//                    ranks_feat = nc*H*W + h*W + w directly;
//   4. intervals   : run heads (bev[t] != bev[t-1]) counted per tile, then each
//                    CTA emits starts and lengths of its runs.
//
// No kernel waits on another CTA: every cross-tile dependency goes through a
// kernel boundary, so nothing can spin or hang.
#include <climits>

#include "bevpool_internal.cuh"

namespace bevpool {
namespace {

constexpr int kItems = 16;
constexpr int kTile = kThreads * kItems;        // 4096 elements per CTA tile
constexpr int kWarpSpan = kTile / kWarps;       // 512 consecutive elements per warp
constexpr int kMaxDigitBits = 11;
constexpr int kMaxBins = 1 << kMaxDigitBits;

__device__ __forceinline__ int div_up_dev(int n) { return (n + kTile - 1) / kTile; }

struct Workspace {
    int32_t *keys_a, *vals_a, *keys_b, *vals_b;   // [n_frustum] each
    int32_t *tile_count, *tile_invalid;           // [ntiles]
    int32_t *hist;                                // [kMaxBins * ntiles]
    int32_t *coltotal;                            // [kMaxBins]
    int32_t *head_count, *head_last;              // [ntiles]
    int32_t *n_dev;                               // [1]
};

// Lays the workspace out (or only measures it when base == nullptr).
size_t carve(void *base, int64_t nf, Workspace *ws) {
    const int64_t nt = div_up(nf, kTile);
    size_t off = 0;
    auto take = [&](int64_t count) -> int32_t * {
        int32_t *p = base ? reinterpret_cast<int32_t *>(static_cast<char *>(base) + off) : nullptr;
        off = align_up(off + static_cast<size_t>(count) * sizeof(int32_t), 256);
        return p;
    };
    Workspace w;
    w.keys_a = take(nf);
    w.vals_a = take(nf);
    w.keys_b = take(nf);
    w.vals_b = take(nf);
    w.tile_count = take(nt);
    w.tile_invalid = take(nt);
    w.hist = take(static_cast<int64_t>(kMaxBins) * nt);
    w.coltotal = take(kMaxBins);
    w.head_count = take(nt);
    w.head_last = take(nt);
    w.n_dev = take(1);
    if (ws) *ws = w;
    return off;
}

// ---------------------------------------------------------------- 1. compaction

__global__ void __launch_bounds__(kThreads)
k_count(const int32_t *__restrict__ cell_ids, int64_t nf, int32_t n_cells,
        int32_t *__restrict__ tile_count, int32_t *__restrict__ tile_invalid) {
    __shared__ long long red[kWarps];
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kTile;
    int kept = 0, invalid = 0;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int64_t e = base + j * kThreads + threadIdx.x;
        if (e < nf) {
            const int c = __ldg(cell_ids + e);
            const bool ok = c >= 0 && c < n_cells;
            kept += ok;
            invalid += (!ok && c != -1);
        }
    }
    const long long tot = cta_sum_ll(static_cast<long long>(kept) + (static_cast<long long>(invalid) << 32), red);
    if (threadIdx.x == 0) {
        tile_count[blockIdx.x] = static_cast<int32_t>(tot & 0xffffffffll);
        tile_invalid[blockIdx.x] = static_cast<int32_t>(tot >> 32);
    }
}

__global__ void __launch_bounds__(kThreads)
k_compact(const int32_t *__restrict__ cell_ids, int64_t nf, int32_t n_cells,
          const int32_t *__restrict__ tile_count, const int32_t *__restrict__ tile_invalid,
          int32_t *__restrict__ keys_out, int32_t *__restrict__ vals_out,
          int32_t *__restrict__ n_dev, int32_t *__restrict__ d_counts) {
    __shared__ long long red[kWarps];
    __shared__ int wtot[2][kWarps];
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    long long pre = 0;
    for (int i = threadIdx.x; i < b; i += kThreads) pre += tile_count[i];
    pre = cta_sum_ll(pre, red);

    int running = static_cast<int>(pre);
    const int64_t base = static_cast<int64_t>(b) * kTile;
#pragma unroll 4
    for (int j = 0; j < kItems; ++j) {
        const int64_t e = base + j * kThreads + threadIdx.x;
        const int c = e < nf ? __ldg(cell_ids + e) : -1;
        const bool kept = c >= 0 && c < n_cells;
        const unsigned m = __ballot_sync(0xffffffffu, kept);
        if (lane == 0) wtot[j & 1][warp] = __popc(m);
        __syncthreads();
        int woff = 0, rtot = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int t = wtot[j & 1][w];
            woff += w < warp ? t : 0;
            rtot += t;
        }
        if (kept) {
            const int pos = running + woff + __popc(m & lanemask_lt());
            keys_out[pos] = c;
            vals_out[pos] = static_cast<int32_t>(e);
        }
        running += rtot;
    }

    if (b == static_cast<int>(gridDim.x) - 1) {
        long long inv = 0;
        for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += kThreads) inv += tile_invalid[i];
        inv = cta_sum_ll(inv, red);
        if (threadIdx.x == 0) {
            n_dev[0] = running;
            d_counts[0] = running;
            d_counts[2] = static_cast<int32_t>(inv < INT_MAX ? inv : INT_MAX);
        }
    }
}

// ---------------------------------------------------------------- 2. radix passes

__global__ void __launch_bounds__(kThreads)
k_upsweep(const int32_t *__restrict__ keys, const int32_t *__restrict__ n_dev, int shift,
          int nbins, int32_t *__restrict__ hist) {
    __shared__ int s_hist[kMaxBins];
    const int n = *n_dev;
    const int ntiles = static_cast<int>(div_up_dev(n));
    const int b = blockIdx.x;
    if (b >= ntiles) return;
    for (int d = threadIdx.x; d < nbins; d += kThreads) s_hist[d] = 0;
    __syncthreads();
    const int base = b * kTile;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int e = base + j * kThreads + threadIdx.x;
        if (e < n) atomicAdd(&s_hist[(__ldg(keys + e) >> shift) & (nbins - 1)], 1);
    }
    __syncthreads();
    for (int d = threadIdx.x; d < nbins; d += kThreads)
        hist[static_cast<int64_t>(d) * ntiles + b] = s_hist[d];
}

// One warp per digit: exclusive scan down that digit's column of tile counts
// (contiguous, digit-major), in place; the column total goes to coltotal.
__global__ void __launch_bounds__(kThreads)
k_colscan(int32_t *__restrict__ hist, const int32_t *__restrict__ n_dev, int nbins,
          int32_t *__restrict__ coltotal) {
    const int n = *n_dev;
    const int ntiles = static_cast<int>(div_up_dev(n));
    const int lane = threadIdx.x & 31;
    const int d = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (d >= nbins) return;
    int32_t *col = hist + static_cast<int64_t>(d) * ntiles;
    int carry = 0;
    for (int i0 = 0; i0 < ntiles; i0 += 32) {
        const int i = i0 + lane;
        const int v = i < ntiles ? col[i] : 0;
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (i < ntiles) col[i] = carry + x - v;
        carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) coltotal[d] = carry;
}

// Exclusive scan of nbins consecutive ints held in shared memory, in place,
// by the whole CTA (each thread owns a run of consecutive entries).
__device__ __forceinline__ void cta_scan_bins(int *a, int nbins, int *scratch) {
    const int per = (nbins + kThreads - 1) / kThreads;
    const int lo = threadIdx.x * per;
    int local = 0;
    for (int i = 0; i < per; ++i)
        if (lo + i < nbins) local += a[lo + i];
    int tot;
    int run = cta_exclusive_sum(local, scratch, &tot);
    for (int i = 0; i < per; ++i)
        if (lo + i < nbins) {
            const int v = a[lo + i];
            a[lo + i] = run;
            run += v;
        }
    __syncthreads();
}

size_t downsweep_smem(int nbins) {
    return static_cast<size_t>(nbins) * sizeof(int) * 2 + static_cast<size_t>(kTile) * sizeof(int) * 2 +
           static_cast<size_t>(kWarps) * nbins * sizeof(unsigned short);
}

// Stable scatter of one tile by the current digit.  Warp w ranks the 512
// consecutive elements it owns in order (match.any peers + per-warp digit
// counters), the CTA turns those into tile-local positions, stages the tile
// sorted in shared memory and writes it out so that consecutive threads
// store consecutive addresses within each digit bucket.
template <bool kFinal>
__global__ void __launch_bounds__(kThreads)
k_downsweep(const int32_t *__restrict__ keys_in, const int32_t *__restrict__ vals_in,
            const int32_t *__restrict__ n_dev, int shift, int nbins,
            const int32_t *__restrict__ colprefix, const int32_t *__restrict__ coltotal,
            int32_t *__restrict__ keys_out, int32_t *__restrict__ vals_out,
            int32_t *__restrict__ ranks_bev, int32_t *__restrict__ ranks_depth,
            int32_t *__restrict__ ranks_feat, uint32_t dhw, uint32_t hw) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int scratch[kWarps + 1];
    int *s_gbase = reinterpret_cast<int *>(smem);
    int *s_tstart = s_gbase + nbins;
    int *s_keys = s_tstart + nbins;
    int *s_vals = s_keys + kTile;
    unsigned short *s_cnt = reinterpret_cast<unsigned short *>(s_vals + kTile);

    const int n = *n_dev;
    const int ntiles = static_cast<int>(div_up_dev(n));
    const int b = blockIdx.x;
    if (b >= ntiles) return;
    const int tile_n = min(kTile, n - b * kTile);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // Global start of every digit bucket for this tile.
    for (int d = threadIdx.x; d < nbins; d += kThreads) s_gbase[d] = coltotal[d];
    for (int i = threadIdx.x; i < kWarps * nbins; i += kThreads) s_cnt[i] = 0;
    __syncthreads();
    cta_scan_bins(s_gbase, nbins, scratch);
    for (int d = threadIdx.x; d < nbins; d += kThreads)
        s_gbase[d] += colprefix[static_cast<int64_t>(d) * ntiles + b];

    // Per-warp stable ranks.
    int key[kItems], val[kItems], rnk[kItems];
    unsigned short *my_cnt = s_cnt + warp * nbins;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int el = warp * kWarpSpan + j * 32 + lane;
        const bool valid = el < tile_n;
        key[j] = valid ? __ldg(keys_in + b * kTile + el) : 0;
        val[j] = valid ? __ldg(vals_in + b * kTile + el) : 0;
        rnk[j] = 0;
        const int d = (key[j] >> shift) & (nbins - 1);
        const unsigned act = __ballot_sync(0xffffffffu, valid);
        if (valid) {
            const unsigned peers = __match_any_sync(act, d);
            const int leader = __ffs(peers) - 1;
            const int before = my_cnt[d];
            __syncwarp(act);
            if (lane == leader) my_cnt[d] = static_cast<unsigned short>(before + __popc(peers));
            rnk[j] = before + __popc(peers & lanemask_lt());
        }
        __syncwarp();
    }
    __syncthreads();

    // Cross-warp offsets per digit, tile totals, tile-local digit starts.
    for (int d = threadIdx.x; d < nbins; d += kThreads) {
        int s = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int t = s_cnt[w * nbins + d];
            s_cnt[w * nbins + d] = static_cast<unsigned short>(s);
            s += t;
        }
        s_tstart[d] = s;
    }
    __syncthreads();
    cta_scan_bins(s_tstart, nbins, scratch);

#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int el = warp * kWarpSpan + j * 32 + lane;
        if (el < tile_n) {
            const int d = (key[j] >> shift) & (nbins - 1);
            const int pos = s_tstart[d] + my_cnt[d] + rnk[j];
            s_keys[pos] = key[j];
            s_vals[pos] = val[j];
        }
    }
    __syncthreads();

    for (int i = threadIdx.x; i < tile_n; i += kThreads) {
        const int k = s_keys[i];
        const int d = (k >> shift) & (nbins - 1);
        const int g = s_gbase[d] + (i - s_tstart[d]);
        const int v = s_vals[i];
        if (kFinal) {
            const uint32_t p = static_cast<uint32_t>(v);
            ranks_bev[g] = k;
            ranks_depth[g] = v;
            ranks_feat[g] = static_cast<int32_t>((p / dhw) * hw + p % hw);
        } else {
            keys_out[g] = k;
            vals_out[g] = v;
        }
    }
}

// ---------------------------------------------------------------- 4. intervals

__global__ void __launch_bounds__(kThreads)
k_heads(const int32_t *__restrict__ bev, const int32_t *__restrict__ n_dev,
        int32_t *__restrict__ head_count, int32_t *__restrict__ head_last) {
    __shared__ long long red[kWarps];
    __shared__ int redi[kWarps];
    const int n = *n_dev;
    const int ntiles = static_cast<int>(div_up_dev(n));
    const int b = blockIdx.x;
    if (b >= ntiles) return;
    int cnt = 0, last = -1;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int t = b * kTile + j * kThreads + threadIdx.x;
        if (t < n) {
            const bool h = t == 0 || __ldg(bev + t) != __ldg(bev + t - 1);
            cnt += h;
            if (h) last = t;
        }
    }
    const long long c = cta_sum_ll(cnt, red);
    last = cta_max(last, redi);
    if (threadIdx.x == 0) {
        head_count[b] = static_cast<int32_t>(c);
        head_last[b] = last;
    }
}

__global__ void __launch_bounds__(kThreads)
k_emit(const int32_t *__restrict__ bev, const int32_t *__restrict__ n_dev,
       const int32_t *__restrict__ head_count, const int32_t *__restrict__ head_last,
       int32_t *__restrict__ starts, int32_t *__restrict__ lengths, int32_t *__restrict__ d_counts) {
    __shared__ long long red[kWarps];
    __shared__ int redi[kWarps];
    __shared__ int s_wcnt[kWarps], s_wlast[kWarps];
    const int n = *n_dev;
    const int ntiles = static_cast<int>(div_up_dev(n));
    const int b = blockIdx.x;
    if (ntiles == 0) {
        if (b == 0 && threadIdx.x == 0) d_counts[1] = 0;
        return;
    }
    if (b >= ntiles) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    long long pre = 0;
    int prev = -1;
    for (int i = threadIdx.x; i < b; i += kThreads) {
        pre += head_count[i];
        prev = max(prev, head_last[i]);
    }
    pre = cta_sum_ll(pre, red);
    prev = cta_max(prev, redi);

    // Flags of the 512 consecutive elements this warp owns.
    const int wbase = b * kTile + warp * kWarpSpan;
    unsigned head_bits = 0, tail_bits = 0;   // bit j: element wbase + j*32 + lane
    int wcnt = 0, wlast = -1;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int t = wbase + j * 32 + lane;
        bool h = false, tl = false;
        if (t < n) {
            const int v = __ldg(bev + t);
            h = t == 0 || __ldg(bev + t - 1) != v;
            tl = t == n - 1 || __ldg(bev + t + 1) != v;
        }
        head_bits |= static_cast<unsigned>(h) << j;
        tail_bits |= static_cast<unsigned>(tl) << j;
        const unsigned hb = __ballot_sync(0xffffffffu, h);
        wcnt += __popc(hb);
        if (hb) wlast = wbase + j * 32 + (31 - __clz(hb));
    }
    if (lane == 0) {
        s_wcnt[warp] = wcnt;
        s_wlast[warp] = wlast;
    }
    __syncthreads();
    int running = static_cast<int>(pre);
    int cur_last = prev;
    int tile_heads = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) {
            running += s_wcnt[w];
            cur_last = max(cur_last, s_wlast[w]);
        }
        tile_heads += s_wcnt[w];
    }
    const unsigned le = lanemask_lt() | (1u << lane);
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int t = wbase + j * 32 + lane;
        const bool h = (head_bits >> j) & 1u;
        const bool tl = (tail_bits >> j) & 1u;
        const unsigned hb = __ballot_sync(0xffffffffu, h);
        const int idx = running + __popc(hb & le) - 1;
        const unsigned upto = hb & le;
        const int hp = upto ? wbase + j * 32 + (31 - __clz(upto)) : cur_last;
        if (h) starts[idx] = t;
        if (tl) lengths[idx] = t - hp + 1;
        running += __popc(hb);
        if (hb) cur_last = wbase + j * 32 + (31 - __clz(hb));
    }
    if (b == ntiles - 1 && threadIdx.x == 0) d_counts[1] = static_cast<int32_t>(pre) + tile_heads;
}

}  // namespace

size_t radix_workspace_bytes(int64_t n_frustum) { return carve(nullptr, n_frustum, nullptr); }

size_t build_map_workspace_bytes(int64_t n_frustum, int32_t n_cells) {
    return n_cells <= kCountingMaxCells ? count_workspace_bytes(n_frustum, n_cells) : radix_workspace_bytes(n_frustum);
}

cudaError_t launch_build_map(const BuildMapArgs &a) {
    return a.counting ? launch_build_map_counting(a) : launch_build_map_radix(a);
}

cudaError_t launch_build_map_radix(const BuildMapArgs &a) {
    const int64_t nf = static_cast<int64_t>(a.NC) * a.D * a.H * a.W;
    const int nt = static_cast<int>(div_up(nf, kTile));
    Workspace ws;
    carve(a.workspace, nf, &ws);
    cudaStream_t s = a.stream;

    k_count<<<nt, kThreads, 0, s>>>(a.cell_ids, nf, a.n_cells, ws.tile_count, ws.tile_invalid);
    count_launch();
    k_compact<<<nt, kThreads, 0, s>>>(a.cell_ids, nf, a.n_cells, ws.tile_count, ws.tile_invalid,
                                      ws.keys_a, ws.vals_a, ws.n_dev, a.d_counts);
    count_launch();

    int bits = 0;
    while (bits < 31 && (1ll << bits) < a.n_cells) ++bits;   // cells fit in `bits` bits
    if (bits == 0) bits = 1;
    const int passes = static_cast<int>(div_up(bits, kMaxDigitBits));

    int32_t *kbuf[2] = {ws.keys_a, ws.keys_b};
    int32_t *vbuf[2] = {ws.vals_a, ws.vals_b};
    int shift = 0;
    for (int pass = 0; pass < passes; ++pass) {
        const int32_t *kin = kbuf[pass & 1], *vin = vbuf[pass & 1];
        int32_t *kout = kbuf[(pass + 1) & 1], *vout = vbuf[(pass + 1) & 1];
        const int width = bits / passes + (pass < bits % passes ? 1 : 0);
        const int nbins = 1 << width;
        k_upsweep<<<nt, kThreads, 0, s>>>(kin, ws.n_dev, shift, nbins, ws.hist);
        count_launch();
        k_colscan<<<static_cast<int>(div_up(nbins, kWarps)), kThreads, 0, s>>>(ws.hist, ws.n_dev, nbins,
                                                                              ws.coltotal);
        count_launch();
        const size_t smem = downsweep_smem(nbins);
        if (pass == passes - 1) {
            cudaError_t e = cudaFuncSetAttribute(k_downsweep<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            k_downsweep<true><<<nt, kThreads, smem, s>>>(
                kin, vin, ws.n_dev, shift, nbins, ws.hist, ws.coltotal, nullptr, nullptr, a.ranks_bev,
                a.ranks_depth, a.ranks_feat, static_cast<uint32_t>(a.D) * a.H * a.W,
                static_cast<uint32_t>(a.H) * a.W);
        } else {
            cudaError_t e = cudaFuncSetAttribute(k_downsweep<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            k_downsweep<false><<<nt, kThreads, smem, s>>>(kin, vin, ws.n_dev, shift, nbins, ws.hist,
                                                          ws.coltotal, kout, vout, nullptr, nullptr, nullptr,
                                                          1u, 1u);
        }
        count_launch();
        shift += width;
    }

    k_heads<<<nt, kThreads, 0, s>>>(a.ranks_bev, ws.n_dev, ws.head_count, ws.head_last);
    count_launch();
    k_emit<<<nt, kThreads, 0, s>>>(a.ranks_bev, ws.n_dev, ws.head_count, ws.head_last, a.interval_starts,
                                   a.interval_lengths, a.d_counts);
    count_launch();
    return cudaGetLastError();
}

}  // namespace bevpool
