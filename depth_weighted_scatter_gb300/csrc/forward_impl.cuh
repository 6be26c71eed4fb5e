// forward_impl.cuh -- the BEV-pooling forward kernel (sm_103a), templated on
// input dtype and channel count.  Included by forward_f16.cu / forward_e4m3.cu.
//
// Computes, for every interval of the scatter map ("Accelerating BEV Pooling
// on NVIDIA GPUs for Physical AI Applications", sections "Eliminate redundant
// scatter traffic" and "Implement interval-owned scatter-reduce"),
//     out[bev, :] = scale * sum_{t in interval} depth[ranks_depth[t]] * feat[ranks_feat[t], :]
// in FP32, rounded once to fp16, and writes every other cell as zeros, so
// each output row is written exactly once and no atomics are used.
//
// One launch, two kinds of CTA (interleaved in blockIdx so both run from the
// first wave):
//
//   compute CTA  owns a fixed chunk of consecutive intervals.  It spreads the
//                chunk's points evenly over its owners (an owner = the LPO
//                lanes that together hold one C-channel row, 16 bytes per lane
//                per load), so a 400-point interval is shared by many owners
//                while 1-3-point intervals cost one owner each.  An owner whose
//                piece covers a whole interval writes that cell straight away;
//                pieces of an interval split between owners go to shared
//                memory and the owner holding the interval's first point sums
//                them in owner order after one barrier (deterministic).
//                Per point: one depth load (the section's "depth loaded once
//                per scatter point"), one feature-row gather, FP32 FMAs.
//                Indices are fetched cooperatively (each lane of an owner loads
//                a different point's ranks, then warp shuffles broadcast them).
//
//   fill CTA     owns a tile of kFillCells consecutive cells.  It finds the
//                tile's points in the sorted ranks_bev with a CTA-wide k-ary
//                search (2-3 dependent loads), marks the cells that have
//                points, and writes zeros to the rest with 16-byte stores.
//                This keeps the (large, uneven) empty regions of the grid off
//                the interval owners and spreads them evenly over the GPU.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "bevpool_internal.cuh"

namespace bevpool {

constexpr int kDtypeF16 = 0;
constexpr int kDtypeE4M3 = 1;
constexpr int kFillCells = 256;

template <int DT, int C>
struct FwdShape {
    static constexpr int EB = DT == kDtypeF16 ? 2 : 1;          // input bytes per element
    static constexpr int ROWB = C * EB;                         // bytes per feature row
    static constexpr int VB = ROWB >= 16 ? 16 : ROWB;           // bytes per vector load
    static constexpr int NVEC = ROWB / VB;                      // vector loads per row
    static constexpr int VPL = (DT == kDtypeF16 && NVEC % 2 == 0) ? 2 : 1;   // loads per lane
    static constexpr int LPO = NVEC / VPL;                      // lanes per owner
    static constexpr int EPL = VPL * VB / EB;                   // channels per lane
    static constexpr int OPW = 32 / LPO;                        // owners per warp
    static constexpr int OWNERS = kWarps * OPW;                 // owners per CTA
    static constexpr int IPC = OWNERS;                          // intervals per compute CTA
    static constexpr int IDX_PER_LANE = LPO >= 4 ? 1 : 4 / LPO; // point indices per lane per round
    static constexpr int ROUND = LPO * IDX_PER_LANE;            // points per index round
    static constexpr int UB = ROUND < 8 ? ROUND : 8;            // points gathered per batch
    static constexpr int OUT_VECS = C * 2 / 16;                 // 16-byte fp16 vectors per out row
    static_assert(ROWB % VB == 0, "row must be a whole number of vectors");
    static_assert(NVEC % VPL == 0 && LPO >= 1 && LPO <= 32, "bad lane mapping");
    static_assert(EPL % 8 == 0, "each lane must own whole 16-byte output vectors");
    static_assert(C % 8 == 0, "C must be a multiple of 8");
};

struct FwdParams {
    const void *depth;
    const void *feat;
    const int32_t *ranks_depth;
    const int32_t *ranks_feat;
    const int32_t *ranks_bev;
    const int32_t *starts;
    const int32_t *lengths;
    const int32_t *d_counts;      // nullable
    int32_t n_points;             // host count or capacity
    int32_t n_intervals;
    int32_t n_cells;
    int32_t n_feat_rows;
    int64_t n_depth;
    float scale;
    int streaming;
    int n_compute;                // compute CTAs
    int n_fill;                   // fill CTAs
    __half *out;
};

// ---------------------------------------------------------------- element access

template <int DT>
__device__ __forceinline__ float load_depth(const void *depth, int idx) {
    if constexpr (DT == kDtypeF16) {
        return __half2float(__ldg(static_cast<const __half *>(depth) + idx));
    } else {
        const unsigned char b = __ldg(static_cast<const unsigned char *>(depth) + idx);
        const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
        return __half2float(__half(h));
    }
}

// Raw bytes of one lane's share of a feature row: VPL vectors of VB bytes.
template <int VB>
struct RawVec;
template <>
struct RawVec<16> {
    uint4 v;
};
template <>
struct RawVec<8> {
    uint2 v;
};

template <int VB>
__device__ __forceinline__ RawVec<VB> load_vec(const unsigned char *p) {
    RawVec<VB> r;
    if constexpr (VB == 16)
        r.v = __ldg(reinterpret_cast<const uint4 *>(p));
    else
        r.v = __ldg(reinterpret_cast<const uint2 *>(p));
    return r;
}

template <int VB>
__device__ __forceinline__ RawVec<VB> zero_vec() {
    RawVec<VB> r;
    if constexpr (VB == 16)
        r.v = make_uint4(0, 0, 0, 0);
    else
        r.v = make_uint2(0, 0);
    return r;
}

// acc[0 .. VB/EB) += d * decode(raw)
template <int DT, int VB>
__device__ __forceinline__ void fma_vec(float *acc, float d, const RawVec<VB> &raw) {
    constexpr int NW = VB / 4;
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&raw.v);
    if constexpr (DT == kDtypeF16) {
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            __half2_raw hr;
            hr.x = static_cast<unsigned short>(w[i] & 0xffffu);
            hr.y = static_cast<unsigned short>(w[i] >> 16);
            const float2 f = __half22float2(__half2(hr));
            acc[2 * i] = fmaf(d, f.x, acc[2 * i]);
            acc[2 * i + 1] = fmaf(d, f.y, acc[2 * i + 1]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>(w[i] & 0xffffu), __NV_E4M3);
            const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
            const float2 a = __half22float2(__half2(lo));
            const float2 b = __half22float2(__half2(hi));
            acc[4 * i + 0] = fmaf(d, a.x, acc[4 * i + 0]);
            acc[4 * i + 1] = fmaf(d, a.y, acc[4 * i + 1]);
            acc[4 * i + 2] = fmaf(d, b.x, acc[4 * i + 2]);
            acc[4 * i + 3] = fmaf(d, b.y, acc[4 * i + 3]);
        }
    }
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Store EPL channels (scaled, rounded to fp16) as EPL/8 16-byte vectors.
template <int EPL>
__device__ __forceinline__ void store_row_part(__half *dst, const float *acc, float scale, bool streaming) {
#pragma unroll
    for (int q = 0; q < EPL / 8; ++q) {
        uint4 v;
        v.x = pack_half2(acc[8 * q + 0] * scale, acc[8 * q + 1] * scale);
        v.y = pack_half2(acc[8 * q + 2] * scale, acc[8 * q + 3] * scale);
        v.z = pack_half2(acc[8 * q + 4] * scale, acc[8 * q + 5] * scale);
        v.w = pack_half2(acc[8 * q + 6] * scale, acc[8 * q + 7] * scale);
        uint4 *p = reinterpret_cast<uint4 *>(dst) + q;
        if (streaming)
            __stcs(p, v);
        else
            *p = v;
    }
}

// ---------------------------------------------------------------- compute CTA

template <int DT, int C>
struct ComputeSmem {
    using S = FwdShape<DT, C>;
    int start[S::IPC];
    int len[S::IPC];
    int pre[S::IPC + 1];          // exclusive prefix of len; pre[nI] = total points
    int bev[S::IPC];
    __align__(16) float part[2][S::OWNERS][C];  // partial sums of split intervals
};

struct FillSmem {
    unsigned mark[kFillCells / 32];
    int probe[2];
};

template <int DT, int C>
union FwdSmem {
    ComputeSmem<DT, C> c;
    FillSmem f;
};

// Accumulate the points t0 .. t0+m-1 into acc (one owner, all LPO lanes).
template <int DT, int C>
__device__ __forceinline__ void accumulate_piece(const FwdParams &p, int t0, int m, int ol, int lane0,
                                                 unsigned gmask, float *acc) {
    using S = FwdShape<DT, C>;
    const unsigned char *feat = static_cast<const unsigned char *>(p.feat);
    const int lane_off = ol * S::VPL * S::VB;   // byte offset of this lane's share of a row
    for (int base = 0; base < m; base += S::ROUND) {
        int rd[S::IDX_PER_LANE], rf[S::IDX_PER_LANE];
#pragma unroll
        for (int q = 0; q < S::IDX_PER_LANE; ++q) {
            const int j = base + q * S::LPO + ol;
            rd[q] = -1;
            rf[q] = -1;
            if (j < m) {
                const int a = __ldg(p.ranks_depth + t0 + j);
                const int b = __ldg(p.ranks_feat + t0 + j);
                if (a >= 0 && a < p.n_depth && b >= 0 && b < p.n_feat_rows) {
                    rd[q] = a;
                    rf[q] = b;
                }
            }
        }
        const int cnt = min(S::ROUND, m - base);
#pragma unroll
        for (int u0 = 0; u0 < S::ROUND; u0 += S::UB) {
            if (u0 >= cnt) break;
            float dv[S::UB];
            RawVec<S::VB> fv[S::UB][S::VPL];
#pragma unroll
            for (int u = 0; u < S::UB; ++u) {
                const int uu = u0 + u;                         // compile-time after unrolling
                const int slot = (uu < S::ROUND ? uu : 0) / S::LPO;
                const int src = lane0 + (uu < S::ROUND ? uu : 0) % S::LPO;
                const int a = __shfl_sync(gmask, rd[slot < S::IDX_PER_LANE ? slot : 0], src);
                const int b = __shfl_sync(gmask, rf[slot < S::IDX_PER_LANE ? slot : 0], src);
                const bool ok = uu < cnt && a >= 0;
                dv[u] = ok ? load_depth<DT>(p.depth, a) : 0.f;
#pragma unroll
                for (int v = 0; v < S::VPL; ++v)
                    fv[u][v] = ok ? load_vec<S::VB>(feat + static_cast<int64_t>(b) * S::ROWB + lane_off + v * S::VB)
                                  : zero_vec<S::VB>();
            }
#pragma unroll
            for (int u = 0; u < S::UB; ++u) {
#pragma unroll
                for (int v = 0; v < S::VPL; ++v) fma_vec<DT, S::VB>(acc + v * (S::VB / S::EB), dv[u], fv[u][v]);
            }
        }
    }
}

template <int DT, int C>
__device__ __forceinline__ void compute_cta(const FwdParams &p, int cidx, ComputeSmem<DT, C> &sm) {
    using S = FwdShape<DT, C>;
    __shared__ int scratch[kWarps + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    int n_int = p.n_intervals, n_pts = p.n_points;
    if (p.d_counts) {
        n_int = min(n_int, __ldg(p.d_counts + 1));
        n_pts = min(n_pts, __ldg(p.d_counts + 0));
    }
    const int i0 = cidx * S::IPC;
    if (i0 >= n_int) return;                       // uniform over the CTA
    const int nI = min(S::IPC, n_int - i0);

    // 1. interval metadata (IPC <= 256: at most one interval per thread)
    int my_len = 0;
    if (threadIdx.x < S::IPC) {
        int s = 0, L = 0, cell = -1;
        if (static_cast<int>(threadIdx.x) < nI) {
            s = __ldg(p.starts + i0 + threadIdx.x);
            L = __ldg(p.lengths + i0 + threadIdx.x);
            if (s < 0 || L < 0 || s > n_pts - L) L = 0;   // outside the point range: skip
            if (L > 0) {
                cell = __ldg(p.ranks_bev + s);
                if (cell < 0 || cell >= p.n_cells) {
                    L = 0;
                    cell = -1;
                }
            }
        }
        sm.start[threadIdx.x] = s;
        sm.bev[threadIdx.x] = cell;
        my_len = L;
        sm.len[threadIdx.x] = L;
    }
    int total;
    const int excl = cta_exclusive_sum(my_len, scratch, &total);
    if (threadIdx.x < S::IPC) sm.pre[threadIdx.x] = excl;
    if (threadIdx.x == 0) sm.pre[S::IPC] = total;
    __syncthreads();

    // 2. each owner walks its even share [beg, end) of the chunk's points
    const int og = lane / S::LPO;                  // owner within warp
    const int ol = lane % S::LPO;                  // lane within owner
    const bool active = og < S::OPW;
    const int o = warp * S::OPW + og;
    const int lane0 = og * S::LPO;
    const unsigned gmask = (S::LPO == 32 ? 0xffffffffu : ((1u << S::LPO) - 1u)) << lane0;
    const int P = total;
    const int beg = active ? static_cast<int>((static_cast<int64_t>(o) * P) / S::OWNERS) : 0;
    const int end = active ? static_cast<int>((static_cast<int64_t>(o + 1) * P) / S::OWNERS) : 0;

    int head_k = -1;       // split interval this owner must combine (it holds its first point)
    int head_slot = 0;
    if (beg < end) {
        // first interval k with pre[k] <= beg < pre[k+1]
        int lo = 0, hi = S::IPC;                   // pre[] is non-decreasing; search the last k with pre[k] <= beg
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (sm.pre[mid] <= beg) lo = mid; else hi = mid;
        }
        int k = lo;
        while (sm.pre[k + 1] <= beg) ++k;           // skip zero-length intervals
        int v = beg;
        bool first = true;
        while (v < end) {
            const int pk = sm.pre[k], pk1 = sm.pre[k + 1];
            const int a = v - pk;
            const int bnd = min(end, pk1) - pk;
            float acc[S::EPL];
#pragma unroll
            for (int e = 0; e < S::EPL; ++e) acc[e] = 0.f;
            accumulate_piece<DT, C>(p, sm.start[k] + a, bnd - a, ol, lane0, gmask, acc);
            const bool whole = a == 0 && bnd == pk1 - pk;
            if (whole) {
                store_row_part<S::EPL>(p.out + static_cast<int64_t>(sm.bev[k]) * C + ol * S::EPL, acc, p.scale,
                                       p.streaming);
            } else {
                const int slot = first ? 0 : 1;
                float *dst = &sm.part[slot][o][ol * S::EPL];
#pragma unroll
                for (int e = 0; e < S::EPL; e += 4)
                    *reinterpret_cast<float4 *>(dst + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
                if (a == 0) {
                    head_k = k;
                    head_slot = slot;
                }
            }
            v = pk + bnd;
            first = false;
            ++k;
            while (k < nI && v < end && sm.pre[k + 1] <= v) ++k;   // skip zero-length intervals
        }
    }
    __syncthreads();

    // 3. combine split intervals in owner order
    if (head_k >= 0) {
        float acc[S::EPL];
        const float *src = &sm.part[head_slot][o][ol * S::EPL];
#pragma unroll
        for (int e = 0; e < S::EPL; ++e) acc[e] = src[e];
        const int stop = sm.pre[head_k + 1];
        for (int o2 = o + 1; o2 < S::OWNERS; ++o2) {
            const int b2 = static_cast<int>((static_cast<int64_t>(o2) * P) / S::OWNERS);
            if (b2 >= stop) break;
            const int e2 = static_cast<int>((static_cast<int64_t>(o2 + 1) * P) / S::OWNERS);
            if (b2 == e2) continue;                // empty share: wrote nothing
            const float *q = &sm.part[0][o2][ol * S::EPL];
#pragma unroll
            for (int e = 0; e < S::EPL; ++e) acc[e] += q[e];
        }
        store_row_part<S::EPL>(p.out + static_cast<int64_t>(sm.bev[head_k]) * C + ol * S::EPL, acc, p.scale,
                               p.streaming);
    }
}

// ---------------------------------------------------------------- fill CTA

// First index in [0, n) whose value is >= key, for two keys at once, by a
// CTA-wide k-ary search over the sorted ranks_bev.
__device__ __forceinline__ void cta_lower_bound2(const int32_t *a, int n, int key0, int key1, int *r0, int *r1) {
    int lo0 = 0, hi0 = n, lo1 = 0, hi1 = n;
    while (hi0 - lo0 > kThreads || hi1 - lo1 > kThreads) {
        const int st0 = (hi0 - lo0 + kThreads - 1) / kThreads;
        const int st1 = (hi1 - lo1 + kThreads - 1) / kThreads;
        const int x0 = lo0 + threadIdx.x * st0;
        const int x1 = lo1 + threadIdx.x * st1;
        const bool p0 = x0 < hi0 && __ldg(a + x0) < key0;
        const bool p1 = x1 < hi1 && __ldg(a + x1) < key1;
        const int c0 = __syncthreads_count(p0);
        const int c1 = __syncthreads_count(p1);
        const int nlo0 = c0 > 0 ? lo0 + (c0 - 1) * st0 + 1 : lo0;
        const int nhi0 = min(hi0, lo0 + c0 * st0);
        const int nlo1 = c1 > 0 ? lo1 + (c1 - 1) * st1 + 1 : lo1;
        const int nhi1 = min(hi1, lo1 + c1 * st1);
        lo0 = nlo0; hi0 = nhi0; lo1 = nlo1; hi1 = nhi1;
    }
    const int x0 = lo0 + threadIdx.x, x1 = lo1 + threadIdx.x;
    const int c0 = __syncthreads_count(x0 < hi0 && __ldg(a + x0) < key0);
    const int c1 = __syncthreads_count(x1 < hi1 && __ldg(a + x1) < key1);
    *r0 = lo0 + c0;
    *r1 = lo1 + c1;
}

template <int DT, int C>
__device__ __forceinline__ void fill_cta(const FwdParams &p, int fidx, FillSmem &sm) {
    using S = FwdShape<DT, C>;
    int n_pts = p.n_points;
    if (p.d_counts) n_pts = min(n_pts, __ldg(p.d_counts + 0));
    if (n_pts < 0) n_pts = 0;
    const int c0 = fidx * kFillCells;
    const int c1 = min(c0 + kFillCells, p.n_cells);
    if (threadIdx.x < kFillCells / 32) sm.mark[threadIdx.x] = 0u;
    int t0, t1;
    cta_lower_bound2(p.ranks_bev, n_pts, c0, c1, &t0, &t1);   // contains barriers
    for (int t = t0 + threadIdx.x; t < t1; t += kThreads) {
        const int cell = __ldg(p.ranks_bev + t) - c0;
        if (cell >= 0 && cell < kFillCells) atomicOr(&sm.mark[cell >> 5], 1u << (cell & 31));
    }
    __syncthreads();
    const int total = (c1 - c0) * S::OUT_VECS;
    uint4 *out = reinterpret_cast<uint4 *>(p.out + static_cast<int64_t>(c0) * C);
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int v = threadIdx.x; v < total; v += kThreads) {
        const int cell = v / S::OUT_VECS;
        if (!((sm.mark[cell >> 5] >> (cell & 31)) & 1u)) {
            if (p.streaming)
                __stcs(out + v, z);
            else
                out[v] = z;
        }
    }
}

// ---------------------------------------------------------------- kernel

template <int DT, int C>
__global__ void __launch_bounds__(kThreads, 2) k_forward(const FwdParams p) {
    __shared__ __align__(16) FwdSmem<DT, C> sm;
    const int b = blockIdx.x;
    const int both = 2 * min(p.n_compute, p.n_fill);
    bool compute;
    int idx;
    if (b < both) {
        compute = (b & 1) == 0;
        idx = b >> 1;
    } else {
        compute = p.n_compute > p.n_fill;
        idx = (both >> 1) + (b - both);
    }
    if (compute)
        compute_cta<DT, C>(p, idx, sm.c);
    else
        fill_cta<DT, C>(p, idx, sm.f);
}

template <int DT, int C>
cudaError_t launch_forward_t(const ForwardArgs &a) {
    using S = FwdShape<DT, C>;
    FwdParams p;
    p.depth = a.depth;
    p.feat = a.feat;
    p.ranks_depth = a.ranks_depth;
    p.ranks_feat = a.ranks_feat;
    p.ranks_bev = a.ranks_bev;
    p.starts = a.interval_starts;
    p.lengths = a.interval_lengths;
    p.d_counts = a.d_counts;
    p.n_points = a.n_points;
    p.n_intervals = a.n_intervals;
    p.n_cells = a.n_cells;
    p.n_feat_rows = a.n_feat_rows;
    p.n_depth = a.n_depth;
    p.scale = a.scale;
    p.streaming = a.streaming_stores;
    p.n_compute = static_cast<int>(div_up(a.n_intervals, S::IPC));
    p.n_fill = static_cast<int>(div_up(a.n_cells, kFillCells));
    p.out = static_cast<__half *>(a.out);
    const int grid = p.n_compute + p.n_fill;
    k_forward<DT, C><<<grid, kThreads, 0, a.stream>>>(p);
    count_launch();
    return cudaGetLastError();
}

}  // namespace bevpool
