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
//   compute CTA  owns a chunk of consecutive intervals.  An owner is the LPO
//                lanes that together hold one C-channel row (VB bytes per
//                lane).  Each interval is cut into pieces of at most kPiece
//                points; owners take pieces round-robin.  A one-piece interval
//                (the common case: the canonical workload averages 3.6 points)
//                is reduced and written by its owner alone.  Pieces of a longer
//                interval leave FP32 partial rows in shared memory; after a
//                barrier the owner of the interval's first piece in the round
//                adds them in piece order (plus a carry from the previous
//                round), so the sum order is fixed and the result
//                deterministic.  Per point: one depth load ("depth loaded once
//                per scatter point"), one feature-row gather, FP32 FMAs; up to
//                four points are in flight per owner.  Point indices are
//                fetched cooperatively (each lane loads a different point's
//                ranks, warp shuffles broadcast them).
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

#ifndef BEVPOOL_FWD_BATCH
#define BEVPOOL_FWD_BATCH 8     // points in flight per owner (fp16, and E4M3 with narrow lanes)
#endif
#ifndef BEVPOOL_FWD_MIN_CTAS
#define BEVPOOL_FWD_MIN_CTAS 3  // resident CTAs per SM the register budget is sized for
#endif

#ifndef BEVPOOL_FWD_LANE_BYTES
#define BEVPOOL_FWD_LANE_BYTES 16   // bytes of a feature row each lane loads (16 or 32) for wide rows
#endif

#ifndef BEVPOOL_FMA_VARIANT
#define BEVPOOL_FMA_VARIANT 1   // 0: convert to f32 + FFMA, 1: f16 x f16 + f32 FMA, 2: convert + packed f32x2 FMA
#endif

namespace bevpool {

constexpr int kDtypeF16 = 0;
constexpr int kDtypeE4M3 = 1;
constexpr int kFillCells = 256;
constexpr int kMaxChunk = 1024;     // max intervals per compute CTA

template <int DT, int C>
struct FwdShape {
    static constexpr int EB = DT == kDtypeF16 ? 2 : 1;          // input bytes per element
    static constexpr int ROWB = C * EB;                         // bytes per feature row
    static constexpr int VB = ROWB >= 4 * BEVPOOL_FWD_LANE_BYTES && ROWB % BEVPOOL_FWD_LANE_BYTES == 0
                                  ? BEVPOOL_FWD_LANE_BYTES
                                  : (ROWB >= 64 ? 16 : ROWB / 4);   // bytes per lane (>= 4 lanes per owner)
    static constexpr int LPO = ROWB / VB;                       // lanes per owner
    static constexpr int EPL = VB / EB;                         // channels per lane
    static constexpr int OPW = 32 / LPO;                        // owners per warp
    static constexpr int OWNERS = kWarps * OPW;                 // owners per CTA
    static constexpr int BATCH_CFG = VB >= 32 ? 4 : ((DT == kDtypeF16 || VB < 16) ? BEVPOOL_FWD_BATCH : 4);
    static constexpr int BATCH = BATCH_CFG < LPO ? BATCH_CFG : LPO;   // points in flight per owner (<= LPO)
    static constexpr int OUT_VECS = C * 2 / 16;                 // 16-byte fp16 vectors per out row
    static_assert(ROWB % VB == 0 && (VB == 2 || VB == 4 || VB == 8 || VB == 16 || VB == 32), "bad vector width");
    static_assert(LPO >= 4 && LPO <= 32, "bad lane mapping");
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
    int ipc;                      // intervals per compute CTA (<= kMaxChunk)
    int n_fill;                   // fill CTAs
    __half *out;
};

// ---------------------------------------------------------------- element access

// Depth value as an fp16 bit pattern (E4M3 values are exact in fp16).
template <int DT>
__device__ __forceinline__ unsigned short load_depth_h(const void *depth, int idx) {
    if constexpr (DT == kDtypeF16) {
        return __ldg(static_cast<const unsigned short *>(depth) + idx);
    } else {
        const unsigned char b = __ldg(static_cast<const unsigned char *>(depth) + idx);
        const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
        return h.x;
    }
}

template <int VB>
struct RawVec {
    static constexpr int NW = VB >= 4 ? VB / 4 : 1;
    uint32_t w[NW];
};

template <int VB>
__device__ __forceinline__ RawVec<VB> load_vec(const unsigned char *p) {
    RawVec<VB> r;
    if constexpr (VB == 32) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
        r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
        r.w[4] = u.x; r.w[5] = u.y; r.w[6] = u.z; r.w[7] = u.w;
    } else if constexpr (VB == 16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
    } else if constexpr (VB == 8) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
        r.w[0] = v.x; r.w[1] = v.y;
    } else if constexpr (VB == 4) {
        r.w[0] = __ldg(reinterpret_cast<const unsigned int *>(p));
    } else {
        r.w[0] = __ldg(reinterpret_cast<const unsigned short *>(p));
    }
    return r;
}

// acc[0], acc[1] += d * (lo, hi) for one packed pair of fp16 values.
__device__ __forceinline__ void fma_h2(float &a0, float &a1, unsigned short d, uint32_t pair) {
#if BEVPOOL_FMA_VARIANT == 1
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "fma.rn.f32.f16 %0, %3, lo, %0;\n\tfma.rn.f32.f16 %1, %3, hi, %1;\n\t}"
        : "+f"(a0), "+f"(a1) : "r"(pair), "h"(d));
#else
    __half2_raw hr;
    hr.x = static_cast<unsigned short>(pair & 0xffffu);
    hr.y = static_cast<unsigned short>(pair >> 16);
    const float2 f = __half22float2(__half2(hr));
    __half_raw dr;
    dr.x = d;
    const float df = __half2float(__half(dr));
#if BEVPOOL_FMA_VARIANT == 2
    unsigned long long acc, fv, dv;
    asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(fv) : "f"(f.x), "f"(f.y));
    asm("mov.b64 %0, {%1, %1};" : "=l"(dv) : "f"(df));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(dv), "l"(fv));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
#else
    a0 = fmaf(df, f.x, a0);
    a1 = fmaf(df, f.y, a1);
#endif
#endif
}

// acc[0 .. EPL) += d * decode(raw)
template <int DT, int VB>
__device__ __forceinline__ void fma_vec(float *acc, unsigned short d, const RawVec<VB> &raw) {
    if constexpr (DT == kDtypeF16) {
        if constexpr (VB == 2) {
            __half_raw hr;
            hr.x = static_cast<unsigned short>(raw.w[0]);
            __half_raw dr;
            dr.x = d;
            acc[0] = fmaf(__half2float(__half(dr)), __half2float(__half(hr)), acc[0]);
        } else {
#pragma unroll
            for (int i = 0; i < VB / 4; ++i) fma_h2(acc[2 * i], acc[2 * i + 1], d, raw.w[i]);
        }
    } else {
        if constexpr (VB == 2) {
            const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(raw.w[0]), __NV_E4M3);
            fma_h2(acc[0], acc[1], d, static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16));
        } else {
#pragma unroll
            for (int i = 0; i < VB / 4; ++i) {
                const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                    static_cast<__nv_fp8x2_storage_t>(raw.w[i] & 0xffffu), __NV_E4M3);
                const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                    static_cast<__nv_fp8x2_storage_t>(raw.w[i] >> 16), __NV_E4M3);
                fma_h2(acc[4 * i + 0], acc[4 * i + 1], d, static_cast<uint32_t>(lo.x) | (static_cast<uint32_t>(lo.y) << 16));
                fma_h2(acc[4 * i + 2], acc[4 * i + 3], d, static_cast<uint32_t>(hi.x) | (static_cast<uint32_t>(hi.y) << 16));
            }
        }
    }
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Store EPL channels (scaled, rounded to fp16) at dst (2*EPL bytes, aligned).
template <int EPL>
__device__ __forceinline__ void store_row_part(__half *dst, const float *acc, float scale, bool streaming) {
    constexpr int NW = EPL / 2;   // 32-bit words
    uint32_t w[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = pack_half2(acc[2 * i] * scale, acc[2 * i + 1] * scale);
    if constexpr (NW % 4 == 0) {
#pragma unroll
        for (int q = 0; q < NW / 4; ++q) {
            const uint4 v = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            uint4 *p = reinterpret_cast<uint4 *>(dst) + q;
            if (streaming) __stcs(p, v); else *p = v;
        }
    } else if constexpr (NW == 2) {
        const uint2 v = make_uint2(w[0], w[1]);
        uint2 *p = reinterpret_cast<uint2 *>(dst);
        if (streaming) __stcs(p, v); else *p = v;
    } else {
        unsigned int *p = reinterpret_cast<unsigned int *>(dst);
        if (streaming) __stcs(p, w[0]); else *p = w[0];
    }
}

// ---------------------------------------------------------------- compute CTA

template <int DT, int C>
struct ComputeSmem {
    using S = FwdShape<DT, C>;
    int pre[kMaxChunk + 1];                       // exclusive prefix of interval lengths
    int bev[kMaxChunk];                           // output row of each interval (-1: skip)
    int len[kMaxChunk];
    __align__(16) float slot[2][S::OWNERS][C];    // partial rows of split (long) intervals
};

struct FillSmem {
    unsigned mark[kFillCells / 32];
};

template <int DT, int C>
union FwdSmem {
    ComputeSmem<DT, C> c;
    FillSmem f;
};

// Interval k of the chunk that holds virtual point v (pre[k] <= v < pre[k+1]),
// for 0 <= v < pre[nI]; empty intervals are never returned.
__device__ __forceinline__ int interval_of(const int *pre, int nI, int v) {
    int lo = 0, hi = nI;                           // pre[lo] <= v < pre[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= v) lo = mid; else hi = mid;
    }
    return lo;
}

// Writes acc (one owner's share of a row) either to the output row or to a
// partial slot in shared memory.
template <int DT, int C>
__device__ __forceinline__ void flush_row(const FwdParams &p, ComputeSmem<DT, C> &sm, const float *acc, int bev,
                                          int where, int o, int ol) {
    using S = FwdShape<DT, C>;
    if (where < 0) {
        if (bev >= 0)
            store_row_part<S::EPL>(p.out + static_cast<int64_t>(bev) * C + ol * S::EPL, acc, p.scale, p.streaming);
    } else {
        float *dst = &sm.slot[where][o][ol * S::EPL];
#pragma unroll
        for (int e = 0; e < S::EPL; ++e) dst[e] = acc[e];
    }
}

template <int DT, int C>
__device__ __forceinline__ void compute_cta(const FwdParams &p, int cidx, ComputeSmem<DT, C> &sm) {
    using S = FwdShape<DT, C>;
    __shared__ int scratch[kWarps + 1];
    __shared__ int s_t0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    int n_int = p.n_intervals, n_pts = p.n_points;
    if (p.d_counts) {
        n_int = min(n_int, __ldg(p.d_counts + 1));
        n_pts = min(n_pts, __ldg(p.d_counts + 0));
    }
    const int ipc = p.ipc;
    const int i0 = cidx * ipc;
    if (i0 >= n_int) return;                       // uniform over the CTA
    const int nI = min(ipc, n_int - i0);

    // 1. chunk metadata: thread t owns intervals [t*ipt, t*ipt + ipt) (blocked, for the scan)
    const int ipt = (ipc + kThreads - 1) / kThreads;
    const int kb = threadIdx.x * ipt;
    int my_sum = 0;
    bool ok = true;
    int prev_end = -1;
    int first_start = -1;
    for (int q = 0; q < ipt; ++q) {
        const int k = kb + q;
        if (k >= nI) break;
        const int s = __ldg(p.starts + i0 + k);
        int L = __ldg(p.lengths + i0 + k);
        int cell = -1;
        if (s < 0 || L < 1 || s > n_pts - L) {
            ok = false;
            L = 0;
        } else {
            cell = __ldg(p.ranks_bev + s);
            if (cell < 0 || cell >= p.n_cells) cell = -1;
        }
        if (q == 0) first_start = s; else if (s != prev_end) ok = false;
        prev_end = s + L;
        sm.len[k] = L;
        sm.bev[k] = cell;
        my_sum += L;
    }
    if (threadIdx.x == 0) s_t0 = first_start;
    int P;
    const int excl = cta_exclusive_sum(my_sum, scratch, &P);   // has barriers: s_t0 visible after
    for (int q = 0; q < ipt; ++q) {
        const int k = kb + q;
        if (k >= nI) break;
        sm.pre[k] = excl + (q ? sm.pre[k - 1] - excl + sm.len[k - 1] : 0);
    }
    if (threadIdx.x == 0) sm.pre[nI] = P;
    // contiguity across threads: my first interval must start where the chunk's
    // points up to it end (start = t0 + prefix)
    if (kb < nI && first_start != s_t0 + excl) ok = false;
    const bool chunk_ok = __syncthreads_and(ok) != 0;
    if (!chunk_ok) return;                          // malformed map: unspecified output, no OOB access
    const int T0 = s_t0;

    // 2. owners take equal shares of the chunk's points and walk them in
    //    lockstep (same trip count for every owner of a warp); an interval cut
    //    by a share boundary leaves partial rows for the combine below.
    const int og = lane / S::LPO;                  // owner within warp
    const int ol = lane % S::LPO;                  // lane within owner
    const bool active = og < S::OPW;
    const int o = active ? warp * S::OPW + og : 0;
    const int lane0 = og * S::LPO;
    const unsigned gmask = (S::LPO == 32 ? 0xffffffffu : ((1u << S::LPO) - 1u)) << lane0;
    const unsigned char *featp = static_cast<const unsigned char *>(p.feat) + ol * S::VB;
    const int share = (P + S::OWNERS - 1) / S::OWNERS;
    const int beg = active ? min(P, o * share) : P;
    const int end = active ? min(P, beg + share) : P;

    int head_k = -1;
    if (active) {
        int k = beg < P ? interval_of(sm.pre, nI, beg) : nI - 1;
        int next_end = sm.pre[k + 1];
        bool seg_head = sm.pre[k] == beg;
        float acc[S::EPL];
#pragma unroll
        for (int e = 0; e < S::EPL; ++e) acc[e] = 0.f;
        // indices of the first batch: lane ol holds point beg + ol (ol < BATCH)
        int rd = -1, rf = -1;
        auto fetch_idx = [&](int v0, int &ra, int &rb) {
            ra = -1;
            rb = -1;
            const int j = v0 + ol;
            if (ol < S::BATCH && j < end) {
                const int x = __ldg(p.ranks_depth + T0 + j);
                const int y = __ldg(p.ranks_feat + T0 + j);
                if (x >= 0 && x < p.n_depth && y >= 0 && y < p.n_feat_rows) {
                    ra = x;
                    rb = y;
                }
            }
        };
        fetch_idx(beg, rd, rf);
        for (int v0 = beg; v0 < beg + share; v0 += S::BATCH) {
            int rd_next, rf_next;
            fetch_idx(v0 + S::BATCH, rd_next, rf_next);      // prefetch the next batch's indices
            int a[S::BATCH], b[S::BATCH];
#pragma unroll
            for (int kk = 0; kk < S::BATCH; ++kk) {
                a[kk] = __shfl_sync(gmask, rd, lane0 + kk);
                b[kk] = __shfl_sync(gmask, rf, lane0 + kk);
            }
            unsigned short d[S::BATCH];
            RawVec<S::VB> f[S::BATCH];
#pragma unroll
            for (int kk = 0; kk < S::BATCH; ++kk) {
                if (a[kk] >= 0) {
                    d[kk] = load_depth_h<DT>(p.depth, a[kk]);
                    f[kk] = load_vec<S::VB>(featp + static_cast<int64_t>(b[kk]) * S::ROWB);
                } else {
                    d[kk] = 0;
#pragma unroll
                    for (int i = 0; i < RawVec<S::VB>::NW; ++i) f[kk].w[i] = 0u;
                }
            }
#pragma unroll
            for (int kk = 0; kk < S::BATCH; ++kk) {
                const int v = v0 + kk + 1;                   // points done after this one
                if (v <= end) {
                    fma_vec<DT, S::VB>(acc, d[kk], f[kk]);
                    if (v == next_end) {                    // interval k ends with this point
                        flush_row<DT, C>(p, sm, acc, sm.bev[k], seg_head ? -1 : 0, o, ol);
#pragma unroll
                        for (int e = 0; e < S::EPL; ++e) acc[e] = 0.f;
                        seg_head = true;
                        if (v < end) {
                            ++k;
                            next_end = sm.pre[k + 1];
                        }
                    }
                }
            }
            rd = rd_next;
            rf = rf_next;
        }
        if (beg < end && end < next_end && end > sm.pre[k]) {   // share ends inside interval k
            if (seg_head) {
                flush_row<DT, C>(p, sm, acc, -1, 1, o, ol);
                head_k = k;
            } else {
                flush_row<DT, C>(p, sm, acc, -1, 0, o, ol);
            }
        }
    }

    // 3. combine cut intervals in owner order
    __syncthreads();
    if (head_k >= 0) {
        float acc[S::EPL];
        const float *src = &sm.slot[1][o][ol * S::EPL];
#pragma unroll
        for (int e = 0; e < S::EPL; ++e) acc[e] = src[e];
        const int stop = sm.pre[head_k + 1];
        for (int o2 = o + 1; o2 < S::OWNERS; ++o2) {
            const int b2 = min(P, o2 * share);
            if (b2 >= stop) break;
            const float *q = &sm.slot[0][o2][ol * S::EPL];
#pragma unroll
            for (int e = 0; e < S::EPL; ++e) acc[e] += q[e];
        }
        flush_row<DT, C>(p, sm, acc, sm.bev[head_k], -1, o, ol);
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
__global__ void __launch_bounds__(kThreads, BEVPOOL_FWD_MIN_CTAS) k_forward(const FwdParams p) {
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
    // Chunk size: about one resident wave of compute CTAs, but at least one
    // interval per owner and at most kMaxChunk.
    const int64_t slots = static_cast<int64_t>(a.sm_count > 0 ? a.sm_count : 148) * BEVPOOL_FWD_MIN_CTAS;
    int64_t ipc = div_up(a.n_intervals, slots);
    if (ipc < S::OWNERS) ipc = S::OWNERS;
    if (ipc > kMaxChunk) ipc = kMaxChunk;
    p.ipc = static_cast<int>(ipc);
    p.n_compute = static_cast<int>(div_up(a.n_intervals, ipc));
    p.n_fill = static_cast<int>(div_up(a.n_cells, kFillCells));
    p.out = static_cast<__half *>(a.out);
    const int grid = p.n_compute + p.n_fill;
    k_forward<DT, C><<<grid, kThreads, 0, a.stream>>>(p);
    count_launch();
    return cudaGetLastError();
}

}  // namespace bevpool
