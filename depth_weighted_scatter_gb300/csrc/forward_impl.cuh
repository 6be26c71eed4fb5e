// forward_impl.cuh -- the BEV-pooling forward kernel (sm_103a), templated on
// input dtype, channel count, output type and kernel variant.  Included by the
// forward_*.cu units, one per (input, output) pair.
//
// Computes, for every interval of the scatter map ("Accelerating BEV Pooling
// on NVIDIA GPUs for Physical AI Applications", sections "Eliminate redundant
// scatter traffic" and "Implement interval-owned scatter-reduce"),
//     out[bev, :] = scale * sum_{t in interval} depth[ranks_depth[t]] * feat[ranks_feat[t], :]
// in FP32, rounded once to the output type (fp16, or E4M3 codes of
// value / out_scale), and writes every other cell as zeros, so
// each output row is written exactly once and no atomics are used.
//
// One launch, two kinds of CTA: compute CTAs take the first block indices (the
// long ones), fill CTAs the rest and run in the slots the compute CTAs leave
// or free:
//
//   compute CTA  owns a chunk of consecutive intervals, i.e. a contiguous
//                range of the sorted point arrays with about the same number
//                of points as every other compute CTA.  It works in rounds:
//                the whole CTA first stages the round's points in shared
//                memory (coalesced loads of the three rank arrays, the depth
//                gather "once per scatter point", and one 16-byte record per
//                point with the feature row, the depth value and an
//                interval-end bit from the change of ranks_bev), then the
//                owners walk the records.  An owner is the LPO lanes that
//                together hold one C-channel row (VB bytes per lane); owners
//                take equal shares of the round and walk them independently,
//                BATCH rows in flight each.  At an interval end the owner
//                rounds its FP32 row to the output type and stores it.  An
//                interval cut by a share boundary leaves FP32 partial rows in
//                shared memory; after a barrier the owner that started it
//                adds them in owner order, so the sum order is fixed and the
//                result deterministic.
//
//   fill CTA     owns a tile of 256-1024 consecutive cells.  It finds the
//                tile's points in the sorted ranks_bev with a CTA-wide k-ary
//                search (2-3 dependent loads), marks the cells that have
//                points, and writes zeros to the rest with 16-byte stores.
//                This keeps the (large, uneven) empty regions of the grid off
//                the interval owners and spreads them evenly over the GPU.
#pragma once

#include <climits>
#include <type_traits>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "bevpool_internal.cuh"

// Launch and inner-loop constants, each chosen by timing it against
// alternatives on GB300; each can be overridden with -D.
#ifndef BEVPOOL_FWD_MIN_CTAS
#define BEVPOOL_FWD_MIN_CTAS 3            // resident CTAs per SM the register budget (80) is sized for
#endif
#ifndef BEVPOOL_FWD_LANE_BYTES
#define BEVPOOL_FWD_LANE_BYTES 16         // bytes of an fp16 feature row one lane loads (16 or 32)
#endif
#ifndef BEVPOOL_FWD_E4M3_LANE_BYTES
#define BEVPOOL_FWD_E4M3_LANE_BYTES 8     // bytes of an E4M3 feature row one lane loads
#endif
#ifndef BEVPOOL_FWD_BATCH
#define BEVPOOL_FWD_BATCH 6               // points in flight per owner: fp16 rows
#endif
#ifndef BEVPOOL_FWD_E4M3_BATCH8
#define BEVPOOL_FWD_E4M3_BATCH8 6         // E4M3 rows at 8 B or less a lane
#endif
#ifndef BEVPOOL_FWD_E4M3_BATCH16
#define BEVPOOL_FWD_E4M3_BATCH16 5        // E4M3 rows at 16 B a lane (5 rows of 16 B beside 16 FP32 sums)
#endif
#ifndef BEVPOOL_FWD_BATCH32
#define BEVPOOL_FWD_BATCH32 4             // rows at 32 B a lane
#endif
#ifndef BEVPOOL_FWD_NVFP4_BATCH
#define BEVPOOL_FWD_NVFP4_BATCH 6         // NVFP4 rows (one 16-element block a lane)
#endif
#ifndef BEVPOOL_FWD_LEAN_BATCH
#define BEVPOOL_FWD_LEAN_BATCH 6          // fp16 rows, output streaming to DRAM: points in flight per owner
#endif
#ifndef BEVPOOL_FWD_E4M3_LEAN_BATCH
#define BEVPOOL_FWD_E4M3_LEAN_BATCH 4     // E4M3 rows in the lean variant (output streaming to DRAM)
#endif
#ifndef BEVPOOL_FWD_SHORT_BATCH
#define BEVPOOL_FWD_SHORT_BATCH 6         // fp16 rows, short intervals: points in flight per owner (80 registers)
#endif
#ifndef BEVPOOL_FWD_LEAN_SHORT_BATCH
#define BEVPOOL_FWD_LEAN_SHORT_BATCH 4    // fp16 rows, lean variant with short intervals
#endif
#ifndef BEVPOOL_FWD_LEAN_MIN_CTAS
#define BEVPOOL_FWD_LEAN_MIN_CTAS 4       // ... with four CTAs per SM (64 registers), all computing
#endif
#ifndef BEVPOOL_FWD_MULTIWAVE
#define BEVPOOL_FWD_MULTIWAVE 64          // > 0: compute CTAs of at most a round less this many points each
#endif
#ifndef BEVPOOL_FWD_STORE_HINT
#define BEVPOOL_FWD_STORE_HINT 1          // 1: output stores take an L2 cache policy instead of a branch
#endif
#ifndef BEVPOOL_FWD_LEAN_WORK_PER_SM
#define BEVPOOL_FWD_LEAN_WORK_PER_SM 131072   // fp16 rows with at least this many point-channels per SM run lean
#endif
// Compute CTAs per SM (one wave of them): with the output resident in L2,
// two, leaving a slot for fill CTAs to run alongside; when the output streams
// to DRAM, three (the gathers need the issue slots more than the fills).
#ifndef BEVPOOL_FWD_WALK_DEPTH_FP8
#define BEVPOOL_FWD_WALK_DEPTH_FP8 1      // 1: E4M3 owners load (and widen) depth values in the walk
#endif
#ifndef BEVPOOL_FWD_WALK_DEPTH
#define BEVPOOL_FWD_WALK_DEPTH 1          // 1: fp16 owners load depth values in the walk (default and lean-short variants)
#endif
#ifndef BEVPOOL_FWD_COMBINE_BATCH
#define BEVPOOL_FWD_COMBINE_BATCH 2       // owners whose partial rows the combine loads at a time
#endif
#ifndef BEVPOOL_FWD_ROUND_MAX_WIDE
#define BEVPOOL_FWD_ROUND_MAX_WIDE 1280   // points per staged round at most, fp16 default and lean-short variants
#endif
#ifndef BEVPOOL_FWD_FILL_AFTER_WAVES
#define BEVPOOL_FWD_FILL_AFTER_WAVES 1    // output streaming to DRAM: fill CTAs follow this many waves of compute CTAs
#endif
#ifndef BEVPOOL_FWD_FILL_PER_SM
#define BEVPOOL_FWD_FILL_PER_SM 4         // output streaming to DRAM: fill tiles grow until this many fill CTAs per SM
#endif
#ifndef BEVPOOL_FWD_CTAS_PER_SM_L2
#define BEVPOOL_FWD_CTAS_PER_SM_L2 2
#endif
#ifndef BEVPOOL_FWD_CTAS_PER_SM_DRAM
#define BEVPOOL_FWD_CTAS_PER_SM_DRAM 3
#endif

namespace bevpool {

constexpr int kDtypeF16 = 0;
constexpr int kDtypeE4M3 = 1;
constexpr int kDtypeNVFP4 = 2;   // E2M1 features with an E4M3 scale per 16 elements, E4M3 depth
constexpr int kOutF16 = 0;     // output element: fp16 (round to nearest even)
constexpr int kOutE4M3 = 1;    // output element: OCP E4M3 code (round to nearest even, saturating)
constexpr int kFillCellsMin = 256;        // cells per fill CTA: a power of two chosen per call, at most
constexpr int kFillCellsMax = 1024;       // kFillCellsMax, at least kFillCellsMin (kFillCellsL2Min with the
constexpr int kFillCellsL2Min = 128;      // output in L2)
constexpr int kFillTileBytesL2 = 80 * 1024;   // output in L2: output bytes of a fill tile at most
constexpr int kFillTilePoints = 1024;         // output in L2: points in a fill tile on average at most

// Kernel variants (a template parameter): the default; lean (fewer points in
// flight, 64 registers, four compute CTAs per SM); short (fp16 rows whose
// intervals are short on average: fewer points in flight at 80 registers);
// lean-short (the lean variant for fp16 rows with short intervals).
constexpr int kVarDefault = 0;
constexpr int kVarLean = 1;
constexpr int kVarShort = 2;
constexpr int kVarLeanShort = 3;

template <int DT, int C, int VAR = 0>
struct FwdShape {
    static constexpr bool LEAN = VAR == kVarLean || VAR == kVarLeanShort;
    static constexpr bool SHORT = VAR == kVarShort;
    static constexpr bool NV = DT == kDtypeNVFP4;
    static constexpr int EB = DT == kDtypeF16 ? 2 : 1;          // input bytes per element (E4M3)
    static constexpr int ROWB = NV ? C / 2 : C * EB;            // bytes per feature row
    static constexpr int LANE_BYTES = DT == kDtypeF16 ? BEVPOOL_FWD_LANE_BYTES : BEVPOOL_FWD_E4M3_LANE_BYTES;
    static constexpr int VB = NV ? 8                            // NVFP4: one 16-element block per lane
                              : (ROWB >= 4 * LANE_BYTES && ROWB % LANE_BYTES == 0
                                     ? LANE_BYTES
                                     : (ROWB >= 64 ? 16 : ROWB / 4));   // bytes per lane (>= 4 lanes per owner)
    static constexpr int LPO = ROWB / VB;                       // lanes per owner
    static constexpr int EPL = NV ? 16 : VB / EB;               // channels per lane
    static constexpr int OPW = 32 / LPO;                        // owners per warp
    static constexpr int OWNERS = kWarps * OPW;                 // owners per CTA
    static constexpr int BATCH_CFG = NV                                  ? BEVPOOL_FWD_NVFP4_BATCH
                                     : VB >= 32                          ? BEVPOOL_FWD_BATCH32
                                     : (DT == kDtypeF16 && VAR == kVarLeanShort) ? BEVPOOL_FWD_LEAN_SHORT_BATCH
                                     : (DT == kDtypeF16 && LEAN)         ? BEVPOOL_FWD_LEAN_BATCH
                                     : (DT == kDtypeF16 && SHORT)        ? BEVPOOL_FWD_SHORT_BATCH
                                     : (DT == kDtypeE4M3 && LEAN)        ? BEVPOOL_FWD_E4M3_LEAN_BATCH
                                     : DT == kDtypeF16                   ? BEVPOOL_FWD_BATCH
                                     : VB < 16                           ? BEVPOOL_FWD_E4M3_BATCH8
                                                                         : BEVPOOL_FWD_E4M3_BATCH16;
    static constexpr int BATCH = BATCH_CFG;                       // points in flight per owner
    static_assert(ROWB % VB == 0 && (VB == 2 || VB == 4 || VB == 8 || VB == 16 || VB == 32), "bad vector width");
    static_assert(LPO >= 4 && LPO <= 32, "bad lane mapping");
    static_assert(C % 8 == 0 && (!NV || C % 16 == 0), "C must be a multiple of 8 (16 for NVFP4)");
};

struct FwdParams {
    const void *depth;
    const void *feat;
    const unsigned char *feat_block;   // NVFP4: E4M3 scale of each 16-element block, [rows, C/16]
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
    FastDiv n_compute_div;        // division by n_compute
    int n_fill;                   // fill CTAs
    int fill_cells;               // cells per fill CTA
    int fill_after;               // block index of the first fill CTA (the compute CTAs before it come first)
    unsigned char *out;           // [n_cells, C] elements of the output type
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

// acc[0], acc[1] += d * (lo, hi) for one packed pair of fp16 values: FP32
// FMAs taking the fp16 operands directly (f16 x f16 products are exact in
// FP32).  Measured faster here than widening to f32 first, with or without
// packed f32x2 FMAs.
__device__ __forceinline__ void fma_h2(float &a0, float &a1, unsigned short d, uint32_t pair) {
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "fma.rn.f32.f16 %0, %3, lo, %0;\n\tfma.rn.f32.f16 %1, %3, hi, %1;\n\t}"
        : "+f"(a0), "+f"(a1) : "r"(pair), "h"(d));
}

// acc[0..8) += d * (eight E2M1 codes of w, lowest nibble first): each byte
// widens to two fp16 values in one conversion (exact), then FP32 FMAs.
__device__ __forceinline__ void fma_e2m1x8(float *acc, unsigned short d, uint32_t w) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 p0, p1, p2, p3;\n\t"
        ".reg .f16 h0, h1, h2, h3, h4, h5, h6, h7;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %8;\n\t"
        "cvt.rn.f16x2.e2m1x2 p0, b0;\n\tcvt.rn.f16x2.e2m1x2 p1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 p2, b2;\n\tcvt.rn.f16x2.e2m1x2 p3, b3;\n\t"
        "mov.b32 {h0, h1}, p0;\n\tmov.b32 {h2, h3}, p1;\n\tmov.b32 {h4, h5}, p2;\n\tmov.b32 {h6, h7}, p3;\n\t"
        "fma.rn.f32.f16 %0, %9, h0, %0;\n\tfma.rn.f32.f16 %1, %9, h1, %1;\n\t"
        "fma.rn.f32.f16 %2, %9, h2, %2;\n\tfma.rn.f32.f16 %3, %9, h3, %3;\n\t"
        "fma.rn.f32.f16 %4, %9, h4, %4;\n\tfma.rn.f32.f16 %5, %9, h5, %5;\n\t"
        "fma.rn.f32.f16 %6, %9, h6, %6;\n\tfma.rn.f32.f16 %7, %9, h7, %7;\n\t}"
        : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3]), "+f"(acc[4]), "+f"(acc[5]), "+f"(acc[6]),
          "+f"(acc[7])
        : "r"(w), "h"(d));
}

// Product of two fp16 values given as bits.  Used for depth x block scale of
// NVFP4 rows: both are E4M3 values, so the product (at most 8 significant
// bits, magnitude between 2^-18 and 448) is exact in fp16.
__device__ __forceinline__ unsigned short mul_f16_bits(unsigned short a, unsigned short b) {
    unsigned short r;
    asm("mul.rn.f16 %0, %1, %2;" : "=h"(r) : "h"(a), "h"(b));
    return r;
}

// acc[0..4) += d * (four E4M3 codes of w, lowest byte first): each pair of
// codes widens to two fp16 values in one conversion (exact), then FP32 FMAs.
__device__ __forceinline__ void fma_e4m3x4(float *acc, unsigned short d, uint32_t w) {
    asm("{\n\t.reg .b16 lo, hi;\n\t.reg .b32 p0, p1;\n\t.reg .f16 a0, a1, a2, a3;\n\t"
        "mov.b32 {lo, hi}, %4;\n\t"
        "cvt.rn.f16x2.e4m3x2 p0, lo;\n\tcvt.rn.f16x2.e4m3x2 p1, hi;\n\t"
        "mov.b32 {a0, a1}, p0;\n\tmov.b32 {a2, a3}, p1;\n\t"
        "fma.rn.f32.f16 %0, %5, a0, %0;\n\tfma.rn.f32.f16 %1, %5, a1, %1;\n\t"
        "fma.rn.f32.f16 %2, %5, a2, %2;\n\tfma.rn.f32.f16 %3, %5, a3, %3;\n\t}"
        : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3])
        : "r"(w), "h"(d));
}

// acc[0 .. EPL) += d * decode(raw)
template <int DT, int VB>
__device__ __forceinline__ void fma_vec(float *acc, unsigned short d, const RawVec<VB> &raw) {
    if constexpr (DT == kDtypeNVFP4) {
#pragma unroll
        for (int i = 0; i < VB / 4; ++i) fma_e2m1x8(acc + 8 * i, d, raw.w[i]);
    } else if constexpr (DT == kDtypeF16) {
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
            for (int i = 0; i < VB / 4; ++i) fma_e4m3x4(acc + 4 * i, d, raw.w[i]);
        }
    }
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

#if BEVPOOL_FWD_STORE_HINT
// Output stores carry an L2 cache policy chosen once per thread (evict-first
// when the output streams to DRAM, normal otherwise) and a predicate (whether
// to store at all): one store instruction, no branch at every interval end.
using StoreMode = uint64_t;
__device__ __forceinline__ StoreMode store_mode(bool streaming) {
    uint64_t pol;
    if (streaming)
        asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    else
        asm("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void store_vec(uint4 *p, const uint4 &v, StoreMode m, bool on = true) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %6, 0;\n\t"
                 "@q st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;\n\t}" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(m), "r"(static_cast<unsigned>(on))
                 : "memory");
}
__device__ __forceinline__ void store_vec(uint2 *p, const uint2 &v, StoreMode m, bool on = true) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %4, 0;\n\t"
                 "@q st.global.L2::cache_hint.v2.b32 [%0], {%1, %2}, %3;\n\t}" ::"l"(p), "r"(v.x), "r"(v.y),
                 "l"(m), "r"(static_cast<unsigned>(on))
                 : "memory");
}
__device__ __forceinline__ void store_vec(unsigned int *p, const unsigned int &v, StoreMode m, bool on = true) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t"
                 "@q st.global.L2::cache_hint.b32 [%0], %1, %2;\n\t}" ::"l"(p), "r"(v), "l"(m),
                 "r"(static_cast<unsigned>(on))
                 : "memory");
}
#else
using StoreMode = bool;                            // true: evict-first (streaming) stores
__device__ __forceinline__ StoreMode store_mode(bool streaming) { return streaming; }
template <typename V>
__device__ __forceinline__ void store_vec(V *p, const V &v, StoreMode streaming, bool on = true) {
    if (!on) return;
    if (streaming) __stcs(p, v); else *p = v;
}
#endif

// Store EPL channels, scaled and rounded to the output type, at dst
// (EPL * element bytes, aligned to that size).
template <int OT, int EPL>
__device__ __forceinline__ void store_row_part(unsigned char *dst, const float *acc, float scale, StoreMode streaming,
                                               bool on = true) {
    if constexpr (OT == kOutF16) {
        constexpr int NW = EPL / 2;   // 32-bit words
        uint32_t w[NW];
#pragma unroll
        for (int i = 0; i < NW; ++i) w[i] = pack_half2(acc[2 * i] * scale, acc[2 * i + 1] * scale);
        if constexpr (NW % 4 == 0) {
#pragma unroll
            for (int q = 0; q < NW / 4; ++q)
                store_vec(reinterpret_cast<uint4 *>(dst) + q,
                          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]), streaming, on);
        } else if constexpr (NW == 2) {
            store_vec(reinterpret_cast<uint2 *>(dst), make_uint2(w[0], w[1]), streaming, on);
        } else {
            store_vec(reinterpret_cast<unsigned int *>(dst), w[0], streaming, on);
        }
    } else {
        static_assert(EPL % 4 == 0, "E4M3 rows are stored four codes at a time");
        constexpr int NW = EPL / 4;   // 32-bit words of four codes
        uint32_t w[NW];
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                make_float2(acc[4 * i] * scale, acc[4 * i + 1] * scale), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                make_float2(acc[4 * i + 2] * scale, acc[4 * i + 3] * scale), __NV_SATFINITE, __NV_E4M3);
            w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        if constexpr (NW % 4 == 0) {
#pragma unroll
            for (int q = 0; q < NW / 4; ++q)
                store_vec(reinterpret_cast<uint4 *>(dst) + q,
                          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]), streaming, on);
        } else if constexpr (NW == 2) {
            store_vec(reinterpret_cast<uint2 *>(dst), make_uint2(w[0], w[1]), streaming, on);
        } else {
            store_vec(reinterpret_cast<unsigned int *>(dst), w[0], streaming, on);
        }
    }
}

// ---------------------------------------------------------------- compute CTA

// One point of a compute CTA's chunk, staged in shared memory by the whole
// CTA before the owners walk it (one 16-byte load per point and lane).
struct __align__(16) PointRec {
    int32_t row;        // feature row (ranks_feat); 0 for a skipped point
    uint32_t dflags;    // depth value as fp16 bits | kEndBit | kSkipBit
    int32_t bev;        // cell (ranks_bev)
    int32_t pad;
};
constexpr uint32_t kEndBit = 1u << 16;    // the point is the last of its interval
constexpr uint32_t kSkipBit = 1u << 17;   // a rank is out of range: the point adds nothing
constexpr uint32_t kNoCellBit = 1u << 18; // the cell is out of range: its interval is not stored

template <int DT, int C, int VAR = 0>
struct ComputeSmem {
    using S = FwdShape<DT, C, VAR>;
    // partial rows: the slot of every owner, and the carry of an interval
    // that runs on into the next round (two buffers, by round parity)
    static constexpr int ROW_BYTES = (S::OWNERS + 2) * C * 4;
    // points per round: as many 16-byte records as fit beside the rows in
    // 46 KB of static shared memory, a multiple of the CTA size, at most 1024
    static constexpr int ROUND_FIT = ((46 * 1024 - ROW_BYTES) / 16) / kThreads * kThreads;
    // fp16 rows of the default and lean-short variants (whose staging has no
    // depth gather) take rounds of up to 1280 points, the rest 1024 (measured
    // warm: BEVDet 9.4 -> 8.3 us, a chunk extended by a long straddling
    // interval no longer needs a second round; DRAM batch 90.3 -> 88.8 us
    // L2-flushed, fewer waves of one-round CTAs; for the short, lean and E4M3
    // rows slower: canonical 10.0 -> 10.5, 572K points 17.9 -> 18.7)
    static constexpr int ROUND_MAX =
        DT == kDtypeF16 && (VAR == kVarDefault || VAR == kVarLeanShort) ? BEVPOOL_FWD_ROUND_MAX_WIDE : 1024;
    static constexpr int ROUND = ROUND_FIT < ROUND_MAX ? ROUND_FIT : ROUND_MAX;
    static_assert(ROUND >= kThreads, "partial rows leave no room for point records");
    PointRec rec[ROUND];
    int state[S::OWNERS];                         // how an owner's share starts (kHead / kCont / kPass / kEmpty)
    int carry_bev[2];
    __align__(16) float slot[S::OWNERS][C];       // first partial row of a share that starts inside an interval
    __align__(16) float carry[2][C];
};

// How an owner's share of a round starts:
constexpr int kHead = 0;    // at the first point of an interval
constexpr int kCont = 1;    // inside an interval that ends within the share: its partial is in the slot
constexpr int kPass = 2;    // inside an interval that runs through the whole share: its partial is in the slot
constexpr int kEmpty = 3;   // the share is empty (the last owners of a short round)

struct FillSmem {
    unsigned mark[kFillCellsMax / 32];
};

template <int DT, int C, int VAR = 0>
union FwdSmem {
    ComputeSmem<DT, C, VAR> c;
    FillSmem f;
};

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

// First interval start at or after x: the smallest t >= x with t == n or
// ranks_bev[t] != ranks_bev[t - 1] (t == 0 counts as a start), for x0 and x1
// at once.  One CTA-wide probe of kThreads points each; a window without a
// start (an interval longer than kThreads) falls back to a k-ary search of
// interval_starts.  Contains barriers.
__device__ __forceinline__ void cta_next_starts(const FwdParams &p, int n, int n_int, int x0, int x1, int *t0,
                                                int *t1, int *s) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < 2) s[threadIdx.x] = INT_MAX;
    __syncthreads();
    const int i = threadIdx.x;
    const int xs[2] = {x0, x1};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int x = xs[k];
        bool hit = false;
        if (i <= n - x) {                                   // t = x + i <= n
            const int t = x + i;
            hit = t == 0 || t == n || __ldg(p.ranks_bev + t) != __ldg(p.ranks_bev + t - 1);
        }
        const unsigned bal = __ballot_sync(0xffffffffu, hit);
        if (lane == 0 && bal) atomicMin(&s[k], x + warp * 32 + __ffs(bal) - 1);
    }
    __syncthreads();
    int r0 = s[0], r1 = s[1];
    if (r0 == INT_MAX || r1 == INT_MAX) {                   // uniform over the CTA
        int j0, j1;
        cta_lower_bound2(p.starts, max(n_int, 0), x0, x1, &j0, &j1);
        if (r0 == INT_MAX) r0 = j0 < n_int ? __ldg(p.starts + j0) : n;
        if (r1 == INT_MAX) r1 = j1 < n_int ? __ldg(p.starts + j1) : n;
    }
    *t0 = min(max(r0, 0), n);
    *t1 = min(max(r1, *t0), n);
}

// acc[0 .. EPL) of an interval: to the output row of cell bev, scaled and
// rounded; nothing is stored unless `on` (the cell is in range).
template <int OT, int C, int EPL>
__device__ __forceinline__ void store_interval(const FwdParams &p, int bev, int ol, const float *acc, StoreMode mode,
                                               bool on) {
    constexpr int OB = OT == kOutF16 ? 2 : 1;
    store_row_part<OT, EPL>(p.out + (static_cast<int64_t>(bev) * C + ol * EPL) * OB, acc, p.scale, mode, on);
}

template <int DT, int C, int OT, int VAR>
__device__ __forceinline__ void compute_cta(const FwdParams &p, int cidx, ComputeSmem<DT, C, VAR> &sm) {
    using S = FwdShape<DT, C, VAR>;
    using SM = ComputeSmem<DT, C, VAR>;
    constexpr int U = S::BATCH;                    // points in flight per owner
    // fp16 rows in the default and lean-short variants, and E4M3 rows: the
    // owners load each point's depth value beside its row (one dependent round
    // trip less in staging; measured: DRAM batch 93.4 -> 91.1 us L2-flushed,
    // 86.8 -> 84.9 warm; C = 128 13.7 -> 13.1 warm; BEVDet 10.0 -> 9.9 warm
    // with six points in flight instead of eight; canonical FP8 10.5 -> 10.0
    // warm, 572K FP8 points 19.3 -> 18.3).  The fp16 short variant keeps the
    // staged value (canonical warm 10.5 -> 10.4 but L2-flushed 16.4 -> 16.9
    // us), as does the plain fp16 lean variant (8.7-point intervals: 18.1 ->
    // 20.2 us warm), and NVFP4 rows (canonical 11.8 -> 12.3 us warm).
    constexpr bool WALKD = BEVPOOL_FWD_WALK_DEPTH &&
                           ((DT == kDtypeF16 && (VAR == kVarDefault || VAR == kVarLeanShort)) ||
                            (DT == kDtypeE4M3 && BEVPOOL_FWD_WALK_DEPTH_FP8));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    __shared__ int s_bounds[2];
    int n_int = p.n_intervals, n_pts = p.n_points;
    if (p.d_counts) {
        n_int = min(n_int, __ldg(p.d_counts + 1));
        n_pts = min(n_pts, __ldg(p.d_counts + 0));
    }
    if (n_pts <= 0) return;                        // uniform over the CTA

    // 1. the CTA's points: [cidx * ppc, (cidx + 1) * ppc) with both ends moved
    //    forward to interval starts (T0, T1), so no interval is split between
    //    CTAs and every CTA gets about the same number of points.  The
    //    starts are found in the staged windows themselves; only a window
    //    without any start (one long interval) falls back to a search.
    const int ppc = static_cast<int>(p.n_compute_div.div(static_cast<uint32_t>(n_pts - 1))) + 1;
    const int64_t x0l = static_cast<int64_t>(cidx) * ppc;
    if (x0l >= n_pts) return;
    const int x0 = static_cast<int>(x0l);
    const int x1 = static_cast<int>(min(static_cast<int64_t>(n_pts), x0l + ppc));
    __shared__ int s_min[2][kWarps];

    const int og = lane / S::LPO;                  // owner within warp
    const int ol = lane % S::LPO;                  // lane within owner
    const bool active = og < S::OPW;
    const int o = active ? warp * S::OPW + og : 0;
    const unsigned char *featp = static_cast<const unsigned char *>(p.feat) + ol * S::VB;
    [[maybe_unused]] const unsigned char *blockp = p.feat_block + ol;   // NVFP4: the lane's block scale
    const StoreMode mode = store_mode(p.streaming != 0);

    int T0 = -1, T1 = -1;                          // known once found (uniform over the CTA)
    int w0 = x0;                                   // first point of the staged window
    bool round_head = true;                        // the round's first point starts an interval
    for (int rnd = 0;; ++rnd) {
        const int W = min(SM::ROUND, n_pts - w0);
        const int cb = rnd & 1;                    // carry buffer read this round (the other is written)

        // 2. stage the window [w0, w0 + W): every thread takes points tid,
        //    tid + 256, ...; all rank loads first, then the depth gathers,
        //    then the records.
        constexpr int K = SM::ROUND / kThreads;
        int cell[K], prv[K], nxt[K], rx[K], ry[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int i = threadIdx.x + k * kThreads;
            const int t = w0 + i;
            cell[k] = prv[k] = nxt[k] = rx[k] = ry[k] = -1;
            if (i < W) {
                cell[k] = __ldg(p.ranks_bev + t);
                if (t > 0) prv[k] = __ldg(p.ranks_bev + t - 1);
                if (t + 1 < n_pts) nxt[k] = __ldg(p.ranks_bev + t + 1);
                rx[k] = __ldg(p.ranks_depth + t);
                ry[k] = __ldg(p.ranks_feat + t);
            }
        }
        bool skip_any = false;
        int f0 = INT_MAX, f1 = INT_MAX;            // first interval start at or after x0 / x1
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int i = threadIdx.x + k * kThreads;
            const int t = w0 + i;
            if (i < W) {
                const bool ok = rx[k] >= 0 && rx[k] < p.n_depth && ry[k] >= 0 && ry[k] < p.n_feat_rows;
                const bool start = t == 0 || prv[k] != cell[k];
                const bool end = t + 1 == n_pts || nxt[k] != cell[k];
                if (start) {
                    f0 = min(f0, t);
                    if (t >= x1) f1 = min(f1, t);
                }
                PointRec q;
                uint32_t d = 0u;
                if constexpr (WALKD) {
                    q.pad = ok ? rx[k] : 0;            // the owners load the depth value beside the row
                } else {
                    d = ok ? load_depth_h<DT>(p.depth, rx[k]) : 0u;
                    q.pad = 0;
                }
                q.row = ok ? ry[k] : 0;
                q.dflags = d | (end ? kEndBit : 0u) | (ok ? 0u : kSkipBit) |
                           ((cell[k] >= 0 && cell[k] < p.n_cells) ? 0u : kNoCellBit);
                q.bev = cell[k];
                sm.rec[i] = q;
                skip_any |= !ok;
            }
        }
        f0 = __reduce_min_sync(0xffffffffu, f0);
        f1 = __reduce_min_sync(0xffffffffu, f1);
        if (lane == 0) {
            s_min[0][warp] = f0;
            s_min[1][warp] = f1;
        }
        const bool checked = __syncthreads_or(skip_any);   // some point of the round is skipped
        int m0 = INT_MAX, m1 = INT_MAX;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            m0 = min(m0, s_min[0][w]);
            m1 = min(m1, s_min[1][w]);
        }
        if (T0 < 0) {
            if (m0 == INT_MAX) {                   // the window lies inside one interval
                cta_next_starts(p, n_pts, n_int, x0, x1, &T0, &T1, s_bounds);   // contains barriers
                if (T1 <= T0) return;              // uniform: the CTA before owns these points
                w0 = T0;                           // stage again from the chunk's first point
                rnd = -1;
                continue;
            }
            T0 = m0;
        }
        if (T1 < 0) {
            if (m1 != INT_MAX) T1 = m1;
            else if (w0 + W >= n_pts) T1 = n_pts;
        }
        if (T1 >= 0 && T1 <= T0) return;           // no interval starts in [x0, x1): the CTA before owns them
        // the chunk's points in this window: records [lo, hi)
        const int lo = max(T0, w0) - w0;
        const int hi = (T1 >= 0 ? min(T1, w0 + W) : w0 + W) - w0;
        const int R = hi - lo;
        const bool first_head = T0 >= w0 ? true : round_head;

        // 3. owners take equal shares of the round and walk them, U points
        //    at a time.  A share that starts inside an interval leaves its
        //    first partial row in its slot; a share that ends inside an
        //    interval it started keeps that partial in registers and adds the
        //    later owners' slots after the barrier.
        const int share = (R + S::OWNERS * U - 1) / (S::OWNERS * U) * U;   // whole groups where possible
        const int beg = lo + min(R, o * share);
        const int end = lo + min(R, o * share + share);
        const bool next_head = (sm.rec[W - 1].dflags & kEndBit) != 0u;
        bool head_cut = false;                     // this owner finishes an interval cut by its share end
        int head_bev = -1;
        float acc[S::EPL];                         // after the walk: the partial row of that interval
        if (active) {
            int st = kEmpty;
            if (beg < end) {
                const bool head = beg == lo ? first_head : (sm.rec[beg - 1].dflags & kEndBit) != 0u;
                bool to_slot = !head;              // the next finished segment continues a previous share
#pragma unroll
                for (int e = 0; e < S::EPL; ++e) acc[e] = 0.f;
                // n < U (a share's tail) or a round with skipped points: checked walk
                auto walk = [&](int v, int n, auto full_tag) {
                    constexpr bool FULL = decltype(full_tag)::value;
                    int rows[U];
                    uint32_t df[U];
                    [[maybe_unused]] int dix[U];           // depth index (depth loaded here, not staged)
#pragma unroll
                    for (int kk = 0; kk < U; ++kk) {
                        if (FULL || kk < n) {
                            const int4 q = *reinterpret_cast<const int4 *>(&sm.rec[v + kk]);
                            rows[kk] = q.x;
                            df[kk] = static_cast<uint32_t>(q.y);
                            if constexpr (WALKD) dix[kk] = q.w;
                        } else {
                            rows[kk] = 0;
                            df[kk] = kSkipBit;
                            if constexpr (WALKD) dix[kk] = 0;
                        }
                    }
                    [[maybe_unused]] unsigned short dw[U];
                    if constexpr (WALKD) {
#pragma unroll
                        for (int kk = 0; kk < U; ++kk) dw[kk] = load_depth_h<DT>(p.depth, dix[kk]);
                    }
                    RawVec<S::VB> f[U];
                    [[maybe_unused]] unsigned short sh[U];
#pragma unroll
                    for (int kk = 0; kk < U; ++kk) {
                        if (FULL || kk < n) {              // skipped points load row 0 and add nothing
                            f[kk] = load_vec<S::VB>(featp + static_cast<int64_t>(rows[kk]) * S::ROWB);
                            if constexpr (S::NV) {
                                const unsigned char sc = __ldg(blockp + static_cast<int64_t>(rows[kk]) * (C / 16));
                                sh[kk] = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(sc), __NV_E4M3).x;
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < RawVec<S::VB>::NW; ++i) f[kk].w[i] = 0u;
                            if constexpr (S::NV) sh[kk] = 0;
                        }
                    }
#pragma unroll
                    for (int kk = 0; kk < U; ++kk) {
                        unsigned short d = WALKD ? dw[kk] : static_cast<unsigned short>(df[kk] & 0xffffu);
                        if constexpr (S::NV) d = mul_f16_bits(d, sh[kk]);   // depth x block scale (exact in fp16)
                        if (FULL || !(df[kk] & kSkipBit)) fma_vec<DT, S::VB>(acc, d, f[kk]);
                        if (df[kk] & kEndBit) {                // an interval ends with this point
                            if (to_slot) {
                                float *dst = &sm.slot[o][ol * S::EPL];
#pragma unroll
                                for (int e = 0; e < S::EPL; ++e) dst[e] = acc[e];
                                to_slot = false;
                            } else {
                                store_interval<OT, C, S::EPL>(p, sm.rec[v + kk].bev, ol, acc, mode,
                                                              !(df[kk] & kNoCellBit));
                            }
#pragma unroll
                            for (int e = 0; e < S::EPL; ++e) acc[e] = 0.f;
                        }
                    }
                };
                int v = beg;
                if (!checked) {
                    for (; v + U <= end; v += U) walk(v, U, std::true_type{});
                }
                for (; v < end; v += U) walk(v, min(U, end - v), std::false_type{});
                const bool cut = (sm.rec[end - 1].dflags & kEndBit) == 0u;   // the share ends inside an interval
                st = head ? kHead : (to_slot && cut ? kPass : kCont);
                if (cut) {
                    if (to_slot) {                 // the whole share continues an earlier interval
                        float *dst = &sm.slot[o][ol * S::EPL];
#pragma unroll
                        for (int e = 0; e < S::EPL; ++e) dst[e] = acc[e];
                    } else {                       // acc keeps the interval's first part
                        head_cut = true;
                        head_bev = sm.rec[end - 1].bev;
                    }
                }
            }
            if (ol == 0) sm.state[o] = st;
        }

        // 4. combine cut intervals in owner order (fixed order: deterministic).
        //    An interval still open at the round's end goes to the carry; the
        //    first owner's lanes take the carry of the previous round.
        __syncthreads();
        // adds the slots of owners o2, o2 + 1, ... to a until one of them ends
        // the interval (then stores it) or the round ends (then carries it)
        auto finish = [&](float *a, int o2, int bev) {
            // the states and slots of CB owners are loaded together, then
            // added in owner order (the same order and sums as one at a time):
            // an interval that spans many owners (BEVDet: up to 464 points)
            // waits on half as many dependent shared loads (measured warm:
            // BEVDet 8.2 -> 7.9 us; the plain lean variant keeps one at a
            // time, 572K points 17.9 -> 18.1 us with two)
            constexpr int CB = VAR == kVarLean ? 1 : BEVPOOL_FWD_COMBINE_BATCH;
            for (; o2 < S::OWNERS; o2 += CB) {
                int st[CB];
                float q[CB][S::EPL];
#pragma unroll
                for (int j = 0; j < CB; ++j) {
                    const int oj = o2 + j < S::OWNERS ? o2 + j : S::OWNERS - 1;   // in bounds; unused past the end
                    st[j] = o2 + j < S::OWNERS ? sm.state[oj] : kHead;
#pragma unroll
                    for (int e = 0; e < S::EPL; ++e) q[j][e] = sm.slot[oj][ol * S::EPL + e];
                }
#pragma unroll
                for (int j = 0; j < CB; ++j) {
                    if (st[j] == kHead || st[j] == kEmpty) goto carry_out;
#pragma unroll
                    for (int e = 0; e < S::EPL; ++e) a[e] += q[j][e];
                    if (st[j] == kCont) {
                        store_interval<OT, C, S::EPL>(p, bev, ol, a, mode, bev >= 0 && bev < p.n_cells);
                        return;
                    }
                }
            }
        carry_out:
            float *dst = &sm.carry[cb ^ 1][ol * S::EPL];
#pragma unroll
            for (int e = 0; e < S::EPL; ++e) dst[e] = a[e];
            if (ol == 0) sm.carry_bev[cb ^ 1] = bev;
        };
        if (!first_head && active && o == 0) {
            float ca[S::EPL];
            const float *src = &sm.carry[cb][ol * S::EPL];
#pragma unroll
            for (int e = 0; e < S::EPL; ++e) ca[e] = src[e];
            finish(ca, 0, sm.carry_bev[cb]);
        }
        if (head_cut) finish(acc, o + 1, head_bev);
        if (T1 >= 0 && T1 <= w0 + W) break;        // uniform: the chunk ends in this window
        round_head = next_head;
        w0 += W;
        __syncthreads();                           // the next round overwrites records, states and slots
    }
}

// ---------------------------------------------------------------- fill CTA

template <int DT, int C, int OT>
__device__ __forceinline__ void fill_cta(const FwdParams &p, int fidx, FillSmem &sm) {
    int n_pts = p.n_points;
    if (p.d_counts) n_pts = min(n_pts, __ldg(p.d_counts + 0));
    if (n_pts < 0) n_pts = 0;
    const int c0 = fidx * p.fill_cells;
    const int c1 = min(c0 + p.fill_cells, p.n_cells);
    if (threadIdx.x < kFillCellsMax / 32) sm.mark[threadIdx.x] = 0u;
    int t0, t1;
    cta_lower_bound2(p.ranks_bev, n_pts, c0, c1, &t0, &t1);   // contains barriers
    for (int t = t0 + threadIdx.x; t < t1; t += kThreads) {
        const int cell = __ldg(p.ranks_bev + t) - c0;
        if (cell >= 0 && cell < p.fill_cells) atomicOr(&sm.mark[cell >> 5], 1u << (cell & 31));
    }
    __syncthreads();
    constexpr int OUT_VECS = C * (OT == kOutF16 ? 2 : 1) / 16;    // 16-byte vectors per output row
    static_assert(OUT_VECS * 16 == C * (OT == kOutF16 ? 2 : 1), "output rows are whole 16-byte vectors");
    const int total = (c1 - c0) * OUT_VECS;
    uint4 *out = reinterpret_cast<uint4 *>(p.out + static_cast<int64_t>(c0) * OUT_VECS * 16);
    const uint4 z = make_uint4(0, 0, 0, 0);
    const StoreMode mode = store_mode(p.streaming != 0);
    for (int v = threadIdx.x; v < total; v += kThreads) {
        const int cell = v / OUT_VECS;
        if (!((sm.mark[cell >> 5] >> (cell & 31)) & 1u)) {
            store_vec(out + v, z, mode);
        }
    }
}

// ---------------------------------------------------------------- kernel

template <int DT, int C, int OT, int VAR>
__global__ void __launch_bounds__(kThreads, FwdShape<DT, C, VAR>::LEAN ? BEVPOOL_FWD_LEAN_MIN_CTAS : BEVPOOL_FWD_MIN_CTAS)
    k_forward(const FwdParams p) {
    grid_dep_wait();                               // the map build may still be draining (dependent launch)
    grid_dep_allow();
    __shared__ __align__(16) FwdSmem<DT, C, VAR> sm;
    const int b = blockIdx.x;
    // compute CTAs (the long ones) first, then fill CTAs in the slots they
    // free; the fill CTAs may come after the first fill_after compute CTAs
    const int fa = p.fill_after;
    const bool compute = b < fa || b >= fa + p.n_fill;
    const int idx = b < fa ? b : (compute ? b - p.n_fill : b - fa);
    if (compute)
        compute_cta<DT, C, OT, VAR>(p, idx, sm.c);
    else
        fill_cta<DT, C, OT>(p, idx, sm.f);
}

// The compute-CTA count and fill tiling of variant VAR for the call's sizes
// (host code; the launch and bevpool_forward_plan both use it).
template <int DT, int C, int VAR>
ForwardPlan plan_variant(const ForwardArgs &a) {
    using S = FwdShape<DT, C, VAR>;
    ForwardPlan pl;
    pl.variant = VAR;
    pl.ctas_per_sm = S::LEAN ? BEVPOOL_FWD_LEAN_MIN_CTAS
                             : (a.streaming_stores ? BEVPOOL_FWD_CTAS_PER_SM_DRAM : BEVPOOL_FWD_CTAS_PER_SM_L2);
    pl.owners = S::OWNERS;
    pl.batch = S::BATCH;
    pl.round = ComputeSmem<DT, C, VAR>::ROUND;
    const int64_t sms = a.sm_count > 0 ? a.sm_count : 148;
    // About one resident wave of compute CTAs, each with at least a batch of
    // points per owner; the points per CTA are set on the device from the
    // actual count.
    const int64_t slots = sms * pl.ctas_per_sm;
    int64_t n_compute = div_up(a.n_points, static_cast<int64_t>(S::OWNERS) * S::BATCH);
    if (n_compute > slots) n_compute = slots;
#if BEVPOOL_FWD_MULTIWAVE
    if (!a.loose_capacity) {
        const int64_t per_cta = pl.round - BEVPOOL_FWD_MULTIWAVE;   // one round each
        const int64_t want = div_up(a.n_points, per_cta);
        if (want > n_compute) n_compute = slots * div_up(want, slots);   // whole waves
    }
#endif
    if (n_compute < 1) n_compute = 1;
    pl.n_compute = static_cast<int32_t>(n_compute);
    // Fill tiles.  With the output in L2: the largest power of two of cells
    // in [128, 1024] whose rows are at most 80 KB of output and which hold at
    // most 1024 points on average (the marking pass reads every point of its
    // tile), keeping at least one fill CTA per SM (measured warm against the
    // rule below: canonical 10.5 -> 10.0 us, BEVDet 9.9 -> 9.4, canonical FP8
    // 11.3 -> 10.9, 105K points 9.4 -> 8.4, 1.28M points 38.3 -> 37.4).  When
    // the output streams to DRAM the zero rows are the bottleneck of the
    // tail: about four fill CTAs per SM (each costs a dependent search before
    // its stores, so large grids take larger tiles; the rule above there:
    // DRAM batch 85.0 -> 92.9 us).
    int fill_cells;
    if (!a.streaming_stores) {
        const int64_t row_bytes = static_cast<int64_t>(C) * (a.out_e4m3 ? 1 : 2);
        fill_cells = kFillCellsMax;
        while (fill_cells > kFillCellsL2Min &&
               (fill_cells * row_bytes > kFillTileBytesL2 ||
                static_cast<int64_t>(a.n_points) * fill_cells > static_cast<int64_t>(kFillTilePoints) * a.n_cells ||
                div_up(a.n_cells, fill_cells) < sms))
            fill_cells /= 2;
    } else {
        fill_cells = kFillCellsMin;
        while (fill_cells < kFillCellsMax && a.n_cells > static_cast<int64_t>(fill_cells) * BEVPOOL_FWD_FILL_PER_SM * sms)
            fill_cells *= 2;
    }
    pl.fill_cells = fill_cells;
    pl.n_fill = static_cast<int32_t>(div_up(a.n_cells, fill_cells));
    return pl;
}

template <int DT, int C, int OT, int VAR>
cudaError_t launch_forward_v(const ForwardArgs &a) {
    const ForwardPlan pl = plan_variant<DT, C, VAR>(a);
    if (a.plan_out) {
        *a.plan_out = pl;
        return cudaSuccess;
    }
    FwdParams p;
    p.depth = a.depth;
    p.feat = a.feat;
    p.feat_block = static_cast<const unsigned char *>(a.feat_block);
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
    p.n_compute = pl.n_compute;
    p.n_compute_div = FastDiv(static_cast<uint32_t>(pl.n_compute));
    p.fill_cells = pl.fill_cells;
    p.n_fill = pl.n_fill;
    p.fill_after = pl.n_compute;
#if BEVPOOL_FWD_FILL_AFTER_WAVES
    if (a.streaming_stores) {
        const int64_t slots = static_cast<int64_t>(a.sm_count > 0 ? a.sm_count : 148) * pl.ctas_per_sm;
        p.fill_after = static_cast<int>(std::min<int64_t>(pl.n_compute, slots * BEVPOOL_FWD_FILL_AFTER_WAVES));
    }
#endif
    p.out = static_cast<unsigned char *>(a.out);
    const int grid = p.n_compute + p.n_fill;
    const cudaError_t e = launch_dependent(k_forward<DT, C, OT, VAR>, dim3(grid), dim3(kThreads), 0, a.stream, p);
    count_launch();
    return e;
}

// fp16 rows take the lean variant when the output streams to DRAM (measured:
// DRAM batch 122.9 -> 114.7 us) and when there is much work per SM even with
// the output in L2 (n_points * C >= 2^17 per SM; measured warm-L2: 572K points
// at C = 80 24.2 -> 21.8 us, 1.28M points 42.8 -> 38.9, 209K points at C = 128
// 16.5 -> 15.3; below it slower: 182K points at C = 64 10.4 -> 13.4 us).
// With the counts on the device n_points is the caller's capacity, which
// stands in for the count unless it is the whole frustum (then it says
// nothing about the frame's points).
// E4M3 rows take it when the output streams to DRAM (wide C = 256: 21.1 -> 20.1
// us warm); with the output in L2 it was mixed (572K points 20.7 -> 18.7,
// 1.28M points 39.4 -> 41.0, C = 128 13.7 -> 14.0).
template <int DT, int C, int OT>
cudaError_t launch_forward_t(const ForwardArgs &a) {
    if constexpr (DT == kDtypeE4M3) {
        if (a.streaming_stores) return launch_forward_v<DT, C, OT, kVarLean>(a);
    }
    if constexpr (DT == kDtypeF16) {
        const int64_t sms = a.sm_count > 0 ? a.sm_count : 148;
        const bool much_work =
            !a.loose_capacity && a.n_points * static_cast<int64_t>(C) >= BEVPOOL_FWD_LEAN_WORK_PER_SM * sms;
        // short intervals (fewer than 8 points on average, host counts or a
        // capacity close to them) take fewer points in flight per owner
        const bool short_intervals =
            !a.loose_capacity && a.n_intervals > 0 && a.n_points < 8 * static_cast<int64_t>(a.n_intervals);
        // lean: 4 points in flight with short intervals (DRAM batch, 3.0 points
        // per interval, 94.2 -> 92.5 us; C = 128 at 3.6 points 20.7 -> 20.5 us),
        // else 6 (8.7-point intervals 25.3 -> 26.6 us at 4)
        if (a.streaming_stores || much_work)
            return short_intervals ? launch_forward_v<DT, C, OT, kVarLeanShort>(a)
                                   : launch_forward_v<DT, C, OT, kVarLean>(a);
        // 6 points in flight at 80 registers (canonical 11.0 -> 10.4 us warm;
        // 19-point intervals 10.0 -> 10.4 us)
        if (short_intervals) return launch_forward_v<DT, C, OT, kVarShort>(a);
    }
    return launch_forward_v<DT, C, OT, kVarDefault>(a);
}

}  // namespace bevpool
