/*
 * bevpool_oracle.c -- plain, slow, single-threaded FP64 oracle for BEV pooling.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library,
 * its Python binding) may include, link or call this file.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline / reference arm use it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (source: "Accelerating BEV Pooling on NVIDIA GPUs for
 * Physical AI Applications", NVIDIA technical blog, Vietnamese mirror on
 * ntcai.vn and Chinese mirror on developer.nvidia.cn):
 *
 *   - section "Eliminate redundant scatter traffic": the BEV scatter-reduce
 *         out[ranks_bev[t], c] += depth[ranks_depth[t]] * feat[ranks_feat[t], c]
 *     summed over every scatter point t;
 *   - same section: the five-array INT32 scatter map (ranks_depth,
 *     ranks_feat, ranks_bev, interval_starts, interval_lengths) with
 *     precomputed explicit indices;
 *   - section "Implement interval-owned scatter-reduce": an interval is the
 *     run of scatter points that share one BEV cell; its owner writes the
 *     cell once.
 *
 * Readings where the pages are silent:
 *   - frustum point index p = ((nc*D + d)*H + h)*W + w; depth is laid out
 *     [NC, D, H, W] so ranks_depth = p; feat is NHWC [NC, H, W, C] so
 *     ranks_feat = (nc*H + h)*W + w; out is [n_cells, C] row-major;
 *   - a frustum point whose cell id is -1 is dropped; any other negative id
 *     or an id >= n_cells is an error;
 *   - points inside an interval are ordered by ascending p (a stable sort of
 *     frustum order by cell), intervals by ascending cell;
 *   - cells no point reaches are 0 in the output;
 *   - FP8 inputs are OCP E4M3 codes with one scale per tensor; the value the
 *     method sees is code_value * scale;
 *   - the FP8 output (section "Eliminate redundant scatter traffic", Figure
 *     4: the FP8 path halves output bytes too; section "Map the algorithm to
 *     hardware": the NVFP4 experiment keeps depth and output in FP8) is the
 *     E4M3 code nearest to value / out_scale, out_scale being one per-tensor
 *     scale the caller chooses; ties to even, saturated at +-448;
 *   - NVFP4 features (section "Map the algorithm to hardware", the NVFP4
 *     experiment: E2M1 elements with an E4M3 scale per 16 elements, depth
 *     kept in FP8): element 2i of a row in the low nibble of byte i, the
 *     block scales in their own [rows, C/16] array, one per-tensor factor.
 *
 * The forward oracle does NOT go through the scatter map: it walks the
 * frustum points in their original order, so it also checks the map.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_RANGE 2
#define ORACLE_ERR_NOMEM 3

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Exponent 0 encodes zero / subnormals (fraction * 2^-24); exponent 31
 * encodes infinity (fraction 0) or NaN. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits
 * (bias 7), 3 mantissa bits, no infinities; S.1111.111 is NaN.  Exponent 0
 * encodes zero / subnormals (mantissa/8 * 2^-6). */
double oracle_e4m3_to_double(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int expo = (b >> 3) & 0xf;
    int mant = b & 0x7;
    double v;
    if (expo == 15 && mant == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)mant, -9);
    else
        v = ldexp((double)(8 + mant), expo - 10);
    return sign ? -v : v;
}

/* OCP 4-bit floating point E2M1 (the element type of NVFP4): 1 sign bit,
 * 2 exponent bits (bias 1), 1 mantissa bit, no infinities or NaN.  Exponent
 * 0 encodes zero / the subnormal 0.5 (mantissa * 0.5). */
double oracle_e2m1_to_double(uint8_t nibble)
{
    int sign = (nibble >> 3) & 1;
    int expo = (nibble >> 1) & 3;
    int mant = nibble & 1;
    double v = expo == 0 ? 0.5 * mant : ldexp(1.0 + 0.5 * mant, expo - 1);
    return sign ? -v : v;
}

/* Bulk helpers so the Python side can decode whole tensors. */
void oracle_half_array_to_double(const uint16_t *src, int64_t n, double *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_half_to_double(src[i]);
}

void oracle_e4m3_array_to_double(const uint8_t *src, int64_t n, double *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_e4m3_to_double(src[i]);
}

void oracle_e2m1_array_to_double(const uint8_t *src, int64_t n, double *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_e2m1_to_double(src[i] & 0xf);
}

/* Nearest OCP E4M3 code to x: round half to even, magnitudes above the
 * largest finite value (448) saturate to it, the sign is kept (a negative
 * value that rounds to zero gives -0).  Written from the format itself: the
 * representable values between 2^e and 2^(e+1) are spaced 2^(e-3) apart for
 * e >= -6, and the subnormals 2^-9 apart below 2^-6. */
uint8_t oracle_e4m3_from_double(double x)
{
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    double step;
    if (a < ldexp(1.0, -6)) {
        step = ldexp(1.0, -9);
    } else {
        int k;
        frexp(a, &k);                    /* a = f * 2^k, f in [0.5, 1): 2^(k-1) <= a < 2^k */
        step = ldexp(1.0, k - 1 - 3);
    }
    double v = rint(a / step) * step;    /* default rounding mode: half to even */
    if (v > 448.0)
        v = 448.0;
    if (v == 0.0)
        return sign;
    int k;
    frexp(v, &k);
    int e = k - 1;                       /* 2^e <= v < 2^(e+1) */
    uint8_t code;
    if (e < -6)
        code = (uint8_t)(v / ldexp(1.0, -9));                 /* subnormal: mantissa only */
    else
        code = (uint8_t)(((e + 7) << 3) | ((int)(v / ldexp(1.0, e - 3)) - 8));
    return sign | code;
}

void oracle_double_array_to_e4m3(const double *src, int64_t n, uint8_t *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_e4m3_from_double(src[i]);
}

typedef struct {
    int32_t cell;
    int32_t p;
} kept_point;

static int compare_cell_then_p(const void *a, const void *b)
{
    const kept_point *x = (const kept_point *)a;
    const kept_point *y = (const kept_point *)b;
    if (x->cell != y->cell)
        return x->cell < y->cell ? -1 : 1;
    if (x->p != y->p)
        return x->p < y->p ? -1 : 1;
    return 0;
}

/*
 * Scatter-map builder.  Output arrays must hold NC*D*H*W entries each.
 * counts[0] = number of scatter points n, counts[1] = number of intervals.
 *
 *   1. walk p = 0 .. NC*D*H*W-1 and keep (cell_ids[p], p) when cell_ids[p] != -1;
 *   2. sort the kept pairs by (cell, p) with the C library sort;
 *   3. ranks_bev = cell, ranks_depth = p,
 *      ranks_feat = nc*H*W + h*W + w  where nc = p / (D*H*W) and
 *      h*W + w = p mod (H*W);
 *   4. intervals are the maximal runs of equal ranks_bev, in order.
 */
int oracle_build_map(const int32_t *cell_ids, int32_t NC, int32_t D, int32_t H, int32_t W,
                     int32_t n_cells, int32_t *ranks_depth, int32_t *ranks_feat,
                     int32_t *ranks_bev, int32_t *interval_starts, int32_t *interval_lengths,
                     int32_t *counts)
{
    if (NC <= 0 || D <= 0 || H <= 0 || W <= 0 || n_cells <= 0)
        return ORACLE_ERR_ARG;
    int64_t n_frustum = (int64_t)NC * D * H * W;
    if (n_frustum > INT32_MAX)
        return ORACLE_ERR_ARG;

    kept_point *kept = (kept_point *)malloc((size_t)n_frustum * sizeof(kept_point));
    if (!kept)
        return ORACLE_ERR_NOMEM;
    int64_t n = 0;
    for (int64_t p = 0; p < n_frustum; ++p) {
        int32_t cell = cell_ids[p];
        if (cell == -1)
            continue;
        if (cell < 0 || cell >= n_cells) {
            free(kept);
            return ORACLE_ERR_RANGE;
        }
        kept[n].cell = cell;
        kept[n].p = (int32_t)p;
        ++n;
    }

    qsort(kept, (size_t)n, sizeof(kept_point), compare_cell_then_p);

    int64_t per_camera = (int64_t)D * H * W;
    int64_t per_image = (int64_t)H * W;
    for (int64_t t = 0; t < n; ++t) {
        int64_t p = kept[t].p;
        int64_t nc = p / per_camera;
        int64_t hw = p % per_image;
        ranks_bev[t] = kept[t].cell;
        ranks_depth[t] = (int32_t)p;
        ranks_feat[t] = (int32_t)(nc * per_image + hw);
    }

    int64_t n_intervals = 0;
    for (int64_t t = 0; t < n; ++t) {
        if (t == 0 || ranks_bev[t] != ranks_bev[t - 1]) {
            interval_starts[n_intervals] = (int32_t)t;
            interval_lengths[n_intervals] = 1;
            ++n_intervals;
        } else {
            interval_lengths[n_intervals - 1] += 1;
        }
    }

    counts[0] = (int32_t)n;
    counts[1] = (int32_t)n_intervals;
    free(kept);
    return ORACLE_OK;
}

/*
 * Forward oracle, FP64, one point at a time in frustum order:
 *     out[cell(p), c] += depth_value(p) * feat_value(row(p), c)
 * with row(p) = (nc*H + h)*W + w.  out has n_cells*C doubles and is fully
 * overwritten (cells no point reaches stay 0).
 *
 * dtype 0: depth and feat are binary16 codes, value = decoded half.
 * dtype 1: depth and feat are E4M3 codes, value = decoded code * scale
 *          (depth_scale for depth, feat_scale for feat).
 */
int oracle_forward(int32_t dtype, const int32_t *cell_ids, int32_t NC, int32_t D, int32_t H,
                   int32_t W, int32_t n_cells, int32_t C, const void *depth, const void *feat,
                   double depth_scale, double feat_scale, double *out)
{
    if (NC <= 0 || D <= 0 || H <= 0 || W <= 0 || n_cells <= 0 || C <= 0)
        return ORACLE_ERR_ARG;
    if (dtype != 0 && dtype != 1)
        return ORACLE_ERR_ARG;
    int64_t n_frustum = (int64_t)NC * D * H * W;
    memset(out, 0, (size_t)n_cells * (size_t)C * sizeof(double));

    const uint16_t *depth16 = (const uint16_t *)depth;
    const uint16_t *feat16 = (const uint16_t *)feat;
    const uint8_t *depth8 = (const uint8_t *)depth;
    const uint8_t *feat8 = (const uint8_t *)feat;

    for (int64_t p = 0; p < n_frustum; ++p) {
        int32_t cell = cell_ids[p];
        if (cell == -1)
            continue;
        if (cell < 0 || cell >= n_cells)
            return ORACLE_ERR_RANGE;
        int64_t w = p % W;
        int64_t h = (p / W) % H;
        int64_t nc = p / ((int64_t)D * H * W);
        int64_t row = (nc * H + h) * W + w;

        double d;
        if (dtype == 0)
            d = oracle_half_to_double(depth16[p]);
        else
            d = oracle_e4m3_to_double(depth8[p]) * depth_scale;

        double *dst = out + (int64_t)cell * C;
        for (int32_t c = 0; c < C; ++c) {
            double f;
            if (dtype == 0)
                f = oracle_half_to_double(feat16[row * C + c]);
            else
                f = oracle_e4m3_to_double(feat8[row * C + c]) * feat_scale;
            dst[c] += d * f;
        }
    }
    return ORACLE_OK;
}

/*
 * The forward with NVFP4 features (section "Map the algorithm to hardware",
 * the NVFP4 experiment): feat element c of row r is the E2M1 value in nibble
 * c of the packed row (element 2i in the low nibble of byte i), times the
 * E4M3 block scale feat_block[r * C/16 + c/16], times the per-tensor
 * feat_scale; depth is E4M3 times depth_scale.  Same point loop as
 * oracle_forward, in double.
 */
int oracle_forward_nvfp4(const int32_t *cell_ids, int32_t NC, int32_t D, int32_t H, int32_t W,
                         int32_t n_cells, int32_t C, const uint8_t *depth8, const uint8_t *feat4,
                         const uint8_t *feat_block, double depth_scale, double feat_scale, double *out)
{
    if (NC <= 0 || D <= 0 || H <= 0 || W <= 0 || n_cells <= 0 || C <= 0 || C % 16 != 0)
        return ORACLE_ERR_ARG;
    int64_t n_frustum = (int64_t)NC * D * H * W;
    memset(out, 0, (size_t)n_cells * (size_t)C * sizeof(double));
    for (int64_t p = 0; p < n_frustum; ++p) {
        int32_t cell = cell_ids[p];
        if (cell == -1)
            continue;
        if (cell < 0 || cell >= n_cells)
            return ORACLE_ERR_RANGE;
        int64_t w = p % W;
        int64_t h = (p / W) % H;
        int64_t nc = p / ((int64_t)D * H * W);
        int64_t row = (nc * H + h) * W + w;
        double d = oracle_e4m3_to_double(depth8[p]) * depth_scale;
        double *dst = out + (int64_t)cell * C;
        for (int32_t c = 0; c < C; ++c) {
            uint8_t byte = feat4[row * (C / 2) + c / 2];
            uint8_t nib = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xf);
            double f = oracle_e2m1_to_double(nib) * oracle_e4m3_to_double(feat_block[row * (C / 16) + c / 16]) *
                       feat_scale;
            dst[c] += d * f;
        }
    }
    return ORACLE_OK;
}
