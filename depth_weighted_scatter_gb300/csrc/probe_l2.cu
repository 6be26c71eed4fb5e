// probe_l2.cu -- L2 streaming probe: how fast the SMs can read, write or copy
// a buffer that stays resident in L2.  This gives the bandwidth denominator
// for the forward's roofline when its working set is L2-resident.  The forward
// itself does not use it.
//
// Read: every thread reads 16-byte vectors with ld.global.cg (cached in L2
// only, so the SM's L1 serves none of them), four in flight per thread, over
// the whole buffer, `passes` times.  The 32-bit words it read are summed
// (mod 2^32) into *d_sink, so the caller can check that every byte was read
// exactly `passes` times.
//
// Write: every thread writes 16-byte vectors, four per iteration, over the
// whole buffer, `passes` times.  Word k of pass p holds k ^ (p * 0x9E3779B9).
//
// Copy: the second half of the buffer receives the first half, word by word
// XORed with p * 0x9E3779B9 in pass p (so every pass writes new values), with
// the loads of the read probe and the stores of the write probe.
//
// Gather (bevpool_probe_gather): the feature-row gather of the forward alone,
// in the forward's lane layout (owners of row_bytes / 16 lanes, one 16-byte
// vector a lane, eight rows in flight, each owner a contiguous equal share of
// the points), over a caller's row list (a map's ranks_feat), with nothing
// else: no depth, no accumulation into rows, no stores.  The words it read
// are summed (mod 2^32) into *d_sink, or, with no sink (the timing mode),
// only kept live so no load is dropped.  It bounds what the forward's walk
// can reach on the same rows.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "bevpool_internal.cuh"

namespace bevpool {
namespace {

constexpr uint32_t kPassSalt = 0x9E3779B9u;   // a fixed odd constant that differs per pass
constexpr int kProbeCtasPerSm = 8;            // 8 x 256 threads: a full SM

__device__ __forceinline__ uint4 ld_cg(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_wb(uint4 *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t word_sum(uint4 v) { return v.x + v.y + v.z + v.w; }

__global__ void __launch_bounds__(kThreads) k_probe_read(const uint4 *buf, int64_t n_vec, int passes, uint32_t *sink) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    uint32_t s = 0;
    for (int pass = 0; pass < passes; ++pass) {
        int64_t i = t0;
        for (; i + 3 * stride < n_vec; i += 4 * stride) {
            const uint4 a = ld_cg(buf + i), b = ld_cg(buf + i + stride);
            const uint4 c = ld_cg(buf + i + 2 * stride), d = ld_cg(buf + i + 3 * stride);
            s += word_sum(a) + word_sum(b) + word_sum(c) + word_sum(d);
        }
        for (; i < n_vec; i += stride) s += word_sum(ld_cg(buf + i));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(sink, s);
}

__device__ __forceinline__ uint4 pattern(int64_t i, uint32_t salt) {
    const uint32_t k = static_cast<uint32_t>(i) * 4u;
    return make_uint4(k ^ salt, (k + 1u) ^ salt, (k + 2u) ^ salt, (k + 3u) ^ salt);
}

__global__ void __launch_bounds__(kThreads) k_probe_write(uint4 *buf, int64_t n_vec, int passes) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (int pass = 0; pass < passes; ++pass) {
        const uint32_t salt = static_cast<uint32_t>(pass) * kPassSalt;
        int64_t i = t0;
        for (; i + 3 * stride < n_vec; i += 4 * stride) {
            st_wb(buf + i, pattern(i, salt));
            st_wb(buf + i + stride, pattern(i + stride, salt));
            st_wb(buf + i + 2 * stride, pattern(i + 2 * stride, salt));
            st_wb(buf + i + 3 * stride, pattern(i + 3 * stride, salt));
        }
        for (; i < n_vec; i += stride) st_wb(buf + i, pattern(i, salt));
    }
}

__device__ __forceinline__ uint4 salted(uint4 v, uint32_t salt) {
    return make_uint4(v.x ^ salt, v.y ^ salt, v.z ^ salt, v.w ^ salt);
}

__global__ void __launch_bounds__(kThreads) k_probe_copy(const uint4 *src, uint4 *dst, int64_t n_vec, int passes) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (int pass = 0; pass < passes; ++pass) {
        const uint32_t salt = static_cast<uint32_t>(pass) * kPassSalt;
        int64_t i = t0;
        for (; i + 3 * stride < n_vec; i += 4 * stride) {
            const uint4 a = ld_cg(src + i), b = ld_cg(src + i + stride);
            const uint4 c = ld_cg(src + i + 2 * stride), d = ld_cg(src + i + 3 * stride);
            st_wb(dst + i, salted(a, salt));
            st_wb(dst + i + stride, salted(b, salt));
            st_wb(dst + i + 2 * stride, salted(c, salt));
            st_wb(dst + i + 3 * stride, salted(d, salt));
        }
        for (; i < n_vec; i += stride) st_wb(dst + i, salted(ld_cg(src + i), salt));
    }
}

constexpr int kGatherBatch = 8;               // rows in flight per owner

__global__ void __launch_bounds__(kThreads) k_probe_gather(const unsigned char *feat, int32_t n_rows, int row_bytes,
                                                           const int32_t *rows, int32_t n_points, uint32_t *sink) {
    const int lpo = row_bytes / 16;               // lanes per owner (1..32)
    const int opw = 32 / lpo;                     // owners per warp
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int og = lane / lpo, ol = lane - og * lpo;
    uint32_t s = 0;
    if (og < opw) {
        const int64_t owners = static_cast<int64_t>(gridDim.x) * kWarps * opw;
        const int64_t o = (static_cast<int64_t>(blockIdx.x) * kWarps + warp) * opw + og;
        const int64_t share = (n_points + owners - 1) / owners;
        const int64_t beg = min(static_cast<int64_t>(n_points), o * share);
        const int64_t end = min(static_cast<int64_t>(n_points), beg + share);
        const unsigned char *base = feat + ol * 16;
        int64_t t = beg;
        for (; t + kGatherBatch <= end; t += kGatherBatch) {
            int r[kGatherBatch];
#pragma unroll
            for (int k = 0; k < kGatherBatch; ++k) r[k] = __ldg(rows + t + k);
            uint4 v[kGatherBatch];
#pragma unroll
            for (int k = 0; k < kGatherBatch; ++k) {
                const bool ok = r[k] >= 0 && r[k] < n_rows;
                v[k] = ok ? __ldg(reinterpret_cast<const uint4 *>(base + static_cast<int64_t>(r[k]) * row_bytes))
                          : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int k = 0; k < kGatherBatch; ++k) s += word_sum(v[k]);
        }
        for (; t < end; ++t) {
            const int r = __ldg(rows + t);
            if (r >= 0 && r < n_rows)
                s += word_sum(__ldg(reinterpret_cast<const uint4 *>(base + static_cast<int64_t>(r) * row_bytes)));
        }
    }
    if (!sink) {                                  // timing: keep the sum live, no atomics, no barrier
        asm volatile("" ::"r"(s));
        return;
    }
    // one atomic per CTA (thousands of warps adding to one word would queue
    // at its L2 slice)
    __shared__ uint32_t part[kWarps];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) part[warp] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t += part[w];
        atomicAdd(sink, t);
    }
}

}  // namespace
}  // namespace bevpool

using namespace bevpool;

extern "C" BEVPOOL_API bevpool_status bevpool_probe_gather(const void *feat, int32_t n_rows, int32_t row_bytes,
                                                           const int32_t *rows, int32_t n_points,
                                                           int32_t ctas_per_sm, uint32_t *d_sink, void *stream) {
    if (!feat || reinterpret_cast<uintptr_t>(feat) % 16 != 0 || n_rows < 1 || row_bytes < 16 || row_bytes > 512 ||
        row_bytes % 16 != 0 || n_points < 0 || (n_points > 0 && !rows) ||
        reinterpret_cast<uintptr_t>(rows) % 4 != 0 || ctas_per_sm < 1 || ctas_per_sm > 8)
        return BEVPOOL_ERR_INVALID_ARG;
    DeviceInfo info;
    if (!device_info(&info)) return BEVPOOL_ERR_CUDA;
    const unsigned grid = static_cast<unsigned>(info.sm_count * ctas_per_sm);
    k_probe_gather<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const unsigned char *>(feat), n_rows, row_bytes, rows, n_points, d_sink);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? BEVPOOL_OK : BEVPOOL_ERR_CUDA;
}

extern "C" BEVPOOL_API bevpool_status bevpool_probe_l2(int32_t mode, void *buf, size_t bytes, int32_t passes,
                                                       uint32_t *d_sink, void *stream) {
    const size_t unit = mode == 2 ? 32 : 16;       // copy: two halves of whole 16-byte vectors
    if (mode < 0 || mode > 2 || !buf || bytes == 0 || bytes % unit != 0 ||
        reinterpret_cast<uintptr_t>(buf) % 16 != 0 || passes < 1 || (mode == 0 && !d_sink))
        return BEVPOOL_ERR_INVALID_ARG;
    if (bytes > (static_cast<size_t>(1) << 32)) return BEVPOOL_ERR_INVALID_ARG;   // word indices are 32-bit
    DeviceInfo info;
    if (!device_info(&info)) return BEVPOOL_ERR_CUDA;
    const int64_t n_vec = static_cast<int64_t>(bytes / 16) / (mode == 2 ? 2 : 1);
    const unsigned grid = static_cast<unsigned>(
        std::min<int64_t>(static_cast<int64_t>(info.sm_count) * kProbeCtasPerSm, div_up(n_vec, kThreads)));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint4 *v = static_cast<uint4 *>(buf);
    if (mode == 0)
        k_probe_read<<<grid, kThreads, 0, st>>>(v, n_vec, passes, d_sink);
    else if (mode == 1)
        k_probe_write<<<grid, kThreads, 0, st>>>(v, n_vec, passes);
    else
        k_probe_copy<<<grid, kThreads, 0, st>>>(v, v + n_vec, n_vec, passes);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? BEVPOOL_OK : BEVPOOL_ERR_CUDA;
}
