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

}  // namespace
}  // namespace bevpool

using namespace bevpool;

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
