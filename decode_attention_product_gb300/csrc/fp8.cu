// fp8.cu -- FP8 E4M3 codebook storage (AQPIM blog §4.2: codebooks kept in a
// low-precision float such as FP8).  Conversion of fp16 codebooks to E4M3
// codes (nearest, ties to even, magnitudes beyond 448 and infinities
// saturated to 448, NaN stays NaN) and the exact widening back to fp16 (every
// E4M3 value is an fp16 value, so encoding against the widened codebook
// decides exactly as against the E4M3 one).
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace aq {

namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;        // one 16-byte fp16 load / 8-byte code store

__device__ __forceinline__ uint32_t e4m3x2_from_h2(uint32_t w) {
    __half2_raw r;
    r.x = static_cast<unsigned short>(w & 0xffffu);
    r.y = static_cast<unsigned short>(w >> 16);
    return static_cast<uint32_t>(__nv_cvt_halfraw2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint32_t h2_from_e4m3x2(uint32_t b) {
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(b & 0xffffu), __NV_E4M3);
    return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}

__global__ void __launch_bounds__(kThreads) to_e4m3_kernel(int64_t n, const __half *src, uint8_t *dst) {
    const int64_t i = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * kPerThread;
    if (i >= n) return;
    if (i + kPerThread <= n) {
        const uint4 u = *reinterpret_cast<const uint4 *>(src + i);
        const uint32_t lo = e4m3x2_from_h2(u.x) | (e4m3x2_from_h2(u.y) << 16);
        const uint32_t hi = e4m3x2_from_h2(u.z) | (e4m3x2_from_h2(u.w) << 16);
        *reinterpret_cast<uint2 *>(dst + i) = make_uint2(lo, hi);
    } else {
        for (int64_t j = i; j < n; ++j) {
            __half_raw r;
            r.x = reinterpret_cast<const unsigned short *>(src)[j];
            dst[j] = static_cast<uint8_t>(__nv_cvt_halfraw_to_fp8(r, __NV_SATFINITE, __NV_E4M3));
        }
    }
}

__global__ void __launch_bounds__(kThreads) from_e4m3_kernel(int64_t n, const uint8_t *src, __half *dst) {
    const int64_t i = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * kPerThread;
    if (i >= n) return;
    if (i + kPerThread <= n) {
        const uint2 b = *reinterpret_cast<const uint2 *>(src + i);
        *reinterpret_cast<uint4 *>(dst + i) = make_uint4(h2_from_e4m3x2(b.x), h2_from_e4m3x2(b.x >> 16),
                                                         h2_from_e4m3x2(b.y), h2_from_e4m3x2(b.y >> 16));
    } else {
        for (int64_t j = i; j < n; ++j) {
            const __half_raw r = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(src[j]), __NV_E4M3);
            reinterpret_cast<unsigned short *>(dst)[j] = r.x;
        }
    }
}

unsigned blocks_for(int64_t n) {
    return static_cast<unsigned>((n + static_cast<int64_t>(kThreads) * kPerThread - 1) /
                                 (static_cast<int64_t>(kThreads) * kPerThread));
}

}  // namespace

cudaError_t launch_to_e4m3(int64_t n, const void *src_f16, uint8_t *dst, cudaStream_t s) {
    to_e4m3_kernel<<<blocks_for(n), kThreads, 0, s>>>(n, reinterpret_cast<const __half *>(src_f16), dst);
    return cudaGetLastError();
}

cudaError_t launch_from_e4m3(int64_t n, const uint8_t *src, void *dst_f16, cudaStream_t s) {
    from_e4m3_kernel<<<blocks_for(n), kThreads, 0, s>>>(n, src, reinterpret_cast<__half *>(dst_f16));
    return cudaGetLastError();
}

}  // namespace aq
