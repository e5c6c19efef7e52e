// encode.cu -- PQ encode-and-append: for every new token, kv head and K-or-V,
// the index of the nearest codeword in each subspace (AQPIM blog §3.1 step 3,
// §5.2 item 2), written as uint8 into the token's page slot (PAM article
// §2.2.2 paged cache).
//
// Decision arithmetic: d_k = sum_{j=0}^{Dsub-1} (x_j - c_kj)^2 in fp32 with
// separately rounded subtract, multiply and add in increasing j (no fused
// multiply-add), argmin with ties to the lowest k.  This is the plain
// definition evaluated in fp32, so the code is a deterministic function of the
// inputs on any device.
//
// Two kernels:
//   encode_cw_kernel   one CTA per (token, kv head), one thread per codeword:
//                      for a decode step's handful of tokens; each codebook row
//                      is read once, all 2*M argmins reduce in parallel.
//   encode_tok_kernel  one CTA per (128-token tile, kv head, K-or-V, subspace),
//                      one thread per token, the subspace codebook staged in
//                      shared memory and read as broadcasts: for prefill.
#include "common.cuh"
#include "internal.h"

namespace aq {

namespace {

__device__ __forceinline__ float sqdist_step(float acc, float x, float c) {
    const float e = __fsub_rn(x, c);
    return __fadd_rn(acc, __fmul_rn(e, e));
}

// (distance, index) packed so that unsigned order = (distance, index) order for
// distances >= 0 (and NaN after +inf).
__device__ __forceinline__ unsigned long long pack_key(float d, int k) {
    return (static_cast<unsigned long long>(__float_as_uint(d)) << 32) | static_cast<unsigned>(k);
}

__device__ __forceinline__ bool slot_ok(const EncodeParams &p, int t, int64_t &slot, int &set) {
    slot = p.slot_mapping[t];
    set = p.token_set[t];
    if (slot < 0) return false;                              // padding token
    bool ok = true;
    if (slot / kPage >= p.num_pages) {
        flag_status(p.status, AQ_DEV_BAD_PAGE);
        ok = false;
    }
    if (set < 0 || static_cast<int64_t>(set) >= p.num_sets) {
        flag_status(p.status, AQ_DEV_BAD_SET);
        ok = false;
    }
    return ok;
}

template <int M>
__global__ void __launch_bounds__(256) encode_cw_kernel(const __grid_constant__ EncodeParams p) {
    constexpr int D = kHeadDim, K = kCodewords, DSUB = D / M, NSEL = 2 * M;
    __shared__ float xs[2 * D];
    __shared__ unsigned long long wkey[8][NSEL];
    const int t = blockIdx.x, kvh = blockIdx.y, tid = threadIdx.x;
    int64_t slot;
    int set;
    const bool ok = slot_ok(p, t, slot, set);               // uniform over the CTA
    if (!ok) return;
    const __half *x = reinterpret_cast<const __half *>(p.kv) +
                      (static_cast<size_t>(t) * p.num_kv_heads + kvh) * 2 * D;
    xs[tid] = __half2float(x[tid]);                          // 256 == 2 * D
    __syncthreads();
    const __half *cb = reinterpret_cast<const __half *>(p.codebooks) +
                       ((static_cast<size_t>(set) * p.num_kv_heads + kvh) * 2) * M * K * DSUB;
    // thread tid = codeword k; its 2*M rows
    unsigned long long key[NSEL];
#pragma unroll
    for (int sel = 0; sel < NSEL; ++sel) {
        const int w = sel / M, m = sel % M;
        const uint4 *row = reinterpret_cast<const uint4 *>(
            cb + ((static_cast<size_t>(w) * M + m) * K + tid) * DSUB);
        const float *xv = xs + w * D + m * DSUB;
        float d = 0.f;
#pragma unroll
        for (int c = 0; c < DSUB / 8; ++c) {
            const uint4 u = __ldg(row + c);
            const float2 f0 = h2_to_f2(u.x), f1 = h2_to_f2(u.y), f2 = h2_to_f2(u.z), f3 = h2_to_f2(u.w);
            d = sqdist_step(d, xv[c * 8 + 0], f0.x);
            d = sqdist_step(d, xv[c * 8 + 1], f0.y);
            d = sqdist_step(d, xv[c * 8 + 2], f1.x);
            d = sqdist_step(d, xv[c * 8 + 3], f1.y);
            d = sqdist_step(d, xv[c * 8 + 4], f2.x);
            d = sqdist_step(d, xv[c * 8 + 5], f2.y);
            d = sqdist_step(d, xv[c * 8 + 6], f3.x);
            d = sqdist_step(d, xv[c * 8 + 7], f3.y);
        }
        key[sel] = pack_key(d, tid);
    }
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int sel = 0; sel < NSEL; ++sel) {
        unsigned long long k = key[sel];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, k, off);
            k = o < k ? o : k;
        }
        if (lane == 0) wkey[warp][sel] = k;
    }
    __syncthreads();
    if (tid < NSEL) {
        unsigned long long k = wkey[0][tid];
#pragma unroll
        for (int w = 1; w < 8; ++w) k = wkey[w][tid] < k ? wkey[w][tid] : k;
        const int w_ = tid / M, m = tid % M;
        const int64_t page = slot / kPage, s = slot % kPage;
        p.code_pages[((static_cast<size_t>(page) * p.num_kv_heads + kvh) * kPage + s) * 2 * M + w_ * M + m] =
            static_cast<uint8_t>(k & 0xffu);
    }
}

constexpr int kTile = 128;

template <int M>
__global__ void __launch_bounds__(kTile) encode_tok_kernel(const __grid_constant__ EncodeParams p) {
    constexpr int D = kHeadDim, K = kCodewords, DSUB = D / M;
    __shared__ __align__(16) float cbs[K * DSUB];             // 32 KiB (M=4) / 16 KiB (M=8)
    __shared__ int tile_set;
    const int kvh = blockIdx.y, sel = blockIdx.z, w = sel / M, m = sel % M;
    const int t0 = blockIdx.x * kTile, tid = threadIdx.x;
    const int t = t0 + tid;
    if (tid == 0) tile_set = p.token_set[t0];
    __syncthreads();
    const int set0 = tile_set;
    const bool set0_ok = set0 >= 0 && static_cast<int64_t>(set0) < p.num_sets;
    if (set0_ok) {
        const __half *cb = reinterpret_cast<const __half *>(p.codebooks) +
                           (((static_cast<size_t>(set0) * p.num_kv_heads + kvh) * 2 + w) * M + m) * K * DSUB;
        for (int i = tid; i < K * DSUB / 2; i += kTile) {
            const float2 f = h2_to_f2(reinterpret_cast<const uint32_t *>(cb)[i]);
            cbs[2 * i] = f.x;
            cbs[2 * i + 1] = f.y;
        }
    }
    __syncthreads();
    if (t >= p.num_tokens) return;
    int64_t slot;
    int set;
    if (!slot_ok(p, t, slot, set)) return;
    float x[DSUB];
    const __half *xp = reinterpret_cast<const __half *>(p.kv) +
                       ((static_cast<size_t>(t) * p.num_kv_heads + kvh) * 2 + w) * D + m * DSUB;
#pragma unroll
    for (int j = 0; j < DSUB; j += 2) {
        const float2 f = h2_to_f2(*reinterpret_cast<const uint32_t *>(xp + j));
        x[j] = f.x;
        x[j + 1] = f.y;
    }
    float best = INFINITY;
    int bk = 0;
    if (set == set0) {
#pragma unroll 2
        for (int k = 0; k < K; ++k) {
            const float4 *c4 = reinterpret_cast<const float4 *>(cbs + k * DSUB);
            float d = 0.f;
#pragma unroll
            for (int j = 0; j < DSUB; j += 4) {
                const float4 c = c4[j / 4];
                d = sqdist_step(d, x[j], c.x);
                d = sqdist_step(d, x[j + 1], c.y);
                d = sqdist_step(d, x[j + 2], c.z);
                d = sqdist_step(d, x[j + 3], c.w);
            }
            if (d < best) { best = d; bk = k; }
        }
    } else {                                                  // token of another set
        const __half *cb = reinterpret_cast<const __half *>(p.codebooks) +
                           (((static_cast<size_t>(set) * p.num_kv_heads + kvh) * 2 + w) * M + m) * K * DSUB;
        for (int k = 0; k < K; ++k) {
            float d = 0.f;
            for (int j = 0; j < DSUB; ++j) d = sqdist_step(d, x[j], __half2float(cb[k * DSUB + j]));
            if (d < best) { best = d; bk = k; }
        }
    }
    const int64_t page = slot / kPage, s = slot % kPage;
    p.code_pages[((static_cast<size_t>(page) * p.num_kv_heads + kvh) * kPage + s) * 2 * M + w * M + m] =
        static_cast<uint8_t>(bk);
}

}  // namespace

cudaError_t launch_encode(const EncodeParams &p, int M, cudaStream_t s) {
    if (p.num_tokens == 0) return cudaSuccess;
    const bool small = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads <= 8192;
    if (small) {
        dim3 grid(static_cast<unsigned>(p.num_tokens), static_cast<unsigned>(p.num_kv_heads));
        if (M == 4) encode_cw_kernel<4><<<grid, 256, 0, s>>>(p);
        else encode_cw_kernel<8><<<grid, 256, 0, s>>>(p);
    } else {
        dim3 grid(static_cast<unsigned>((p.num_tokens + kTile - 1) / kTile),
                  static_cast<unsigned>(p.num_kv_heads), static_cast<unsigned>(2 * M));
        if (M == 4) encode_tok_kernel<4><<<grid, kTile, 0, s>>>(p);
        else encode_tok_kernel<8><<<grid, kTile, 0, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace aq
