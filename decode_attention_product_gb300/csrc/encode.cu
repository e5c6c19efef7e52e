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
//   encode_mma_kernel  one CTA per (128-token tile, kv head, K-or-V): for
//                      prefill.  Tensor cores (tcgen05, accumulator in TMEM)
//                      give every token's dot products with all codewords; a
//                      bound on their rounding leaves a few candidates per
//                      token, which the exact rule then decides.
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

constexpr int kTile = 128;          // tokens per CTA = MMA tile M
constexpr uint32_t kTmemCols = 256;  // one fp32 accumulator column per codeword

// Shared-memory plan of encode_mma_kernel.  The token tile and the codebook are
// stored as grids of 8-row x 16-byte core matrices (the tensor cores' plain
// K-major layout): token r, 16-byte chunk c of its 128-dim K or V vector at
// ((r/8)*16 + c)*128 + (r%8)*16; codeword k, chunk c of subspace m's row at
// m*KB + ((k/8)*CH + c)*128 + (k%8)*16.
template <int M>
struct EncMma {
    static constexpr int DSUB = kHeadDim / M;
    static constexpr int CH = DSUB / 8;                      // 16-byte chunks per sub-vector
    static constexpr int KSTEPS = DSUB / 16;                 // MMAs of K = 16 per subspace
    static constexpr int A_BYTES = kTile * kHeadDim * 2;     // 32 KiB
    static constexpr int KB = kCodewords * DSUB * 2;         // one subspace codebook
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + A_BYTES;
    static constexpr int OFF_N = OFF_B + M * KB;             // |c_k|^2, fp32 [M][K]
    static constexpr int OFF_NMAX = OFF_N + M * kCodewords * 4;
    static constexpr int OFF_BAR = OFF_NMAX + 64;
    static constexpr int OFF_TMEM = OFF_BAR + 8;
    static constexpr int OFF_NEXT = OFF_TMEM + 4;
    static constexpr int SMEM = OFF_NEXT + 4;
    static constexpr uint32_t IDESC = idesc_f16_f32(kTile, kCodewords);
};

// Exact-rule distance from the thread's sub-vector (fp32 pairs) to codeword k.
template <int M>
__device__ __forceinline__ float exact_dist(const unsigned long long (&x2)[EncMma<M>::DSUB / 2],
                                            uint32_t bsub, int k) {
    using C = EncMma<M>;
    float d = 0.f;
#pragma unroll
    for (int c = 0; c < C::CH; ++c) {
        uint4 u;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                     : "r"(bsub + ((((k >> 3) * C::CH + c)) << 7) + ((k & 7) << 4)));
        const uint32_t h[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const unsigned long long e = f2_sub(x2[c * 4 + i], h2_to_f2p(h[i]));
            const float2 sq = f2_unpack(f2_mul(e, e));
            d = __fadd_rn(d, sq.x);
            d = __fadd_rn(d, sq.y);
        }
    }
    return d;
}

// One CTA per (128-token tile, kv head, K-or-V), 4 warps, one thread per token.
//
// For each subspace the tensor cores form a_k = x . c_k for all 128 tokens x
// 256 codewords (fp16 operands, fp32 accumulation in TMEM).  With
// n_k = |c_k|^2, dt_k = n_k - 2 a_k equals |x - c_k|^2 - |x|^2 up to rounding,
// and the exact-rule distance d_k (fp32 separately rounded subtract, multiply
// and add in increasing j) differs from dt_k + |x|^2 by at most
// 2^-14 (|x|^2 + max_k n_k): the exact products and fp32 sums of the MMA, the
// fp32 norms and d_k itself each contribute a few dozen units of 2^-24 of that
// scale, far inside the bound.  So the exact-rule argmin is among the
// candidates dt_k <= min_k dt_k + 2^-13 (|x|^2 + max_k n_k); those (usually
// the nearest codeword and its exact duplicates) are scored with the exact
// rule in increasing k, and the lowest index of the least distance wins: the
// same code as a full scan.  A token whose threshold is not finite (an inf or
// NaN among its inputs) takes the full scan.
template <int M>
__global__ void __launch_bounds__(kTile) encode_mma_kernel(const __grid_constant__ EncodeParams p) {
    using C = EncMma<M>;
    constexpr int D = kHeadDim, K = kCodewords, DSUB = C::DSUB, CH = C::CH;
    extern __shared__ __align__(1024) uint8_t smem[];
    float *sN = reinterpret_cast<float *>(smem + C::OFF_N);
    unsigned *sNmax = reinterpret_cast<unsigned *>(smem + C::OFF_NMAX);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM);
    int *sNext = reinterpret_cast<int *>(smem + C::OFF_NEXT);
    const uint32_t aBase = smem_u32(smem + C::OFF_A), bBase = smem_u32(smem + C::OFF_B);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.y, w = blockIdx.z, t0 = blockIdx.x * kTile, t = t0 + tid;

    int64_t slot = -1;
    int set = 0;
    bool todo = t < p.num_tokens && slot_ok(p, t, slot, set);

    if (warp == 0) tmem_alloc(smem_u32(sTmem), kTmemCols);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    // the token tile (rows past the end are zero)
    for (int i = tid; i < kTile * 16; i += kTile) {
        const int r = i >> 4, c = i & 15;
        const uint32_t dst = aBase + ((((r >> 3) << 4) + c) << 7) + ((r & 7) << 4);
        if (t0 + r < p.num_tokens)
            cp_async_16(dst, reinterpret_cast<const __half *>(p.kv) +
                                 ((static_cast<size_t>(t0 + r) * p.num_kv_heads + kvh) * 2 + w) * D + c * 8);
        else
            asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0u) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    uint32_t phase = 0;
    bool timed_out = false;

    // one pass per distinct set among the tile's tokens (prefill: usually one)
    while (true) {
        if (tid == 0) *sNext = INT_MAX;
        if (tid < M) sNmax[tid] = 0u;
        __syncthreads();
        if (todo) atomicMin(sNext, set);
        __syncthreads();
        const int cur = *sNext;
        if (cur == INT_MAX) break;
        const __half *cb = reinterpret_cast<const __half *>(p.codebooks) +
                           ((static_cast<size_t>(cur) * p.num_kv_heads + kvh) * 2 + w) * M * K * DSUB;
        for (int i = tid; i < M * K * CH; i += kTile) {
            const int m = i / (K * CH), k = (i / CH) % K, c = i % CH;
            cp_async_16(bBase + m * C::KB + (((k >> 3) * CH + c) << 7) + ((k & 7) << 4), cb + static_cast<size_t>(i) * 8);
        }
        cp_async_wait_all();
        __syncthreads();
        // codeword norms (fp32 pair FMAs of exact fp16 squares) and their maxima
#pragma unroll 1
        for (int m = 0; m < M; ++m) {
            unsigned nmax = 0u;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int k = tid + h * kTile;
                unsigned long long acc = 0ull;
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    uint4 u;
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                                 : "r"(bBase + m * C::KB + (((k >> 3) * CH + c) << 7) + ((k & 7) << 4)));
                    const uint32_t hh[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const unsigned long long f = h2_to_f2p(hh[i]);
                        acc = f2_fma(f, f, acc);
                    }
                }
                const float2 a2 = f2_unpack(acc);
                const float n = a2.x + a2.y;
                sN[m * K + k] = n;
                nmax = max(nmax, __float_as_uint(n));         // n >= 0; a NaN orders last
            }
            const unsigned mx = __reduce_max_sync(0xffffffffu, nmax);
            if (lane == 0) atomicMax(&sNmax[m], mx);
        }
        fence_proxy_async_shared();                           // cp.async writes -> tensor-core reads
        __syncthreads();

        const bool mine = todo && set == cur;
        const bool warp_mine = __any_sync(0xffffffffu, mine);
        unsigned long long codes = 0ull;           // byte m = code of subspace m
#pragma unroll 1
        for (int m = 0; m < M; ++m) {
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < C::KSTEPS; ++s) {
                    const uint64_t ad = smem_desc(aBase + ((m * CH + 2 * s) << 7), 128, 16 * 128);
                    const uint64_t bd = smem_desc(bBase + m * C::KB + ((2 * s) << 7), 128, CH * 128);
                    umma_f16(tmem, ad, bd, C::IDESC, s > 0);
                }
                umma_commit(bar);
            }
            if (!mbar_wait_bounded(bar, phase)) timed_out = true;
            phase ^= 1u;
            tc_fence_after();
            if (warp_mine) {                                  // warp-uniform
                // this token's sub-vector and |x|^2
                unsigned long long x2[DSUB / 2];
                float X = 0.f;
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    uint4 u;
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                                 : "r"(aBase + ((((tid >> 3) << 4) + m * CH + c) << 7) + ((tid & 7) << 4)));
                    const uint32_t hh[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x2[c * 4 + i] = h2_to_f2p(hh[i]);
                        const float2 f = f2_unpack(x2[c * 4 + i]);
                        X = fmaf(f.x, f.x, X);
                        X = fmaf(f.y, f.y, X);
                    }
                }
                const float *nrow = sN + m * K;
                const unsigned long long m2 = f2_pack(-2.f, -2.f);
                // pass 1: least dt
                float dmin = INFINITY;
#pragma unroll 1
                for (int j = 0; j < K / 32; j += 2) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(trow + j * 32, r0);
                    tmem_ld32(trow + j * 32 + 32, r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 n0 = *reinterpret_cast<const float2 *>(nrow + j * 32 + i);
                        const float2 n1 = *reinterpret_cast<const float2 *>(nrow + j * 32 + 32 + i);
                        const float2 d0 = f2_unpack(f2_fma(f2_pack(__uint_as_float(r0[i]), __uint_as_float(r0[i + 1])), m2,
                                                           f2_pack(n0.x, n0.y)));
                        const float2 d1 = f2_unpack(f2_fma(f2_pack(__uint_as_float(r1[i]), __uint_as_float(r1[i + 1])), m2,
                                                           f2_pack(n1.x, n1.y)));
                        dmin = min3_f32(dmin, d0.x, d0.y);
                        dmin = min3_f32(dmin, d1.x, d1.y);
                    }
                }
                const float thr = dmin + 0x1p-13f * (X + __uint_as_float(sNmax[m]));
                const bool full = !(fabsf(thr) <= 3.402823466e38f);
                // pass 2: candidates dt <= thr, in increasing k (up to 8 kept)
                unsigned long long list = 0ull;
                int cnt = 0;
#pragma unroll 1
                for (int j = 0; j < K / 32; j += 2) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(trow + j * 32, r0);
                    tmem_ld32(trow + j * 32 + 32, r1);
                    tmem_wait_ld();
                    uint32_t mask0 = 0u, mask1 = 0u;
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 n0 = *reinterpret_cast<const float2 *>(nrow + j * 32 + i);
                        const float2 n1 = *reinterpret_cast<const float2 *>(nrow + j * 32 + 32 + i);
                        const float2 d0 = f2_unpack(f2_fma(f2_pack(__uint_as_float(r0[i]), __uint_as_float(r0[i + 1])), m2,
                                                           f2_pack(n0.x, n0.y)));
                        const float2 d1 = f2_unpack(f2_fma(f2_pack(__uint_as_float(r1[i]), __uint_as_float(r1[i + 1])), m2,
                                                           f2_pack(n1.x, n1.y)));
                        if (d0.x <= thr) mask0 |= 1u << i;
                        if (d0.y <= thr) mask0 |= 2u << i;
                        if (d1.x <= thr) mask1 |= 1u << i;
                        if (d1.y <= thr) mask1 |= 2u << i;
                    }
                    while (mask0) {
                        const int i = __ffs(mask0) - 1;
                        mask0 &= mask0 - 1u;
                        if (cnt < 8) list |= static_cast<unsigned long long>(j * 32 + i) << (8 * cnt);
                        ++cnt;
                    }
                    while (mask1) {
                        const int i = __ffs(mask1) - 1;
                        mask1 &= mask1 - 1u;
                        if (cnt < 8) list |= static_cast<unsigned long long>(j * 32 + 32 + i) << (8 * cnt);
                        ++cnt;
                    }
                }
                // exact rule over the candidates
                const uint32_t bsub = bBase + m * C::KB;
                const bool scan_all = full || cnt > 8;
                const int nc = scan_all ? 0 : cnt;
                const int ncmax = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(nc));
                float best = INFINITY;
                int bk = 0;
                for (int c = 0; c < ncmax; ++c) {
                    if (c < nc) {
                        const int k = static_cast<int>((list >> (8 * c)) & 0xffu);
                        const float d = exact_dist<M>(x2, bsub, k);
                        if (d < best) {
                            best = d;
                            bk = k;
                        }
                    }
                }
                if (scan_all) {
                    for (int k = 0; k < K; ++k) {
                        const float d = exact_dist<M>(x2, bsub, k);
                        if (d < best) {
                            best = d;
                            bk = k;
                        }
                    }
                }
                codes |= static_cast<unsigned long long>(bk) << (8 * m);
            }
            tc_fence_before();
            __syncthreads();                                  // TMEM reads done before the next MMA
        }
        if (mine) {
            const int64_t page = slot / kPage, s = slot % kPage;
            uint8_t *dst = p.code_pages + ((static_cast<size_t>(page) * p.num_kv_heads + kvh) * kPage + s) * 2 * M + w * M;
            if (timed_out) {
                // the accumulators may be incomplete: leave the slot as it was
            } else if (M == 4) {
                *reinterpret_cast<uint32_t *>(dst) = static_cast<uint32_t>(codes);
            } else {
                *reinterpret_cast<unsigned long long *>(dst) = codes;
            }
            todo = false;
        }
    }
    if (timed_out) flag_status(p.status, AQ_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

template <int M>
static cudaError_t launch_encode_mma(const EncodeParams &p, cudaStream_t s) {
    static bool configured = false;                       // attribute set once per process
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(encode_mma_kernel<M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             EncMma<M>::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid(static_cast<unsigned>((p.num_tokens + kTile - 1) / kTile), static_cast<unsigned>(p.num_kv_heads), 2u);
    encode_mma_kernel<M><<<grid, kTile, EncMma<M>::SMEM, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_encode(const EncodeParams &p, int M, cudaStream_t s) {
    if (p.num_tokens == 0) return cudaSuccess;
    const bool small = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads <= 8192;
    if (small) {
        dim3 grid(static_cast<unsigned>(p.num_tokens), static_cast<unsigned>(p.num_kv_heads));
        if (M == 4) encode_cw_kernel<4><<<grid, 256, 0, s>>>(p);
        else encode_cw_kernel<8><<<grid, 256, 0, s>>>(p);
        return cudaGetLastError();
    }
    return M == 4 ? launch_encode_mma<4>(p, s) : launch_encode_mma<8>(p, s);
}

}  // namespace aq
