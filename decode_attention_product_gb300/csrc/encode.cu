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
constexpr int kEncThreads = 256;    // two threads per token, one per half of the codewords
constexpr uint32_t kTmemCols = 256;  // one fp32 accumulator column per codeword

// Shared-memory plan of encode_mma_kernel.  Every tensor-core operand is a
// grid of 8-row x 16-byte core matrices (the plain K-major layout):
//   A   token r, 16-byte chunk c of its 128-dim K or V vector at
//       ((r/8)*16 + c)*128 + (r%8)*16 (fp16)
//   B   codeword k, chunk c of subspace m's row at m*KB + ((k/8)*CH + c)*128 + (k%8)*16
//   BN  codeword k's norm |c_k|^2 as three tf32-exact parts (hi, mid, lo, 0),
//       then 16 zero bytes: ((k/8)*2 + h)*128 + (k%8)*16 (fp32)
//   ONE every row (-1/2, -1/2, -1/2, 0) then zeros, same geometry as BN (fp32)
template <int M>
struct EncMma {
    static constexpr int DSUB = kHeadDim / M;
    static constexpr int CH = DSUB / 8;                      // 16-byte chunks per sub-vector
    static constexpr int KSTEPS = DSUB / 16;                 // fp16 MMAs of K = 16 per subspace
    static constexpr int A_BYTES = kTile * kHeadDim * 2;     // 32 KiB
    static constexpr int KB = kCodewords * DSUB * 2;         // one subspace codebook
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + A_BYTES;
    static constexpr int OFF_BN = OFF_B + M * KB;
    static constexpr int OFF_ONE = OFF_BN + kCodewords * 32;
    static constexpr int OFF_XMAX = OFF_ONE + kTile * 32;    // [2][kTile] fp32 half maxima
    static constexpr int OFF_XBEST = OFF_XMAX + 2 * kTile * 4; // [2][kTile] (distance, index)
    static constexpr int OFF_NMAX = OFF_XBEST + 2 * kTile * 8;
    static constexpr int OFF_BAR = OFF_NMAX + 64;
    static constexpr int OFF_TMEM = OFF_BAR + 8;
    static constexpr int OFF_NEXT = OFF_TMEM + 4;
    static constexpr int SMEM = OFF_NEXT + 4;
    static constexpr uint32_t IDESC = idesc_f16_f32(kTile, kCodewords);
    static constexpr uint32_t IDESC_N = idesc_tf32_f32(kTile, kCodewords);
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 u;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w) : "r"(addr));
    return u;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Exact-rule distance from the thread's sub-vector (fp32 pairs) to a codeword
// row given as its raw fp16 words.
template <int M>
__device__ __forceinline__ float exact_dist(const unsigned long long (&x2)[EncMma<M>::DSUB / 2],
                                            const uint32_t (&row)[EncMma<M>::DSUB / 2]) {
    float d = 0.f;
#pragma unroll
    for (int i = 0; i < EncMma<M>::DSUB / 2; ++i) {
        const unsigned long long e = f2_sub(x2[i], h2_to_f2p(row[i]));
        const float2 sq = f2_unpack(f2_mul(e, e));
        d = __fadd_rn(d, sq.x);
        d = __fadd_rn(d, sq.y);
    }
    return d;
}

template <int M>
__device__ __forceinline__ void load_row(uint32_t bsub, int k, uint32_t (&row)[EncMma<M>::DSUB / 2]) {
#pragma unroll
    for (int c = 0; c < EncMma<M>::CH; ++c) {
        const uint4 u = lds128(bsub + (((k >> 3) * EncMma<M>::CH + c) << 7) + ((k & 7) << 4));
        row[4 * c] = u.x;
        row[4 * c + 1] = u.y;
        row[4 * c + 2] = u.z;
        row[4 * c + 3] = u.w;
    }
}

// tf32 keeps 10 fraction bits: clearing the other 13 leaves a value the tensor
// core takes as it is.
__device__ __forceinline__ float tf32_trunc(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u); }

// Synchronise the two warps (w and w + 4) that share TMEM lanes 32(w%4)...
__device__ __forceinline__ void pair_sync(int warp) {
    asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
}

// One CTA per (128-token tile, kv head, K-or-V), 8 warps: thread (h, r) serves
// token r against codewords [128h, 128h + 128); warps w and w + 4 read the same
// TMEM lanes.
//
// For each subspace the tensor cores accumulate, for all 128 tokens x 256
// codewords, acc_k = x . c_k - |c_k|^2 / 2: two (Dsub 32) or one (Dsub 16)
// fp16 MMAs of x against the codebook, then one tf32 MMA of a constant
// (-1/2, -1/2, -1/2) tile against the norms split into three tf32-exact parts
// (their sum is the fp32 norm exactly; tf32 has the fp32 exponent range).
// dt_k = -2 acc_k equals |x - c_k|^2 - |x|^2 up to rounding, and the
// exact-rule distance d_k (fp32 separately rounded subtract, multiply and add
// in increasing j) differs from dt_k + |x|^2 by at most 2^-13 (|x|^2 + max n):
// exact products, fp32 sums in the MMAs (a few dozen units of 2^-24 of
// sum |x_j c_kj| + |c_k|^2 / 2 even for truncating adders), the fp32 norm and
// d_k itself stay far inside that.  So the exact-rule argmin is among the
// candidates acc_k >= max acc - 2^-13 (|x|^2 + max n); those (usually the
// nearest codeword and its exact duplicates) are scored with the exact rule in
// increasing k and the lowest index of the least distance wins: the code a
// full scan gives.  A token whose threshold is not finite (an inf or NaN among
// its inputs) takes the full scan.
template <int M>
__global__ void __launch_bounds__(kEncThreads, 2) encode_mma_kernel(const __grid_constant__ EncodeParams p) {
    using C = EncMma<M>;
    constexpr int D = kHeadDim, K = kCodewords, DSUB = C::DSUB, CH = C::CH, KH = K / 2;
    extern __shared__ __align__(1024) uint8_t smem[];
    float *sXmax = reinterpret_cast<float *>(smem + C::OFF_XMAX);
    uint2 *sXbest = reinterpret_cast<uint2 *>(smem + C::OFF_XBEST);
    unsigned *sNmax = reinterpret_cast<unsigned *>(smem + C::OFF_NMAX);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM);
    int *sNext = reinterpret_cast<int *>(smem + C::OFF_NEXT);
    const uint32_t aBase = smem_u32(smem + C::OFF_A), bBase = smem_u32(smem + C::OFF_B);
    const uint32_t bnBase = smem_u32(smem + C::OFF_BN), oneBase = smem_u32(smem + C::OFF_ONE);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = tid & (kTile - 1), half = tid >> 7;
    const int kvh = blockIdx.y, w = blockIdx.z, t0 = blockIdx.x * kTile, t = t0 + r;

    int64_t slot = -1;
    int set = 0;
    bool todo = t < p.num_tokens && slot_ok(p, t, slot, set);

    if (warp == 0) tmem_alloc(smem_u32(sTmem), kTmemCols);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    // the token tile (rows past the end are zero)
    for (int i = tid; i < kTile * 16; i += kEncThreads) {
        const int rr = i >> 4, c = i & 15;
        const uint32_t dst = aBase + ((((rr >> 3) << 4) + c) << 7) + ((rr & 7) << 4);
        if (t0 + rr < p.num_tokens)
            cp_async_16(dst, reinterpret_cast<const __half *>(p.kv) +
                                 ((static_cast<size_t>(t0 + rr) * p.num_kv_heads + kvh) * 2 + w) * D + c * 8);
        else
            sts128(dst, 0u, 0u, 0u, 0u);
    }
    // the constant tile (row r, half h of its 32 bytes) and the zero halves of
    // the norm rows (row tid)
    {
        const uint32_t hv = half ? 0u : __float_as_uint(-0.5f);
        sts128(oneBase + ((r >> 3) << 8) + (half << 7) + ((r & 7) << 4), hv, hv, hv, 0u);
        sts128(bnBase + ((tid >> 3) << 8) + 128 + ((tid & 7) << 4), 0u, 0u, 0u, 0u);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + half * KH;
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
        for (int i = tid; i < M * K * CH; i += kEncThreads) {
            const int m = i / (K * CH), k = (i / CH) % K, c = i % CH;
            cp_async_16(bBase + m * C::KB + (((k >> 3) * CH + c) << 7) + ((k & 7) << 4), cb + static_cast<size_t>(i) * 8);
        }
        cp_async_wait_all();
        __syncthreads();

        const bool mine = todo && set == cur;
        const bool warp_mine = __any_sync(0xffffffffu, mine);   // the same for warps w and w + 4
        unsigned long long codes = 0ull;                      // byte m = code of subspace m
#pragma unroll 1
        for (int m = 0; m < M; ++m) {
            // norm of codeword tid of subspace m (fp32 pair FMAs of exact fp16
            // squares), stored as tf32 parts; the maximum norm
            {
                unsigned long long acc = 0ull;
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    const uint4 u = lds128(bBase + m * C::KB + (((tid >> 3) * CH + c) << 7) + ((tid & 7) << 4));
                    const uint32_t h4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const unsigned long long f = h2_to_f2p(h4[i]);
                        acc = f2_fma(f, f, acc);
                    }
                }
                const float2 a2 = f2_unpack(acc);
                const float n = a2.x + a2.y;
                const float hi = tf32_trunc(n), r1 = n - hi, mid = tf32_trunc(r1), lo = r1 - mid;
                sts128(bnBase + ((tid >> 3) << 8) + ((tid & 7) << 4), __float_as_uint(hi), __float_as_uint(mid),
                       __float_as_uint(lo), 0u);
                const unsigned mx = __reduce_max_sync(0xffffffffu, __float_as_uint(n));   // n >= 0; NaN last
                if (lane == 0) atomicMax(&sNmax[m], mx);
            }
            fence_proxy_async_shared();                       // generic writes -> tensor-core reads
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < C::KSTEPS; ++s) {
                    const uint64_t ad = smem_desc(aBase + ((m * CH + 2 * s) << 7), 128, 16 * 128);
                    const uint64_t bd = smem_desc(bBase + m * C::KB + ((2 * s) << 7), 128, CH * 128);
                    umma_f16(tmem, ad, bd, C::IDESC, s > 0);
                }
                umma_tf32(tmem, smem_desc(oneBase, 128, 256), smem_desc(bnBase, 128, 256), C::IDESC_N, 1u);
                umma_commit(bar);
            }
            if (!mbar_wait_bounded(bar, phase)) timed_out = true;
            phase ^= 1u;
            tc_fence_after();
            if (warp_mine) {                                  // uniform over the warp pair
                // this token's sub-vector and |x|^2
                unsigned long long x2[DSUB / 2];
                float X = 0.f;
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    const uint4 u = lds128(aBase + ((((r >> 3) << 4) + m * CH + c) << 7) + ((r & 7) << 4));
                    const uint32_t h4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x2[c * 4 + i] = h2_to_f2p(h4[i]);
                        const float2 f = f2_unpack(x2[c * 4 + i]);
                        X = fmaf(f.x, f.x, X);
                        X = fmaf(f.y, f.y, X);
                    }
                }
                // pass 1: the largest acc of this half, then of both
                float amax = -INFINITY;
#pragma unroll 1
                for (int j = 0; j < KH / 32; j += 2) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(trow + j * 32, r0);
                    tmem_ld32(trow + j * 32 + 32, r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        amax = max3_f32(amax, __uint_as_float(r0[i]), __uint_as_float(r0[i + 1]));
                        amax = max3_f32(amax, __uint_as_float(r1[i]), __uint_as_float(r1[i + 1]));
                    }
                }
                sXmax[half * kTile + r] = amax;
                pair_sync(warp);
                amax = fmaxf(sXmax[r], sXmax[kTile + r]);
                const float thr = amax - 0x1p-13f * (X + __uint_as_float(sNmax[m]));
                const bool full = !(fabsf(thr) <= 3.402823466e38f);
                // pass 2: this half's candidates acc >= thr, in increasing k (up to 16 kept)
                unsigned long long list0 = 0ull, list1 = 0ull;
                int cnt = 0;
#pragma unroll 1
                for (int j = 0; j < KH / 32; j += 2) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(trow + j * 32, r0);
                    tmem_ld32(trow + j * 32 + 32, r1);
                    tmem_wait_ld();
                    uint32_t mask0 = 0u, mask1 = 0u;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (__uint_as_float(r0[i]) >= thr) mask0 |= 1u << i;
                        if (__uint_as_float(r1[i]) >= thr) mask1 |= 1u << i;
                    }
                    while (mask0) {
                        const int i = __ffs(mask0) - 1;
                        mask0 &= mask0 - 1u;
                        const unsigned long long kk = static_cast<unsigned long long>(j * 32 + i) << (8 * (cnt & 7));
                        if (cnt < 8) list0 |= kk;
                        else if (cnt < 16) list1 |= kk;
                        ++cnt;
                    }
                    while (mask1) {
                        const int i = __ffs(mask1) - 1;
                        mask1 &= mask1 - 1u;
                        const unsigned long long kk = static_cast<unsigned long long>(j * 32 + 32 + i) << (8 * (cnt & 7));
                        if (cnt < 8) list0 |= kk;
                        else if (cnt < 16) list1 |= kk;
                        ++cnt;
                    }
                }
                // exact rule over this half's candidates (indices relative to
                // the half).  A candidate whose row equals the current best's
                // bit for bit has the same distance at a higher index and
                // cannot win: it is skipped (the codebook fit leaves many exact
                // copies of its seed rows).
                const uint32_t bsub = bBase + m * C::KB;
                const int kbase = half * KH;
                const bool scan_all = full || cnt > 16;
                const int nc = scan_all ? 0 : cnt;
                const int ncmax = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(nc));
                float best = INFINITY;
                int bk = 0;
                uint32_t brow[DSUB / 2];
                for (int c = 0; c < ncmax; ++c) {
                    if (c < nc) {
                        const int k = kbase + static_cast<int>(((c < 8 ? list0 : list1) >> (8 * (c & 7))) & 0xffu);
                        uint32_t row[DSUB / 2];
                        load_row<M>(bsub, k, row);
                        bool same = c > 0;
#pragma unroll
                        for (int i = 0; i < DSUB / 2; ++i) same = same && row[i] == brow[i];
                        if (!same) {
                            const float d = exact_dist<M>(x2, row);
                            if (d < best || c == 0) {
                                if (d < best) {
                                    best = d;
                                    bk = k;
                                }
#pragma unroll
                                for (int i = 0; i < DSUB / 2; ++i) brow[i] = row[i];
                            }
                        }
                    }
                }
                if (scan_all) {
                    for (int k = kbase; k < kbase + KH; ++k) {
                        uint32_t row[DSUB / 2];
                        load_row<M>(bsub, k, row);
                        const float d = exact_dist<M>(x2, row);
                        if (d < best) {
                            best = d;
                            bk = k;
                        }
                    }
                }
                // lower half first: the upper half wins only with a strictly
                // smaller distance (its indices are all higher)
                sXbest[half * kTile + r] = make_uint2(__float_as_uint(best), static_cast<unsigned>(bk));
                pair_sync(warp);
                if (half == 0) {
                    const uint2 up = sXbest[kTile + r];
                    if (__uint_as_float(up.x) < best) bk = static_cast<int>(up.y);
                    codes |= static_cast<unsigned long long>(bk) << (8 * m);
                }
            }
            tc_fence_before();                                // TMEM reads before the next MMA
        }
        if (mine && half == 0) {
            const int64_t page = slot / kPage, s = slot % kPage;
            uint8_t *dst = p.code_pages + ((static_cast<size_t>(page) * p.num_kv_heads + kvh) * kPage + s) * 2 * M + w * M;
            if (timed_out) {
                // the accumulators may be incomplete: leave the slot as it was
            } else if (M == 4) {
                *reinterpret_cast<uint32_t *>(dst) = static_cast<uint32_t>(codes);
            } else {
                *reinterpret_cast<unsigned long long *>(dst) = codes;
            }
        }
        if (mine) todo = false;
        __syncthreads();                                      // B and the norms free for the next set
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
    static SmemAttr attr_state;                           // opt-in dynamic shared memory, per device
    if (cudaError_t e = ensure_smem_attr(attr_state, reinterpret_cast<const void *>(encode_mma_kernel<M>),
                                         EncMma<M>::SMEM);
        e != cudaSuccess)
        return e;
    dim3 grid(static_cast<unsigned>((p.num_tokens + kTile - 1) / kTile), static_cast<unsigned>(p.num_kv_heads), 2u);
    encode_mma_kernel<M><<<grid, kEncThreads, EncMma<M>::SMEM, s>>>(p);
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
