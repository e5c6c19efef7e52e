// fit.cu -- codebook fit by Lloyd k-means (AQPIM blog §3.2 item 2 and §5.2
// item 1: per-sequence codebooks initialised from its first tokens by a quick
// k-means on a small sample set).
//
// One CTA per (unit, subspace).  The unit's N samples (sub-vectors, fp16) and
// the 256 centroids (fp32, plus their fp16 rounding) live in shared memory.
// One step:
//   assign  each sample to its nearest centroid: fp32 squared distance with
//           separately rounded subtract / multiply / add in increasing j, ties
//           to the lowest index (the same decision rule as encode);
//   update  each centroid with members to their mean.  Member sums are formed
//           exactly: an fp16 value is an integer multiple of 2^-24 below 2^16,
//           so x * 2^24 is an int64 and sums of up to 1024 of them are exact in
//           int64 and in double.  Only centroids with members need a sum row:
//           each takes a slot of a compact [min(N, K)][Dsub] array, which keeps
//           the shared memory of a small sample set low enough for several
//           CTAs per SM.  The mean is that exact sum divided by the
//           count in double (correctly rounded), then rounded to fp32 for the
//           next assignment and to fp16 (nearest even) for the codebook.  A
//           centroid without members keeps both values.
// Initial centroid k is sample (k mod N), or (refine) row k of a given codebook:
// the periodic codebook update of AQPIM blog §6.1 item 3 (a few k-means
// iterations on recent vectors, starting from the codebook in use).  A CTA
// reads its own codebook slice before it writes it, so the update may be in
// place.
#include "common.cuh"
#include "internal.h"

namespace aq {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxSamples = 1024;

template <int M>
struct FitCfg {
    static constexpr int D = kHeadDim, K = kCodewords, DSUB = D / M;
    static constexpr int CSTR = DSUB + 4;                   // padded fp32 centroid row
    static size_t smem(int n) {
        size_t b = 0;
        b += static_cast<size_t>(n < K ? n : K) * DSUB * 8;  // isum  int64 [min(N,K)][DSUB]
        b += static_cast<size_t>(K) * CSTR * 4;             // cent  fp32  [K][CSTR]
        b += static_cast<size_t>(K) * DSUB * 2;             // c16   fp16  [K][DSUB]
        b += static_cast<size_t>(n) * DSUB * 2;             // xs    fp16  [N][DSUB]
        b += static_cast<size_t>(n) * 4;                    // assign int  [N]
        b += static_cast<size_t>(K) * 4;                    // cnt   int   [K]
        b += static_cast<size_t>(K) * 4;                    // slot  int   [K]
        return b + 64;                                      // nused, chg
    }
};

template <int M>
__global__ void __launch_bounds__(kThreads) fit_kernel(const __grid_constant__ FitParams p) {
    using F = FitCfg<M>;
    constexpr int D = F::D, K = F::K, DSUB = F::DSUB, CSTR = F::CSTR;
    extern __shared__ __align__(16) unsigned char smem[];
    const int N = p.n_samples;
    const int nslot = N < K ? N : K;
    long long *isum = reinterpret_cast<long long *>(smem);
    float *cent = reinterpret_cast<float *>(isum + nslot * DSUB);
    __half *c16 = reinterpret_cast<__half *>(cent + K * CSTR);
    __half *xs = c16 + K * DSUB;
    int *asg = reinterpret_cast<int *>(xs + static_cast<size_t>(N) * DSUB);
    int *cnt = asg + N;
    int *slot = cnt + K;
    int *nused = slot + K;
    int *chg = nused + 1;                                   // [2]: an assignment changed in step it (it & 1)

    const int64_t u = blockIdx.x;
    const int m = blockIdx.y, tid = threadIdx.x;
    const __half *src = reinterpret_cast<const __half *>(p.samples) + static_cast<size_t>(u) * N * D + m * DSUB;
    for (int i = tid; i < N * DSUB; i += kThreads) xs[i] = src[(i / DSUB) * D + (i % DSUB)];
    __syncthreads();
    const size_t cbase = (static_cast<size_t>(u) * M + m) * K * DSUB;
    for (int i = tid; i < K * DSUB; i += kThreads) {
        const int k = i / DSUB, j = i % DSUB;
        if (p.cent_in) {
            cent[k * CSTR + j] = p.cent_in[cbase + i];
        } else if (p.cb_init) {                          // refine: start from a codebook
            const __half h = reinterpret_cast<const __half *>(p.cb_init)[cbase + i];
            cent[k * CSTR + j] = __half2float(h);
            c16[i] = h;
        } else {
            const __half h = xs[(k % N) * DSUB + j];
            cent[k * CSTR + j] = __half2float(h);
            c16[i] = h;
        }
    }
    if (tid == 0) chg[0] = chg[1] = 0;
    __syncthreads();

    // assignment mapping: NCH threads per sample, each over K / NCH centroids
    int nch = 1;
    while (nch < 8 && nch * 2 * N <= kThreads) nch *= 2;
    const int spass = kThreads / nch;                        // samples per pass
    const int ch = tid % nch, kspan = K / nch;
    const int iters = p.cent_in ? 1 : p.iters;
    for (int it = 0; it < iters; ++it) {
        for (int n0 = 0; n0 < N; n0 += spass) {
            const int n = n0 + tid / nch;
            unsigned long long key = ~0ull;
            if (n < N) {
                unsigned long long x2[DSUB / 2];
#pragma unroll
                for (int j = 0; j < DSUB; j += 2)
                    x2[j / 2] = h2_to_f2p(*reinterpret_cast<const uint32_t *>(xs + n * DSUB + j));
                float best = INFINITY;
                int bk = 0;
                for (int i = 0; i < kspan; ++i) {
                    const int k = ch * kspan + ((i + ch) % kspan);   // staggered: no bank conflicts
                    const float4 *c4 = reinterpret_cast<const float4 *>(cent + k * CSTR);
                    // separately rounded subtract and multiply (pairs), adds in increasing j
                    float d = 0.f;
#pragma unroll
                    for (int j = 0; j < DSUB; j += 4) {
                        const float4 c = c4[j / 4];
                        const unsigned long long e0 = f2_sub(x2[j / 2], f2_pack(c.x, c.y));
                        const unsigned long long e1 = f2_sub(x2[j / 2 + 1], f2_pack(c.z, c.w));
                        const float2 s0 = f2_unpack(f2_mul(e0, e0)), s1 = f2_unpack(f2_mul(e1, e1));
                        d = __fadd_rn(d, s0.x);
                        d = __fadd_rn(d, s0.y);
                        d = __fadd_rn(d, s1.x);
                        d = __fadd_rn(d, s1.y);
                    }
                    if (d < best || (d == best && k < bk)) { best = d; bk = k; }
                }
                key = (static_cast<unsigned long long>(__float_as_uint(best)) << 32) | static_cast<unsigned>(bk);
            }
            for (int off = 1; off < nch; off <<= 1) {
                const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, off);
                key = o < key ? o : key;
            }
            if (n < N && ch == 0) {
                const int a = static_cast<int>(key & 0xffffffffu);
                if (it > 0 && asg[n] != a) chg[it & 1] = 1;
                asg[n] = a;
            }
        }
        for (int i = tid; i < nslot * DSUB; i += kThreads) isum[i] = 0;
        for (int i = tid; i < K; i += kThreads) cnt[i] = 0;
        if (tid == 0) *nused = 0;
        __syncthreads();
        // Exact early exit: an assignment equal to the previous step's gives
        // the same members, hence the same exact sums and centroids, so every
        // later step would repeat it -- the result is the full fit's.
        if (it > 0 && chg[it & 1] == 0) break;
        if (tid == 0) chg[(it + 1) & 1] = 0;
        // member counts; the first member of a centroid claims its sum slot
        for (int n = tid; n < N; n += kThreads) {
            const int k = asg[n];
            if (atomicAdd(&cnt[k], 1) == 0) slot[k] = atomicAdd(nused, 1);
        }
        __syncthreads();
        for (int i = tid; i < N * DSUB; i += kThreads) {
            const int n = i / DSUB, j = i % DSUB;
            // fp16 -> exact int64 multiple of 2^-24
            const long long v = static_cast<long long>(ldexpf(__half2float(xs[i]), 24));
            atomicAdd(reinterpret_cast<unsigned long long *>(&isum[slot[asg[n]] * DSUB + j]),
                      static_cast<unsigned long long>(v));
        }
        __syncthreads();
        for (int i = tid; i < K * DSUB; i += kThreads) {
            const int k = i / DSUB, j = i % DSUB;
            const int c = cnt[k];
            if (c > 0) {
                const double mean = __ddiv_rn(ldexp(static_cast<double>(isum[slot[k] * DSUB + j]), -24),
                                              static_cast<double>(c));
                cent[k * CSTR + j] = __double2float_rn(mean);
                c16[i] = __double2half(mean);
            }
        }
        __syncthreads();
    }
    if (p.assign) {
        for (int n = tid; n < N; n += kThreads)
            p.assign[(static_cast<size_t>(u) * N + n) * M + m] = asg[n];
    }
    if (p.cent_out) {
        for (int i = tid; i < K * DSUB; i += kThreads)
            p.cent_out[cbase + i] = cent[(i / DSUB) * CSTR + (i % DSUB)];
    }
    if (p.codebooks) {
        __half *dst = reinterpret_cast<__half *>(p.codebooks) + cbase;
        for (int i = tid; i < K * DSUB; i += kThreads) dst[i] = c16[i];
    }
}

template <int M>
cudaError_t launch_m(const FitParams &p, cudaStream_t s) {
    const size_t smem = FitCfg<M>::smem(p.n_samples);
    static SmemAttr attr_state;                    // opt-in dynamic shared memory, per device
    if (cudaError_t e = ensure_smem_attr(attr_state, reinterpret_cast<const void *>(fit_kernel<M>),
                                         FitCfg<M>::smem(kMaxSamples));
        e != cudaSuccess)
        return e;
    dim3 grid(static_cast<unsigned>(p.num_units), static_cast<unsigned>(M));
    fit_kernel<M><<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t fit_smem_bytes(int M, int n_samples) {
    return M == 4 ? FitCfg<4>::smem(n_samples) : FitCfg<8>::smem(n_samples);
}

cudaError_t launch_fit(const FitParams &p, int M, cudaStream_t s) {
    if (p.num_units == 0) return cudaSuccess;
    return M == 4 ? launch_m<4>(p, s) : launch_m<8>(p, s);
}

}  // namespace aq
