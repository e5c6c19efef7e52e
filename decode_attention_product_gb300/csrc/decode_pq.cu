// decode_pq.cu -- fused PQ decode attention for sm_103a.
//
// One thread-block cluster of C CTAs handles one (request b, kv head, split).
// CTA `rank` owns subspaces [rank*M/C, (rank+1)*M/C) of both the key and the
// value codebook and 1/C of the split's tokens:
//
//  1. bulk-copy its key and value codebook slices (64/C KiB each) to shared
//     memory (cp.async.bulk + mbarrier), load the G query vectors of the GQA
//     group;
//  2. LUT[m][k][g] = <q_g[m], C^K_m[k]> * scale * log2(e) for its own m
//     (AQPIM blog §4.1: per-subspace partial dot products with the codebook;
//     §5.1 item 3: index -> codebook -> sub-dot -> accumulate, nothing
//     intermediate written to global memory); the rows are exchanged through
//     distributed shared memory so every CTA holds the full M x 256 x G table;
//  3. stream its tokens' uint8 codes through the block table (PAM article
//     §2.2.2), score s = sum_m LUT[m][kcode_m] by table gathers, keep a running
//     max / sum per query head (online softmax, PAM article §2.2.3 item 1) and
//     scatter exp2(s - max) into 256-bin value accumulators W[m][vcode_m][g];
//  4. merge the C CTAs' (max, sum, bins) over distributed shared memory (the
//     hierarchical reduction of PAM article §2.2.3 item 3, inside one cluster)
//     and apply the value codebook slice it owns: o[m*Dsub+j] = sum_k W[m][k]
//     * C^V_m[k][j];
//  5. normalise and store, or store (max, sum, o) partials for the split-KV
//     combine kernel.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace aq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int M, int G, int C>
struct PqCfg {
    static constexpr int D = kHeadDim, K = kCodewords, P = kPage;
    static constexpr int DSUB = D / M;
    static constexpr int MC = M / C;                        // subspaces owned per CTA
    static constexpr int CB_HALVES = MC * K * DSUB;         // owned part of one codebook
    static constexpr int CB_BYTES = CB_HALVES * 2;
    static constexpr int LUT_FLOATS = M * K * G;
    static constexpr int TPT = 8;                           // tokens per thread per chunk
    static constexpr int TOK_PER_PASS = kThreads / G;
    static constexpr int CHUNK = TOK_PER_PASS * TPT;
    // V-product thread mapping
    static constexpr int NJP = MC * DSUB / 2;               // owned j-pairs
    static constexpr int KS = kThreads / NJP;               // k slices
    static constexpr int KSL = K / KS;                      // k per slice
    // shared-memory layout (bytes)
    static constexpr int OFF_BAR = 0;                       // 2 mbarriers
    static constexpr int OFF_MISC = 16;                     // int flags
    static constexpr int OFF_CBK = 128;
    static constexpr int OFF_CBV = OFF_CBK + CB_BYTES;
    static constexpr int OFF_LUT = OFF_CBV + CB_BYTES;
    static constexpr int OFF_BINS = OFF_LUT + LUT_FLOATS * 4;
    static constexpr int OFF_Q = OFF_BINS + LUT_FLOATS * 4;
    static constexpr int OFF_RED = OFF_Q + G * D * 4;       // red_max, red_sum [kWarps][G]
    static constexpr int OFF_XCH = OFF_RED + 2 * kWarps * G * 4;  // m, l [G] (read by peers)
    static constexpr int OFF_FAC = OFF_XCH + 2 * G * 4;     // fac[C][G], mst[G], lst[G], cfac[G]
    static constexpr int SMEM = OFF_FAC + (C + 3) * G * 4 + 16;
    static_assert(K == kThreads, "one thread per codeword in the table build");
    static_assert(KS * NJP == kThreads && KS * KSL == K, "V-product mapping");
    static_assert(KS * MC * DSUB * G * 4 <= CB_BYTES, "V-product reduction fits in the K slice");
    static_assert(CB_BYTES % 16 == 0 && OFF_CBV % 16 == 0 && OFF_LUT % 16 == 0, "alignment");
};

template <int N>
__device__ __forceinline__ void store_vec(float *dst, const float (&v)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4)
            *reinterpret_cast<float4 *>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else if constexpr (N == 2) {
        *reinterpret_cast<float2 *>(dst) = make_float2(v[0], v[1]);
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) dst[i] = v[i];
    }
}

template <int N>
__device__ __forceinline__ void load_vec(float (&v)[N], const float *src) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            float4 t = *reinterpret_cast<const float4 *>(src + i);
            v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
        }
    } else if constexpr (N == 2) {
        float2 t = *reinterpret_cast<const float2 *>(src);
        v[0] = t.x; v[1] = t.y;
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] = src[i];
    }
}

// Code bytes of one token: M key codes then M value codes.
template <int M>
struct Codes;
template <>
struct Codes<4> {
    uint2 v;
    __device__ __forceinline__ void load(const uint8_t *p) { v = ldg_stream_v2(p); }
    __device__ __forceinline__ void zero() { v = make_uint2(0, 0); }
    __device__ __forceinline__ int k(int m) const { return (v.x >> (8 * m)) & 0xff; }
    __device__ __forceinline__ int vv(int m) const { return (v.y >> (8 * m)) & 0xff; }
};
template <>
struct Codes<8> {
    uint4 v;
    __device__ __forceinline__ void load(const uint8_t *p) { v = ldg_stream_v4(p); }
    __device__ __forceinline__ void zero() { v = make_uint4(0, 0, 0, 0); }
    __device__ __forceinline__ int k(int m) const {
        return ((m < 4 ? v.x : v.y) >> (8 * (m & 3))) & 0xff;
    }
    __device__ __forceinline__ int vv(int m) const {
        return ((m < 4 ? v.z : v.w) >> (8 * (m & 3))) & 0xff;
    }
};

template <int C>
__device__ __forceinline__ void cluster_sync_if() {
    if constexpr (C > 1) cg::this_cluster().sync();
}

template <int M, int G, int C>
__global__ void __launch_bounds__(kThreads) pq_decode_kernel(const __grid_constant__ DecodeParams p) {
    using S = PqCfg<M, G, C>;
    constexpr int D = S::D, K = S::K, P = S::P, DSUB = S::DSUB, MC = S::MC;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
    int *sflag = reinterpret_cast<int *>(smem + S::OFF_MISC);   // [0] bad bits of this CTA
    __half *cbk = reinterpret_cast<__half *>(smem + S::OFF_CBK);
    __half *cbv = reinterpret_cast<__half *>(smem + S::OFF_CBV);
    float *lut = reinterpret_cast<float *>(smem + S::OFF_LUT);
    float *bins = reinterpret_cast<float *>(smem + S::OFF_BINS);
    float *qs = reinterpret_cast<float *>(smem + S::OFF_Q);
    float *red_max = reinterpret_cast<float *>(smem + S::OFF_RED);
    float *red_sum = red_max + kWarps * G;
    float *xch = reinterpret_cast<float *>(smem + S::OFF_XCH);  // [0,G): m  [G,2G): l
    float *fac = reinterpret_cast<float *>(smem + S::OFF_FAC);  // [C][G]
    float *mst = fac + C * G;
    float *lst = mst + G;
    float *cfac = lst + G;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int rank = 0;
    if constexpr (C > 1) rank = static_cast<int>(cg::this_cluster().block_rank());
    const int split = blockIdx.x / C;
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int Hq = p.num_q_heads, Hkv = p.num_kv_heads;
    const int S_ = p.num_splits;

    // ---- request-level checks: uniform over the cluster ------------------
    const int L_raw = p.seq_lens[b];
    const int set = p.req_set[b];
    int bad0 = 0;
    if (L_raw < 0 || L_raw > p.max_pages * P || L_raw > p.max_seq_len) bad0 |= AQ_DEV_BAD_LENGTH;
    if (set < 0 || static_cast<int64_t>(set) >= p.num_sets) bad0 |= AQ_DEV_BAD_SET;
    const int ts = split * p.split_len;
    const int te = bad0 ? ts : min(L_raw, ts + p.split_len);
    if (bad0 || ts >= te) {
        // nothing to stream: NaN for a bad request, zeros / empty partials otherwise
        if (rank == 0) {
            if (bad0 && tid == 0) flag_status(p.status, bad0);
            const float v = bad0 ? __int_as_float(0x7fc00000) : 0.0f;
            for (int i = tid; i < G * D; i += kThreads) {
                const int g = i / D, d = i % D;
                const size_t bh = static_cast<size_t>(b) * Hq + kvh * G + g;
                if (S_ == 1) p.out[bh * D + d] = v;
                else if (d == 0) {
                    p.part_ml[(bh * S_ + split) * 2 + 0] = bad0 ? v : -INFINITY;
                    p.part_ml[(bh * S_ + split) * 2 + 1] = bad0 ? v : 0.0f;
                }
            }
        }
        return;
    }

    // ---- 1. async codebook copies, queries, zeroed bins -------------------
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        sflag[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const size_t cb_unit = static_cast<size_t>(M) * K * DSUB;
    const __half *gK = reinterpret_cast<const __half *>(p.codebooks) +
                       ((static_cast<size_t>(set) * Hkv + kvh) * 2) * cb_unit +
                       static_cast<size_t>(rank) * S::CB_HALVES;
    const __half *gV = gK + cb_unit;
    if (tid == 0) {
        const uint64_t pol = policy_evict_first();
        mbar_arrive_expect_tx(&bar[0], S::CB_BYTES);
        bulk_g2s_hint(cbk, gK, S::CB_BYTES, &bar[0], pol);
        mbar_arrive_expect_tx(&bar[1], S::CB_BYTES);
        bulk_g2s_hint(cbv, gV, S::CB_BYTES, &bar[1], pol);
    }
    {
        const float4 *qg = reinterpret_cast<const float4 *>(
            p.q + (static_cast<size_t>(b) * Hq + static_cast<size_t>(kvh) * G) * D);
        for (int i = tid; i < G * D / 4; i += kThreads) reinterpret_cast<float4 *>(qs)[i] = qg[i];
        for (int i = tid; i < S::LUT_FLOATS / 4; i += kThreads)
            reinterpret_cast<float4 *>(bins)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();

    // ---- 2. lookup table for the owned subspaces --------------------------
    if (!mbar_wait_bounded(&bar[0], 0)) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
    {
        constexpr int NCH = DSUB / 8;                   // 16-byte chunks per codeword row
        constexpr int ROWS128 = 128 / (DSUB * 2);       // rows per 128 bytes
        const int rot = (tid / ROWS128) % NCH;          // bank-conflict-free chunk order
#pragma unroll
        for (int mi = 0; mi < MC; ++mi) {
            const int m = rank * MC + mi;
            const __half *row = cbk + (static_cast<size_t>(mi) * K + tid) * DSUB;
            float acc[G];
#pragma unroll
            for (int g = 0; g < G; ++g) acc[g] = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < NCH; ++c0) {
                const int c = (c0 + rot) % NCH;
                const uint4 u = *reinterpret_cast<const uint4 *>(row + c * 8);
                const float2 f0 = h2_to_f2(u.x), f1 = h2_to_f2(u.y), f2 = h2_to_f2(u.z),
                             f3 = h2_to_f2(u.w);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float4 *qv = reinterpret_cast<const float4 *>(qs + g * D + m * DSUB + c * 8);
                    const float4 qa = qv[0], qb = qv[1];
                    float a = acc[g];
                    a = fmaf(qa.x, f0.x, a); a = fmaf(qa.y, f0.y, a);
                    a = fmaf(qa.z, f1.x, a); a = fmaf(qa.w, f1.y, a);
                    a = fmaf(qb.x, f2.x, a); a = fmaf(qb.y, f2.y, a);
                    a = fmaf(qb.z, f3.x, a); a = fmaf(qb.w, f3.y, a);
                    acc[g] = a;
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) acc[g] *= p.scale_log2;
            store_vec<G>(lut + (static_cast<size_t>(m) * K + tid) * G, acc);
        }
    }
    if constexpr (C > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();                                 // every CTA's own rows are written
        constexpr int ROW_F4 = MC * K * G / 4;
#pragma unroll 1
        for (int r = 0; r < C; ++r) {
            if (r == rank) continue;
            float *mine = lut + static_cast<size_t>(r) * MC * K * G;
            const float4 *src = reinterpret_cast<const float4 *>(cluster.map_shared_rank(mine, r));
            float4 *dst = reinterpret_cast<float4 *>(mine);
            for (int i = tid; i < ROW_F4; i += kThreads) dst[i] = src[i];
        }
    }
    __syncthreads();

    // ---- 3. code stream: scores, online softmax, value bins ----------------
    const int n_tok = te - ts;
    const int per = ((n_tok + C - 1) / C + P - 1) / P * P;        // page-aligned share
    const int a0 = ts + rank * per;
    const int e0 = min(te, a0 + per);
    const int g = tid % G, jslot = tid / G;
    const int32_t *bt = p.block_table + static_cast<size_t>(b) * p.max_pages;
    float m_run = -INFINITY, l_run = 0.f;
    int badpage = 0;
#pragma unroll 1
    for (int cb = a0; cb < e0; cb += S::CHUNK) {
        Codes<M> cd[S::TPT];
        float s[S::TPT];
#pragma unroll
        for (int i = 0; i < S::TPT; ++i) {
            const int t = cb + i * S::TOK_PER_PASS + jslot;
            cd[i].zero();
            s[i] = -INFINITY;
            if (t < e0) {
                const int pg = bt[t / P];
                if (pg < 0 || static_cast<int64_t>(pg) >= p.num_pages) {
                    badpage = 1;
                } else {
                    cd[i].load(p.code_pages +
                               ((static_cast<size_t>(pg) * Hkv + kvh) * P + (t % P)) * (2 * M));
                    s[i] = 0.f;          // marks the token valid
                }
            }
        }
        float cm = -INFINITY;
#pragma unroll
        for (int i = 0; i < S::TPT; ++i) {
            if (s[i] == 0.f) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < M; ++m) acc += lut[(m * K + cd[i].k(m)) * G + g];
                s[i] = acc;
                cm = fmaxf(cm, acc);
            }
        }
#pragma unroll
        for (int off = G; off < 32; off <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
        if (lane < G) red_max[warp * G + lane] = cm;
        __syncthreads();
        float cmax = red_max[g];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) cmax = fmaxf(cmax, red_max[w * G + g]);
        const float m_new = fmaxf(m_run, cmax);
        // rescale the bins when a head's running max moved (never on its first
        // chunk); both barriers are unconditional
        const bool have_prev = (m_run != -INFINITY);
        if (tid < G) cfac[tid] = have_prev ? exp2f(m_run - m_new) : 1.f;
        if (__syncthreads_or(have_prev && m_new > m_run)) {
            for (int i = tid; i < S::LUT_FLOATS; i += kThreads) bins[i] *= cfac[i % G];
        }
        if (have_prev) l_run *= exp2f(m_run - m_new);
        m_run = m_new;
        __syncthreads();
        if (m_new != -INFINITY) {
#pragma unroll
            for (int i = 0; i < S::TPT; ++i) {
                if (s[i] != -INFINITY) {
                    const float pv = exp2f(s[i] - m_new);
                    l_run += pv;
#pragma unroll
                    for (int m = 0; m < M; ++m) atomicAdd(&bins[(m * K + cd[i].vv(m)) * G + g], pv);
                }
            }
        }
    }
    if (badpage) atomicOr(&sflag[0], AQ_DEV_BAD_PAGE);
    // per-head sum of this CTA
#pragma unroll
    for (int off = G; off < 32; off <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
    if (lane < G) red_sum[warp * G + lane] = l_run;
    __syncthreads();
    if (tid < G) {
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) l += red_sum[w * G + tid];
        xch[tid] = m_run;          // m_run is uniform per head
        xch[G + tid] = l;
    }
    __syncthreads();

    // ---- 4. merge (max, sum, bins) across the cluster ----------------------
    cluster_sync_if<C>();          // peers' bins and statistics are final
    int bad_all = 0;
    if (tid < G) {
        float mr[C], lr[C];
        float ms = -INFINITY;
#pragma unroll
        for (int r = 0; r < C; ++r) {
            const float *x = xch;
            if constexpr (C > 1) x = cg::this_cluster().map_shared_rank(xch, r);
            mr[r] = x[tid];
            lr[r] = x[G + tid];
            if (lr[r] > 0.f) ms = fmaxf(ms, mr[r]);
        }
        float ls = 0.f;
#pragma unroll
        for (int r = 0; r < C; ++r) {
            const float f = (lr[r] > 0.f) ? exp2f(mr[r] - ms) : 0.f;
            fac[r * G + tid] = f;
            ls += f * lr[r];
        }
        mst[tid] = ms;
        lst[tid] = ls;
    }
    if (tid == 0) {
        int bb = 0;
#pragma unroll
        for (int r = 0; r < C; ++r) {
            const int *f = sflag;
            if constexpr (C > 1) f = cg::this_cluster().map_shared_rank(sflag, r);
            bb |= *f;
        }
        sflag[1] = bb;
        if (sflag[0]) flag_status(p.status, sflag[0]);
    }
    __syncthreads();
    bad_all = sflag[1];
    // W_tot for the owned subspaces -> the LUT region (peers finished reading it)
    float *wtot = lut;
    {
        constexpr int N4 = MC * K * G / 4;
        const size_t base4 = static_cast<size_t>(rank) * MC * K * G / 4;
        for (int i = tid; i < N4; i += kThreads) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int r = 0; r < C; ++r) {
                const float4 *br = reinterpret_cast<const float4 *>(bins);
                if constexpr (C > 1)
                    br = reinterpret_cast<const float4 *>(cg::this_cluster().map_shared_rank(bins, r));
                const float4 v = br[base4 + i];
                const int g0 = (4 * i) % G;
                acc.x += fac[r * G + g0] * v.x;
                acc.y += fac[r * G + (g0 + 1) % G] * v.y;
                acc.z += fac[r * G + (g0 + 2) % G] * v.z;
                acc.w += fac[r * G + (g0 + 3) % G] * v.w;
            }
            reinterpret_cast<float4 *>(wtot)[i] = acc;
        }
    }
    __syncthreads();

    // ---- 5. value codebook product for the owned subspaces -----------------
    if (!mbar_wait_bounded(&bar[1], 0)) {
        atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
        bad_all |= AQ_DEV_TIMEOUT;
    }
    float *ored = reinterpret_cast<float *>(cbk);      // [KS][MC*DSUB][G]
    {
        const int jp = tid % S::NJP, ks = tid / S::NJP;
        const int mi = jp / (DSUB / 2), j2 = (jp % (DSUB / 2)) * 2;
        float acc0[G], acc1[G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) { acc0[gg] = 0.f; acc1[gg] = 0.f; }
#pragma unroll 4
        for (int i = 0; i < S::KSL; ++i) {
            const int k = ks * S::KSL + ((i + ks) % S::KSL);
            const float2 cv = h2_to_f2(
                *reinterpret_cast<const uint32_t *>(cbv + (static_cast<size_t>(mi) * K + k) * DSUB + j2));
            float w[G];
            load_vec<G>(w, wtot + (static_cast<size_t>(mi) * K + k) * G);
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                acc0[gg] = fmaf(w[gg], cv.x, acc0[gg]);
                acc1[gg] = fmaf(w[gg], cv.y, acc1[gg]);
            }
        }
        float *dst = ored + (static_cast<size_t>(ks) * MC * DSUB + mi * DSUB + j2) * G;
        store_vec<G>(dst, acc0);
        store_vec<G>(dst + G, acc1);
    }
    __syncthreads();
    {
        constexpr int NOUT = MC * DSUB * G;
        for (int i = tid; i < NOUT; i += kThreads) {
            float o = 0.f;
#pragma unroll
            for (int ks = 0; ks < S::KS; ++ks) o += ored[static_cast<size_t>(ks) * NOUT + i];
            const int gg = i % G, dl = i / G;                 // dl in [0, MC*DSUB)
            const int d = rank * MC * DSUB + dl;
            const size_t bh = static_cast<size_t>(b) * Hq + static_cast<size_t>(kvh) * G + gg;
            const float nan = __int_as_float(0x7fc00000);
            if (S_ == 1) {
                const float l = lst[gg];
                p.out[bh * D + d] = bad_all ? nan : (l > 0.f ? o / l : 0.f);
            } else {
                p.part_o[(bh * S_ + split) * D + d] = o;
                if (rank == 0 && dl == 0) {
                    p.part_ml[(bh * S_ + split) * 2 + 0] = bad_all ? nan : mst[gg];
                    p.part_ml[(bh * S_ + split) * 2 + 1] = bad_all ? nan : lst[gg];
                }
            }
        }
    }
    // A copy that timed out may still be landing: wait again (bounded) before
    // the shared memory is released.
    if (sflag[0] & AQ_DEV_TIMEOUT) {
        mbar_wait_bounded(&bar[0], 0);
        mbar_wait_bounded(&bar[1], 0);
    }
    cluster_sync_if<C>();          // no CTA leaves while a peer may read its smem
}

__global__ void __launch_bounds__(128) combine_kernel(const __grid_constant__ DecodeParams p) {
    const size_t bh = blockIdx.x;
    const int d = threadIdx.x;
    const int S_ = p.num_splits;
    const float *ml = p.part_ml + bh * S_ * 2;
    float ms = -INFINITY;
    bool nan = false;
    for (int s = 0; s < S_; ++s) {
        const float m = ml[2 * s], l = ml[2 * s + 1];
        if (l != l) nan = true;
        if (l > 0.f) ms = fmaxf(ms, m);
    }
    float num = 0.f, den = 0.f;
    for (int s = 0; s < S_; ++s) {
        const float l = ml[2 * s + 1];
        if (l > 0.f) {
            const float w = exp2f(ml[2 * s] - ms);
            den += w * l;
            num += w * p.part_o[(bh * S_ + s) * kHeadDim + d];
        }
    }
    p.out[bh * kHeadDim + d] = nan ? __int_as_float(0x7fc00000) : (den > 0.f ? num / den : 0.f);
}

template <int M, int G, int C>
cudaError_t launch_one(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    using S = PqCfg<M, G, C>;
    auto kern = pq_decode_kernel<M, G, C>;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C * plan.num_splits), static_cast<unsigned>(p.num_kv_heads),
                       static_cast<unsigned>(p.batch));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = S::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int M, int G>
cudaError_t dispatch_c(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    switch (plan.cluster) {
        case 1: return launch_one<M, G, 1>(p, plan, s);
        case 2: return launch_one<M, G, 2>(p, plan, s);
        case 4: return launch_one<M, G, 4>(p, plan, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

template <int M>
cudaError_t dispatch_g(const DecodeParams &p, int G, const Plan &plan, cudaStream_t s) {
    switch (G) {
        case 1: return dispatch_c<M, 1>(p, plan, s);
        case 2: return dispatch_c<M, 2>(p, plan, s);
        case 4: return dispatch_c<M, 4>(p, plan, s);
        case 8: return dispatch_c<M, 8>(p, plan, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

template <int M>
size_t smem_g(int G, int C) {
#define AQ_SM(GG, CC) \
    if (G == GG && C == CC) return PqCfg<M, GG, CC>::SMEM;
    AQ_SM(1, 1) AQ_SM(1, 2) AQ_SM(1, 4)
    AQ_SM(2, 1) AQ_SM(2, 2) AQ_SM(2, 4)
    AQ_SM(4, 1) AQ_SM(4, 2) AQ_SM(4, 4)
    AQ_SM(8, 1) AQ_SM(8, 2) AQ_SM(8, 4)
#undef AQ_SM
    return 0;
}

}  // namespace

size_t pq_decode_smem_bytes(int M, int G, int cluster) {
    if (M == 4) return smem_g<4>(G, cluster);
    if (M == 8) return smem_g<8>(G, cluster);
    return 0;
}

cudaError_t launch_pq_decode(const DecodeParams &p, int M, int G, const Plan &plan, cudaStream_t s) {
    cudaError_t e;
    if (M == 4) e = dispatch_g<4>(p, G, plan, s);
    else if (M == 8) e = dispatch_g<8>(p, G, plan, s);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    if (plan.num_splits > 1) return launch_combine(p, s);
    return cudaSuccess;
}

cudaError_t launch_combine(const DecodeParams &p, cudaStream_t s) {
    const unsigned n = static_cast<unsigned>(p.batch) * static_cast<unsigned>(p.num_q_heads);
    combine_kernel<<<n, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace aq
