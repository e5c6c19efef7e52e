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
    static constexpr int ROW_FLOATS = MC * K * G;           // one rank's rows of LUT / bins
    static constexpr int TPT = 8;                           // tokens per thread per chunk
    static constexpr int TOK_PER_PASS = kThreads / G;
    static constexpr int CHUNK = TOK_PER_PASS * TPT;
    // statistics pushed with the bins: m[G], l[G], new-token score[G], bad flag
    static constexpr int STAT_FLOATS = 3 * G + 1;
    static constexpr int INC_STRIDE = ROW_FLOATS + (STAT_FLOATS + 3) / 4 * 4;
    // shared-memory layout (bytes)
    static constexpr int OFF_BAR = 0;                       // 5 mbarriers
    static constexpr int OFF_MISC = 64;                     // int flags
    static constexpr int OFF_CBK = 128;
    static constexpr int OFF_CBV = OFF_CBK + CB_BYTES;
    static constexpr int OFF_LUT = OFF_CBV + CB_BYTES;
    static constexpr int OFF_BINS = OFF_LUT + LUT_FLOATS * 4;
    static constexpr int BIN_WORDS = LUT_FLOATS;            // u32 value bins [M][K][G]
    // [C-1][INC_STRIDE] from the peers; sender src lands in slot (src - dst - 1) mod C
    static constexpr int OFF_INC = OFF_BINS + BIN_WORDS * 4;
    static constexpr int OFF_Q = OFF_INC + (C > 1 ? (C - 1) * INC_STRIDE * 4 : 0);
    static constexpr int OFF_RED = OFF_Q + G * D * 4;       // red_max, red_sum [kWarps][G]
    static constexpr int OFF_STAT = OFF_RED + 2 * kWarps * G * 4;  // mst, lst, cfac [G], fac [C][G]
    // fused step: the new token's owned sub-vectors [2][MC][DSUB] f32, its codes
    // [2][M] int, its score [G], argmin keys [kWarps] u64
    static constexpr int OFF_NEW = (OFF_STAT + (3 + C) * G * 4 + 15) / 16 * 16;
    static constexpr int NEW_BYTES = 2 * MC * DSUB * 4 + 2 * M * 4 + G * 4 + 8 * kWarps + 8;
    static constexpr int OFF_CODES = (OFF_NEW + NEW_BYTES + 15) / 16 * 16;  // [share][2M] uint8
    static constexpr int PAGE_BYTES = P * 2 * M;            // one page's codes for one kv head
    static constexpr int PPL = kMaxShare / P / 32;          // page ids per lane of warp 0
    static size_t smem(int share) { return OFF_CODES + static_cast<size_t>(share) * 2 * M; }
    static_assert(K == kThreads, "one thread per codeword in the table build");
    static_assert((MC * DSUB / 4) <= 32 && 32 % (MC * DSUB / 4) == 0, "V-product quads within a warp");
    static_assert(kWarps * MC * DSUB * G * 4 <= CB_BYTES, "V-product reduction fits in the K slice");
    static_assert(CB_BYTES % 16 == 0 && OFF_LUT % 16 == 0 && OFF_INC % 16 == 0 && OFF_Q % 16 == 0,
                  "alignment");
    static_assert(ROW_FLOATS % 4 == 0 && INC_STRIDE % 4 == 0, "vector pushes");
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

// Push N floats from registers to the same offset in a peer's shared memory.
template <int N>
__device__ __forceinline__ void push_vec(uint32_t raddr, const float (&v)[N], uint32_t rbar) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4)
            st_async_v4(raddr + 4 * i, make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]), rbar);
    } else if constexpr (N == 2) {
        st_async_v2(raddr, v[0], v[1], rbar);
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) st_async_f32(raddr + 4 * i, v[i], rbar);
    }
}

// Code bytes of one token: M key codes then M value codes.
template <int M>
struct Codes;
template <>
struct Codes<4> {
    uint2 v;
    __device__ __forceinline__ void load(const uint8_t *p) { v = *reinterpret_cast<const uint2 *>(p); }
    __device__ __forceinline__ int k(int m) const { return (v.x >> (8 * m)) & 0xff; }
    __device__ __forceinline__ int vv(int m) const { return (v.y >> (8 * m)) & 0xff; }
};
template <>
struct Codes<8> {
    uint4 v;
    __device__ __forceinline__ void load(const uint8_t *p) { v = *reinterpret_cast<const uint4 *>(p); }
    __device__ __forceinline__ int k(int m) const {
        return ((m < 4 ? v.x : v.y) >> (8 * (m & 3))) & 0xff;
    }
    __device__ __forceinline__ int vv(int m) const {
        return ((m < 4 ? v.z : v.w) >> (8 * (m & 3))) & 0xff;
    }
};

// One codeword row (DSUB halves, NCH 16-byte chunks) into registers, chunk c
// of the row landing in u[(c - rot) mod NCH]: threads that read neighbouring
// rows start at different chunks, so a quarter-warp's 16-byte reads fall in
// distinct banks.
template <int NCH>
__device__ __forceinline__ void load_row_rotated(uint4 (&u)[NCH], const __half *row, int rot) {
    const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
#pragma unroll
    for (int c0 = 0; c0 < NCH; ++c0) u[c0] = r4[(c0 + rot) % NCH];
}

// Squared distance between x (NCH*8 floats) and a row held by load_row_rotated:
// fp32 with separately rounded subtract / multiply / add in increasing
// dimension order (the encode decision rule).
template <int NCH>
__device__ __forceinline__ float row_distance(const uint4 (&u)[NCH], const float *x, int rot) {
    float d = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int c0 = (c - rot + NCH) % NCH;
        uint4 w = u[0];
#pragma unroll
        for (int i = 1; i < NCH; ++i)
            if (c0 == i) w = u[i];
        const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float2 f = h2_to_f2(w4[h]);
            float e = __fsub_rn(x[c * 8 + 2 * h], f.x);
            d = __fadd_rn(d, __fmul_rn(e, e));
            e = __fsub_rn(x[c * 8 + 2 * h + 1], f.y);
            d = __fadd_rn(d, __fmul_rn(e, e));
        }
    }
    return d;
}

// CTA-wide argmin over one distance per thread (thread = codeword), lowest
// index on ties; returns the code to every thread.  Distances are >= 0, so
// their bit patterns order like their values.
__device__ __forceinline__ int block_argmin(float d, unsigned long long *keys) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long key = (static_cast<unsigned long long>(__float_as_uint(d)) << 32) | static_cast<unsigned>(tid);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, off);
        key = o < key ? o : key;
    }
    __syncthreads();                                   // keys[] free from a previous use
    if (lane == 0) keys[warp] = key;
    __syncthreads();
    unsigned long long best = keys[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) best = keys[w] < best ? keys[w] : best;
    return static_cast<int>(best & 0xffu);
}

// CTAs per SM the register budget is sized for: shared memory (LUT, bins and
// pushed rows all scale with G) allows about 4 / 2 / 1 resident CTAs.
template <int G>
constexpr int kMinBlocks = G <= 2 ? 4 : (G == 4 ? 2 : 1);

// APPEND = the fused decode step: the token at position seq_len-1 of every
// request is encoded here (each cluster CTA encodes the subspaces it owns) and
// written to its page slot, and the attention includes it.
template <int M, int G, int C, bool APPEND>
__global__ void __launch_bounds__(kThreads, kMinBlocks<G>) pq_decode_kernel(const __grid_constant__ DecodeParams p) {
    using S = PqCfg<M, G, C>;
    constexpr int D = S::D, K = S::K, P = S::P, DSUB = S::DSUB, MC = S::MC, TPT = S::TPT;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);   // CK, CV, LUT in, bins in, codes+q
    int *sflag = reinterpret_cast<int *>(smem + S::OFF_MISC);           // [0] local bad, [1] all
    __half *cbk = reinterpret_cast<__half *>(smem + S::OFF_CBK);
    __half *cbv = reinterpret_cast<__half *>(smem + S::OFF_CBV);
    float *lut = reinterpret_cast<float *>(smem + S::OFF_LUT);
    float *bins = reinterpret_cast<float *>(smem + S::OFF_BINS);
    float *inc = reinterpret_cast<float *>(smem + S::OFF_INC);
    float *qs = reinterpret_cast<float *>(smem + S::OFF_Q);
    float *red_max = reinterpret_cast<float *>(smem + S::OFF_RED);
    float *red_sum = red_max + kWarps * G;
    float *mst = reinterpret_cast<float *>(smem + S::OFF_STAT);
    float *lst = mst + G;
    float *cfac = lst + G;
    float *fac = cfac + G;                                              // [C][G]
    float *xnew = reinterpret_cast<float *>(smem + S::OFF_NEW);        // [2][MC][DSUB]
    int *newc = reinterpret_cast<int *>(xnew + 2 * MC * DSUB);          // [2][M]
    float *snew = reinterpret_cast<float *>(newc + 2 * M);              // [G]
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(
        smem + ((S::OFF_NEW + 2 * MC * DSUB * 4 + 2 * M * 4 + G * 4 + 7) / 8 * 8));
    uint8_t *codes_s = smem + S::OFF_CODES;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int rank = 0;
    if constexpr (C > 1) rank = static_cast<int>(cluster_ctarank());
    const int split = blockIdx.x / C;
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int Hq = p.num_q_heads, Hkv = p.num_kv_heads;
    const int S_ = p.num_splits;

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
        sflag[0] = 0;
    }
    // ---- codebook set and the K slice first: the only reads allowed before
    // the preceding kernel on the stream completes (programmatic dependent
    // launch): codebooks and req_set are not written by it ------------------
    const int share = p.share;
    const int ts = split * p.split_len;
    const int a0 = ts + rank * share;
    const int g = tid % G, jslot = tid / G;
    const int32_t *bt = p.block_table + static_cast<size_t>(b) * p.max_pages;
    const int set = __ldg(p.req_set + b);
    const bool set_ok = set >= 0 && static_cast<int64_t>(set) < p.num_sets;
    const size_t cb_unit = static_cast<size_t>(M) * K * DSUB;
    const __half *gK = reinterpret_cast<const __half *>(p.codebooks) +
                       ((static_cast<size_t>(set_ok ? set : 0) * Hkv + kvh) * 2) * cb_unit +
                       static_cast<size_t>(rank) * S::CB_HALVES;
    const __half *gV = gK + cb_unit;
    uint64_t pol = 0;
    if (warp == 0) __syncwarp();
    auto issue_k_slice = [&]() {
        if (warp == 0 && lane == 0 && set_ok) {
            pol = policy_evict_first();
            mbar_arrive_expect_tx(&bar[0], S::CB_BYTES);
            bulk_g2s_hint(cbk, gK, S::CB_BYTES, &bar[0], pol);
        }
    };
    // overlapped with the preceding kernel, the slice goes first; otherwise it
    // goes after the length and page-id loads, which it would delay
    if (p.overlap) issue_k_slice();
    grid_dependency_wait();

    // ---- length and page ids ----------------------------------------------
    const int L_raw = __ldg(p.seq_lens + b);
    int pgw[S::PPL];
    if (warp == 0) {
        const int np_lim = min(share / P, p.max_pages - a0 / P);
#pragma unroll
        for (int j = 0; j < S::PPL; ++j) {
            const int idx = lane + 32 * j;
            pgw[j] = idx < np_lim ? __ldg(bt + a0 / P + idx) : -1;
        }
    }
    // the new token's owned K and V sub-vector elements, one per thread
    __half xreg = __float2half(0.f);
    if constexpr (APPEND) {
        if (tid < 2 * MC * DSUB) {
            const int w = tid / (MC * DSUB), r = tid % (MC * DSUB);
            xreg = __ldg(reinterpret_cast<const __half *>(p.kv_new) +
                         ((static_cast<size_t>(b) * Hkv + kvh) * 2 + w) * D + rank * MC * DSUB + r);
        }
    }
    if (!p.overlap) issue_k_slice();

    // ---- request-level checks: uniform over the cluster ------------------
    int bad0 = 0;
    if (L_raw < 0 || L_raw > p.max_pages * P || L_raw > p.max_seq_len) bad0 |= AQ_DEV_BAD_LENGTH;
    if (!set_ok) bad0 |= AQ_DEV_BAD_SET;
    const int te = bad0 ? ts : min(L_raw, ts + p.split_len);
    if (bad0 || ts >= te) {
        // nothing to stream: NaN for a bad request, zeros / empty partials otherwise
        if (rank == 0) {
            if (bad0 && tid == 0) flag_status(p.status, bad0);
            const float v = bad0 ? __int_as_float(0x7fc00000) : 0.0f;
            for (int i = tid; i < G * D; i += kThreads) {
                const int gg = i / D, d = i % D;
                const size_t bh = static_cast<size_t>(b) * Hq + kvh * G + gg;
                if (S_ == 1) p.out[bh * D + d] = v;
                else if (d == 0) {
                    p.part_ml[(bh * S_ + split) * 2 + 0] = bad0 ? v : -INFINITY;
                    p.part_ml[(bh * S_ + split) * 2 + 1] = bad0 ? v : 0.0f;
                }
            }
        }
        if (tid == 0 && set_ok) mbar_wait_bounded(&bar[0], 0);   // the K slice copy lands first
        return;
    }
    const int e0 = min(te, a0 + share);
    // the fused step's new token: position L-1, held by the cluster of its split
    // and streamed by no CTA (it is scored from its fresh codes instead)
    const int new_pos = APPEND ? L_raw - 1 : -1;
    const bool cl_new = APPEND && new_pos >= ts && new_pos < te;
    const bool own_new = cl_new && new_pos >= a0 && new_pos < e0;
    const int eS = own_new ? new_pos : e0;
    const int npg = eS > a0 ? (eS - a0 + P - 1) / P : 0;
    const int pg_new = cl_new ? __ldg(bt + new_pos / P) : -1;   // checked where it is used

    // ---- warp 0 issues the rest: code pages + query, then the V slice ------
    if (warp == 0) {
        bool ok[S::PPL];
        int nvalid = 0, bad = 0;
#pragma unroll
        for (int j = 0; j < S::PPL; ++j) {
            const int idx = lane + 32 * j;
            ok[j] = idx < npg && pgw[j] >= 0 && static_cast<int64_t>(pgw[j]) < p.num_pages;
            bad |= (idx < npg && !ok[j]);
            nvalid += __popc(__ballot_sync(0xffffffffu, ok[j]));
        }
        if (bad) atomicOr(&sflag[0], AQ_DEV_BAD_PAGE);
        if (lane == 0) mbar_arrive_expect_tx(&bar[4], nvalid * S::PAGE_BYTES + G * D * 4);
        __syncwarp();
#pragma unroll
        for (int j = 0; j < S::PPL; ++j) {
            if (ok[j]) {
                const int idx = lane + 32 * j;
                bulk_g2s(codes_s + idx * S::PAGE_BYTES,
                         p.code_pages + (static_cast<size_t>(pgw[j]) * Hkv + kvh) * S::PAGE_BYTES,
                         S::PAGE_BYTES, &bar[4]);
            }
        }
        if (lane == 0) {
            bulk_g2s(qs, p.q + (static_cast<size_t>(b) * Hq + static_cast<size_t>(kvh) * G) * D, G * D * 4,
                     &bar[4]);
            mbar_arrive_expect_tx(&bar[1], S::CB_BYTES);
            bulk_g2s_hint(cbv, gV, S::CB_BYTES, &bar[1], pol);
            if constexpr (C > 1) {
                mbar_arrive_expect_tx(&bar[2], (C - 1) * (S::ROW_FLOATS + (cl_new ? MC : 0)) * 4);
                mbar_arrive_expect_tx(&bar[3], (C - 1) * (S::ROW_FLOATS + S::STAT_FLOATS) * 4);
            }
        }
    }
    for (int i = tid; i < S::LUT_FLOATS / 4; i += kThreads)
        reinterpret_cast<float4 *>(bins)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < G) snew[tid] = -INFINITY;
    if (cl_new && tid < 2 * MC * DSUB) xnew[tid] = __half2float(xreg);
    grid_launch_dependents();                          // every read of this CTA is issued
    if constexpr (C > 1) {
        cluster_arrive_relaxed();          // peers' mbarriers exist before anyone pushes
        cluster_wait_acquire();
    } else {
        __syncthreads();
    }

    // ---- lookup-table rows of the owned subspaces, pushed to the peers ------
    if (!mbar_wait_bounded(&bar[0], 0)) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
    if (!mbar_wait_bounded(&bar[4], 0)) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
    constexpr int NCH = DSUB / 8;                       // 16-byte chunks per codeword row
    // per-thread chunk order: lanes of a quarter-warp read distinct banks
    const int rot = (tid / (128 / (DSUB * 2))) % NCH;
    {
        // thread tid = codeword k: its row is read once into registers and
        // gives the G table entries and (fused step) its distance to the new
        // key's sub-vector
#pragma unroll
        for (int mi = 0; mi < MC; ++mi) {
            const int m = rank * MC + mi;
            uint4 u[NCH];
            load_row_rotated<NCH>(u, cbk + (static_cast<size_t>(mi) * K + tid) * DSUB, rot);
            float acc[G];
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int c0 = 0; c0 < NCH; ++c0) {
                    const int c = (c0 + rot) % NCH;
                    const float2 f0 = h2_to_f2(u[c0].x), f1 = h2_to_f2(u[c0].y), f2 = h2_to_f2(u[c0].z),
                                 f3 = h2_to_f2(u[c0].w);
                    const float4 *qv = reinterpret_cast<const float4 *>(qs + gg * D + m * DSUB + c * 8);
                    const float4 qa = qv[0], qb = qv[1];
                    a0 = fmaf(qa.x, f0.x, a0); a1 = fmaf(qb.x, f2.x, a1);
                    a0 = fmaf(qa.y, f0.y, a0); a1 = fmaf(qb.y, f2.y, a1);
                    a0 = fmaf(qa.z, f1.x, a0); a1 = fmaf(qb.z, f3.x, a1);
                    a0 = fmaf(qa.w, f1.y, a0); a1 = fmaf(qb.w, f3.y, a1);
                }
                acc[gg] = (a0 + a1) * p.scale_log2;
            }
            float *dst = lut + (static_cast<size_t>(m) * K + tid) * G;
            store_vec<G>(dst, acc);
            if constexpr (C > 1) {
                const uint32_t la = smem_u32(dst), lb = smem_u32(&bar[2]);
#pragma unroll
                for (int r = 1; r < C; ++r) {
                    const uint32_t pr = (rank + r) % C;
                    push_vec<G>(mapa_u32(la, pr), acc, mapa_u32(lb, pr));
                }
            }
            if constexpr (APPEND) {
                if (cl_new) {                          // K code of the new token in subspace m
                    const int code = block_argmin(row_distance<NCH>(u, xnew + mi * DSUB, rot), keys);
                    if (tid == 0) {
                        newc[m] = code;
                        if constexpr (C > 1) {
                            const uint32_t la = smem_u32(&newc[m]), lb = smem_u32(&bar[2]);
#pragma unroll
                            for (int r = 1; r < C; ++r) {
                                const uint32_t pr = (rank + r) % C;
                                st_async_f32(mapa_u32(la, pr), __int_as_float(code), mapa_u32(lb, pr));
                            }
                        }
                    }
                }
            }
        }
    }
    if constexpr (C > 1) {
        if (!mbar_wait_bounded(&bar[2], 0)) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
    }
    __syncthreads();

    // ---- code stream: scores, softmax statistics, value bins -------------------
    // Three passes over the share: (1) scores by M table gathers and the per-head
    // max, (2) per-head sum of exp2(s - max), (3) scatter of each weight into the
    // 256-bin value accumulators as the unsigned fixed-point integer
    // floor(p 2^32 (1 - 2^-16) / l): the bins cannot overflow (the margin covers
    // the rounding of the float sum), integer shared-memory atomics are exact
    // and fast, and the result does not depend on their order.  The first
    // chunk's codes and scores stay in registers, so (2) and (3) read shared
    // memory only for the atomics (a share is one chunk whenever G = 1).  The
    // fused step's new token enters (1) and (2) from its fresh codes; its value
    // bin is added after the merge, once its V code is known.
    unsigned *ibins = reinterpret_cast<unsigned *>(bins);
    auto gather = [&](const Codes<M> &cd) -> float {
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < M; ++m) acc += lut[(m * K + cd.k(m)) * G + g];
        return acc;
    };
    float s_new = -INFINITY;
    if constexpr (APPEND) {
        if (own_new && tid < G) {
            s_new = 0.f;
#pragma unroll
            for (int m = 0; m < M; ++m) s_new += lut[(m * K + newc[m]) * G + tid];
            snew[tid] = s_new;
        }
    }
    Codes<M> cc[TPT];
    float sc[TPT];
    float mx = s_new;
#pragma unroll 1
    for (int cb = a0; cb < eS; cb += S::CHUNK) {
#pragma unroll
        for (int i = 0; i < TPT; ++i) {
            const int t = cb + i * S::TOK_PER_PASS + jslot;
            if (t < eS) {
                Codes<M> cd;
                cd.load(codes_s + (t - a0) * (2 * M));
                const float s = gather(cd);
                if (cb == a0) { cc[i] = cd; sc[i] = s; }
                mx = fmaxf(mx, s);
            }
        }
    }
#pragma unroll
    for (int off = G; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane < G) red_max[warp * G + lane] = mx;
    __syncthreads();
    mx = red_max[g];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, red_max[w * G + g]);
    float l_run = (s_new != -INFINITY) ? exp2f(s_new - mx) : 0.f;
    if (mx != -INFINITY) {
#pragma unroll 1
        for (int cb = a0; cb < eS; cb += S::CHUNK) {
#pragma unroll
            for (int i = 0; i < TPT; ++i) {
                const int t = cb + i * S::TOK_PER_PASS + jslot;
                if (t < eS) {
                    float s;
                    if (cb == a0) {
                        s = sc[i];
                    } else {
                        Codes<M> cd;
                        cd.load(codes_s + (t - a0) * (2 * M));
                        s = gather(cd);
                    }
                    l_run += exp2f(s - mx);
                }
            }
        }
    }
#pragma unroll
    for (int off = G; off < 32; off <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
    if (lane < G) red_sum[warp * G + lane] = l_run;
    __syncthreads();
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) lsum += red_sum[w * G + g];
    const float qscale = lsum > 0.f ? 4294901760.0f / lsum : 0.f;
    if (mx != -INFINITY) {
#pragma unroll 1
        for (int cb = a0; cb < eS; cb += S::CHUNK) {
#pragma unroll
            for (int i = 0; i < TPT; ++i) {
                const int t = cb + i * S::TOK_PER_PASS + jslot;
                if (t < eS) {
                    Codes<M> cd;
                    float s;
                    if (cb == a0) {
                        cd = cc[i];
                        s = sc[i];
                    } else {
                        cd.load(codes_s + (t - a0) * (2 * M));
                        s = gather(cd);
                    }
                    const unsigned q = __float2uint_rz(exp2f(s - mx) * qscale);
#pragma unroll
                    for (int m = 0; m < M; ++m) atomicAdd(&ibins[(m * K + cd.vv(m)) * G + g], q);
                }
            }
        }
    }
    if (tid < G) {
        mst[tid] = mx;                                 // this CTA's statistics for now
        lst[tid] = lsum;
        cfac[tid] = qscale > 0.f ? 1.0f / qscale : 0.f;  // integer bin -> weight
    }
    __syncthreads();

    // ---- push bins rows (as weights) and statistics to the peers that own them
    if constexpr (C > 1) {
        const uint32_t lb = smem_u32(&bar[3]);
#pragma unroll 1
        for (int r = 1; r < C; ++r) {
            const uint32_t pr = (rank + r) % C;
            const int slot = (C - r - 1) % C;          // (rank - pr - 1) mod C
            const uint32_t rslot = mapa_u32(smem_u32(inc + slot * S::INC_STRIDE), pr);
            const uint32_t rbar = mapa_u32(lb, pr);
            const uint4 *src = reinterpret_cast<const uint4 *>(ibins + pr * S::ROW_FLOATS);
            for (int i = tid; i < S::ROW_FLOATS / 4; i += kThreads) {
                const uint4 v = src[i];
                const int g0 = (4 * i) % G;
                st_async_v4(rslot + 16 * i,
                            make_float4(static_cast<float>(v.x) * cfac[g0], static_cast<float>(v.y) * cfac[(g0 + 1) % G],
                                        static_cast<float>(v.z) * cfac[(g0 + 2) % G],
                                        static_cast<float>(v.w) * cfac[(g0 + 3) % G]),
                            rbar);
            }
            if (tid < G) {
                st_async_f32(rslot + 4 * (S::ROW_FLOATS + tid), mst[tid], rbar);
                st_async_f32(rslot + 4 * (S::ROW_FLOATS + G + tid), lst[tid], rbar);
                st_async_f32(rslot + 4 * (S::ROW_FLOATS + 2 * G + tid), snew[tid], rbar);
            }
            if (tid == 0) st_async_f32(rslot + 4 * (S::ROW_FLOATS + 3 * G), __int_as_float(sflag[0]), rbar);
        }
        if (!mbar_wait_bounded(&bar[3], 0)) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
        cluster_arrive_relaxed();                      // all traffic into this CTA has landed
    }

    // ---- merge statistics, then the owned rows of the value bins ------------
    if (tid < G) {
        float mr[C], lr[C];
        float ms = -INFINITY, sn = snew[tid];
#pragma unroll
        for (int r = 0; r < C; ++r) {
            if (r == rank) { mr[r] = mst[tid]; lr[r] = lst[tid]; }
            else {
                const float *sl = inc + ((r - rank - 1 + C) % C) * S::INC_STRIDE;
                mr[r] = sl[S::ROW_FLOATS + tid];
                lr[r] = sl[S::ROW_FLOATS + G + tid];
                sn = fmaxf(sn, sl[S::ROW_FLOATS + 2 * G + tid]);
            }
            if (lr[r] > 0.f) ms = fmaxf(ms, mr[r]);
        }
        float ls = 0.f;
#pragma unroll
        for (int r = 0; r < C; ++r) {
            const float f = (lr[r] > 0.f) ? exp2f(mr[r] - ms) : 0.f;
            fac[r * G + tid] = f;
            ls += f * lr[r];
        }
        fac[rank * G + tid] *= cfac[tid];              // own rows are still integers
        mst[tid] = ms;
        lst[tid] = ls;
        snew[tid] = sn;
    }
    if (tid == 0) {
        int bb = sflag[0];
#pragma unroll
        for (int r = 0; r < C; ++r)
            if (r != rank)
                bb |= __float_as_int(inc[((r - rank - 1 + C) % C) * S::INC_STRIDE + S::ROW_FLOATS + 3 * G]);
        sflag[1] = bb;
        if (sflag[0]) flag_status(p.status, sflag[0]);
    }
    __syncthreads();
    int bad_all = sflag[1];
    float *wtot = lut;                                 // [MC][K][G]; the LUT is no longer read
    {
        constexpr int N4 = S::ROW_FLOATS / 4;
        const uint4 *own = reinterpret_cast<const uint4 *>(ibins + rank * S::ROW_FLOATS);
        for (int i = tid; i < N4; i += kThreads) {
            const int g0 = (4 * i) % G;
            const uint4 o = own[i];
            float4 acc = make_float4(fac[rank * G + g0] * static_cast<float>(o.x),
                                     fac[rank * G + (g0 + 1) % G] * static_cast<float>(o.y),
                                     fac[rank * G + (g0 + 2) % G] * static_cast<float>(o.z),
                                     fac[rank * G + (g0 + 3) % G] * static_cast<float>(o.w));
#pragma unroll
            for (int r = 0; r < C; ++r) {
                if (r == rank) continue;
                const float4 v = reinterpret_cast<const float4 *>(inc + ((r - rank - 1 + C) % C) * S::INC_STRIDE)[i];
                acc.x += fac[r * G + g0] * v.x;
                acc.y += fac[r * G + (g0 + 1) % G] * v.y;
                acc.z += fac[r * G + (g0 + 2) % G] * v.z;
                acc.w += fac[r * G + (g0 + 3) % G] * v.w;
            }
            reinterpret_cast<float4 *>(wtot)[i] = acc;
        }
    }
    __syncthreads();

    // ---- value codebook product for the owned subspaces -----------------------
    if (!mbar_wait_bounded(&bar[1], 0)) {
        atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
        bad_all |= AQ_DEV_TIMEOUT;
    }
    if constexpr (APPEND) {
        if (cl_new) {                                  // V codes of the new token, its value bins
#pragma unroll 1
            for (int mi = 0; mi < MC; ++mi) {
                uint4 u[NCH];
                load_row_rotated<NCH>(u, cbv + (static_cast<size_t>(mi) * K + tid) * DSUB, rot);
                const int code = block_argmin(row_distance<NCH>(u, xnew + (MC + mi) * DSUB, rot), keys);
                if (tid < G && snew[tid] != -INFINITY)
                    wtot[(static_cast<size_t>(mi) * K + code) * G + tid] += exp2f(snew[tid] - mst[tid]);
                if (tid == 0) newc[M + rank * MC + mi] = code;
            }
            const bool pg_ok = pg_new >= 0 && static_cast<int64_t>(pg_new) < p.num_pages;
            if (tid == 0 && !pg_ok) flag_status(p.status, AQ_DEV_BAD_PAGE);
            if (!pg_ok) bad_all |= AQ_DEV_BAD_PAGE;
            if (tid == 0 && pg_ok) {                   // the new token's codes into its page slot
                uint8_t *dst = p.code_pages_w +
                               ((static_cast<size_t>(pg_new) * Hkv + kvh) * P + new_pos % P) * (2 * M);
#pragma unroll
                for (int mi = 0; mi < MC; ++mi) {
                    dst[rank * MC + mi] = static_cast<uint8_t>(newc[rank * MC + mi]);
                    dst[M + rank * MC + mi] = static_cast<uint8_t>(newc[M + rank * MC + mi]);
                }
            }
            __syncthreads();
        }
    }
    // thread = (k slice, 4-dim quad of the owned dims): 8-byte codebook loads,
    // the slices of a warp reduced by shuffles, the warps through shared memory
    float *ored = reinterpret_cast<float *>(cbk);      // [kWarps][MC*DSUB][G]
    {
        constexpr int NQ = MC * DSUB / 4, KSQ = kThreads / NQ, KSLQ = K / KSQ;
        const int qd = tid % NQ, ks = tid / NQ;
        const int mi = qd / (DSUB / 4), j4 = (qd % (DSUB / 4)) * 4;
        float acc[G][4];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) acc[gg][0] = acc[gg][1] = acc[gg][2] = acc[gg][3] = 0.f;
#pragma unroll 4
        for (int i = 0; i < KSLQ; ++i) {
            const int k = ks * KSLQ + ((i + ks) % KSLQ);
            const uint2 cv2 = *reinterpret_cast<const uint2 *>(cbv + (static_cast<size_t>(mi) * K + k) * DSUB + j4);
            const float2 c01 = h2_to_f2(cv2.x), c23 = h2_to_f2(cv2.y);
            float w[G];
            load_vec<G>(w, wtot + (static_cast<size_t>(mi) * K + k) * G);
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                acc[gg][0] = fmaf(w[gg], c01.x, acc[gg][0]);
                acc[gg][1] = fmaf(w[gg], c01.y, acc[gg][1]);
                acc[gg][2] = fmaf(w[gg], c23.x, acc[gg][2]);
                acc[gg][3] = fmaf(w[gg], c23.y, acc[gg][3]);
            }
        }
#pragma unroll
        for (int off = NQ; off < 32; off <<= 1) {
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[gg][e] += __shfl_xor_sync(0xffffffffu, acc[gg][e], off);
        }
        if (lane < NQ) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v[G];
#pragma unroll
                for (int gg = 0; gg < G; ++gg) v[gg] = acc[gg][e];
                store_vec<G>(ored + (static_cast<size_t>(warp) * MC * DSUB + mi * DSUB + j4 + e) * G, v);
            }
        }
    }
    __syncthreads();
    {
        constexpr int NOUT = MC * DSUB * G;
        for (int i = tid; i < NOUT; i += kThreads) {
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) o += ored[static_cast<size_t>(w) * NOUT + i];
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
    // A wait that ran out may leave a copy or a push still landing: wait again
    // (bounded) before the shared memory is released.
    if (sflag[0] & AQ_DEV_TIMEOUT) {
        mbar_wait_bounded(&bar[0], 0);
        mbar_wait_bounded(&bar[1], 0);
        mbar_wait_bounded(&bar[4], 0);
        if constexpr (C > 1) {
            mbar_wait_bounded(&bar[2], 0);
            mbar_wait_bounded(&bar[3], 0);
        }
    }
    if constexpr (C > 1) cluster_wait_acquire();      // no CTA leaves while a peer may push to it
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

template <int M, int G, int C, bool APPEND>
cudaError_t launch_one(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    using S = PqCfg<M, G, C>;
    auto kern = pq_decode_kernel<M, G, C, APPEND>;
    if (plan.share > kMaxShare || plan.share % kPage) return cudaErrorInvalidValue;
    static size_t attr_bytes = 0;                  // opt-in dynamic shared memory set so far
    const size_t need = S::smem(plan.share);
    if (need > attr_bytes) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(need));
        if (e != cudaSuccess) return e;
        attr_bytes = need;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C * plan.num_splits), static_cast<unsigned>(p.num_kv_heads),
                       static_cast<unsigned>(p.batch));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = need;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.overlap ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int M, int G, bool APPEND>
cudaError_t dispatch_c(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    switch (plan.cluster) {
        case 1: return launch_one<M, G, 1, APPEND>(p, plan, s);
        case 2: return launch_one<M, G, 2, APPEND>(p, plan, s);
        case 4: return launch_one<M, G, 4, APPEND>(p, plan, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

template <int M, bool APPEND>
cudaError_t dispatch_g(const DecodeParams &p, int G, const Plan &plan, cudaStream_t s) {
    switch (G) {
        case 1: return dispatch_c<M, 1, APPEND>(p, plan, s);
        case 2: return dispatch_c<M, 2, APPEND>(p, plan, s);
        case 4: return dispatch_c<M, 4, APPEND>(p, plan, s);
        case 8: return dispatch_c<M, 8, APPEND>(p, plan, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

template <int M>
size_t smem_g(int G, int C, int share) {
#define AQ_SM(GG, CC) \
    if (G == GG && C == CC) return PqCfg<M, GG, CC>::smem(share);
    AQ_SM(1, 1) AQ_SM(1, 2) AQ_SM(1, 4)
    AQ_SM(2, 1) AQ_SM(2, 2) AQ_SM(2, 4)
    AQ_SM(4, 1) AQ_SM(4, 2) AQ_SM(4, 4)
    AQ_SM(8, 1) AQ_SM(8, 2) AQ_SM(8, 4)
#undef AQ_SM
    return 0;
}

}  // namespace

size_t pq_decode_smem_bytes(int M, int G, int cluster, int share) {
    if (M == 4) return smem_g<4>(G, cluster, share);
    if (M == 8) return smem_g<8>(G, cluster, share);
    return 0;
}

cudaError_t launch_pq_decode(const DecodeParams &p, int M, int G, const Plan &plan, cudaStream_t s) {
    cudaError_t e;
    if (M == 4) e = dispatch_g<4, false>(p, G, plan, s);
    else if (M == 8) e = dispatch_g<8, false>(p, G, plan, s);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    if (plan.num_splits > 1) return launch_combine(p, s);
    return cudaSuccess;
}

cudaError_t launch_pq_decode_step(const DecodeParams &p, int M, int G, const Plan &plan, cudaStream_t s) {
    cudaError_t e;
    if (M == 4) e = dispatch_g<4, true>(p, G, plan, s);
    else if (M == 8) e = dispatch_g<8, true>(p, G, plan, s);
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
