// decode_pq.cu -- fused PQ decode attention for sm_103a.
//
// One thread-block cluster of C CTAs handles one (request b, kv head, split).
// CTA `rank` owns subspaces [rank*M/C, (rank+1)*M/C) of both the key and the
// value codebook and 1/C of the split's tokens:
//
//  1. copy its key and value codebook slices (64/C KiB each) into shared
//     memory with cp.async, each codeword row's 16-byte chunks at XOR-swizzled
//     positions so that rows read in their natural order are bank-conflict
//     free; load its tokens' uint8 codes straight into registers (page ids
//     from the block table, PAM article §2.2.2) and the G query vectors of
//     the GQA group;
//  2. LUT[m][k][g] = <q_g[m], C^K_m[k]> * scale * log2(e) for its own m
//     (AQPIM blog §4.1: per-subspace partial dot products with the codebook;
//     §5.1 item 3: index -> codebook -> sub-dot -> accumulate, nothing
//     intermediate written to global memory); the rows are exchanged through
//     distributed shared memory so every CTA holds the full M x 256 x G table;
//  3. score its tokens, s = sum_m LUT[m][kcode_m] by table gathers, reduce the
//     per-head (max, sum) of the block (online softmax statistics, PAM article
//     §2.2.3 item 1) and scatter exp2(s - max) into 256-bin value
//     accumulators W[m][vcode_m][g];
//  4. merge the C CTAs' (max, sum, bins) over distributed shared memory (the
//     hierarchical reduction of PAM article §2.2.3 item 3, inside one cluster)
//     and apply the value codebook slice it owns: o[m*Dsub+j] = sum_k W[m][k]
//     * C^V_m[k][j];
//  5. normalise and store, or store (max, sum, o) partials for the split-KV
//     combine kernel.
//
// The fused decode step (APPEND) also encodes the token at position
// seq_len-1 of every request in step 2 (each CTA its owned subspaces, from the
// codebook rows it already holds in registers), scores it from its fresh
// codes, adds it to the value bins after the merge and writes its codes to
// its page slot.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace aq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int M, int G, int C>
struct PqCfg {
    static constexpr int D = kHeadDim, K = kCodewords, P = kPage;
    static constexpr int DSUB = D / M;
    static constexpr int NCH = DSUB / 8;                    // 16-byte chunks per codeword row
    static constexpr int MC = M / C;                        // subspaces owned per CTA
    static constexpr int CB_HALVES = MC * K * DSUB;         // owned part of one codebook
    static constexpr int CB_BYTES = CB_HALVES * 2;
    static constexpr int CB_CHUNKS = CB_BYTES / 16;
    static constexpr int LUT_FLOATS = M * K * G;
    static constexpr int BIN_WORDS = LUT_FLOATS;            // u32 value bins [M][K][G]
    static constexpr int ROW_FLOATS = MC * K * G;           // one rank's rows of LUT / bins
    static constexpr int TOK_PER_PASS = kThreads / G;
    // tokens per thread, held in registers (codes and scores)
    static constexpr int TPT = (M == 8 && G <= 2) ? 4 : 8;
    static constexpr int MAX_SHARE = TPT * TOK_PER_PASS;    // tokens per CTA
    // statistics pushed with the bins: m[G], l[G], new-token score[G], the
    // scale of the (integer) bins of each head [G], bad flag
    static constexpr int STAT_FLOATS = 4 * G + 1;
    static constexpr int INC_STRIDE = ROW_FLOATS + (STAT_FLOATS + 3) / 4 * 4;
    static constexpr int NKEY = 2 * MC;
    // value product: the k-slice order of subspace mi is XOR-ed with mi * VP_XOR,
    // so that the rows one half-warp reads (several subspaces, neighbouring
    // k-slices) fall in distinct 32- or 64-byte parts of their lines
    static constexpr int VP_XOR = (M == 8 && C == 4) ? 2 : 1;                     // new-token argmins: K then V, owned subspaces
    // shared-memory layout (bytes), the codebook slices first: TMA copies them
    // with the hardware swizzle when the dynamic shared memory starts on a
    // 1024-byte boundary.  With clusters of 4 (4 resident CTAs per SM either
    // way) one buffer each, both slices issued at the start; with fewer CTAs
    // per cluster (larger slices) one buffer holds the K slice until the table
    // build and the new key's encode are done, then the V slice
    static constexpr bool SHARED_CB = C < 4;
    static constexpr int OFF_CB = 0;
    static constexpr int OFF_CBV = OFF_CB + (SHARED_CB ? 0 : CB_BYTES);
    static constexpr int OFF_LUT = OFF_CBV + CB_BYTES;
    static constexpr int OFF_BINS = OFF_LUT + LUT_FLOATS * 4;
    // [C-1][INC_STRIDE] from the peers; sender src lands in slot (src - dst - 1) mod C
    static constexpr int OFF_INC = OFF_BINS + BIN_WORDS * 4;
    static constexpr int OFF_Q = OFF_INC + (C > 1 ? (C - 1) * INC_STRIDE * 4 : 0);
    static constexpr int OFF_RED = OFF_Q + G * D * 4;       // red_m, red_l [kWarps][G], twice (streamed shares)
    static constexpr int OFF_STAT = OFF_RED + 4 * kWarps * G * 4;  // merged mst, lst [G]
    // new token: owned sub-vectors [2][MC][DSUB] f32, codes [2][M] int, score [G]
    static constexpr int OFF_NEW = (OFF_STAT + 2 * G * 4 + 15) / 16 * 16;
    static constexpr int OFF_KEYS = (OFF_NEW + 2 * MC * DSUB * 4 + 2 * M * 4 + G * 4 + 7) / 8 * 8;
    static constexpr int OFF_BAR = OFF_KEYS + NKEY * 8;     // 5 mbarriers
    static constexpr int OFF_MISC = OFF_BAR + 5 * 8;        // int flags
    static constexpr int END = OFF_MISC + 16;
    static size_t smem() { return END; }
    static_assert(CB_BYTES % 1024 == 0, "slices keep the swizzle alignment");
    static_assert(K == kThreads, "one thread per codeword in the table build");
    static_assert(CB_CHUNKS % kThreads == 0, "whole slice chunks per thread");
    static_assert((NCH & (NCH - 1)) == 0 && NCH <= 8, "XOR swizzle over a power-of-two chunk count");
    static_assert((MC * DSUB / 4) <= 32 && 32 % (MC * DSUB / 4) == 0, "V-product quads within a warp");
    // V-product partials: in the peers' rows once merged (this CTA's own bins may
    // still be in flight to its peers), or in the bins without peers
    static_assert(C > 1 ? kWarps * MC * DSUB * G <= (C - 1) * INC_STRIDE : kWarps * MC * DSUB * G <= BIN_WORDS,
                  "V-product reduction space");
    static_assert(CB_BYTES % 16 == 0 && OFF_LUT % 16 == 0 && OFF_INC % 16 == 0 && OFF_Q % 16 == 0,
                  "alignment");
    static_assert(ROW_FLOATS % 4 == 0 && INC_STRIDE % 4 == 0, "bulk copies of whole rows");
};

constexpr int kMaxChunks = kMaxStreamChunks;

// CTAs per SM the register budget is sized for: shared memory (LUT, bins and
// pushed rows all scale with G) allows about 4 / 2 / 1 resident CTAs.
template <int G, int C>
constexpr int kMinBlocks = G <= 2 ? (C == 2 ? 5 : 4) : (G == 4 ? 2 : 1);

// Position of 16-byte chunk c of codeword row k in shared memory: c XOR a
// function of k, so that the 8 rows a quarter-warp reads at once (two or four
// rows per 128-byte line) cover all eight 16-byte bank groups.
template <int DSUB>
__device__ __forceinline__ int chunk_pos(int k, int c) {
    constexpr int NCH = DSUB / 8, ROWS128 = 128 / (DSUB * 2);
    return c ^ ((k / ROWS128) & (NCH - 1));
}

// Copy an owned codebook slice [rows][DSUB] fp16 to shared memory in the
// swizzled layout: thread tid takes chunks tid, tid + kThreads, ... (coalesced
// global reads) and arrives on `bar` once its copies have landed.
template <int DSUB, int CHUNKS>
__device__ __forceinline__ void copy_slice(__half *dst, const __half *src, uint64_t *bar) {
    constexpr int NCH = DSUB / 8, ROWS128 = 128 / (DSUB * 2);
    // chunk tid + i*kThreads lies kThreads/NCH rows below chunk tid, a multiple
    // of the swizzle period, so it keeps chunk tid's position within its row
    static_assert((kThreads / NCH) % (ROWS128 * NCH) == 0, "swizzle period");
    const int t = static_cast<int>(threadIdx.x);
    const int r0 = t / NCH, c = t % NCH;
    const uint32_t d0 = smem_u32(dst) + static_cast<uint32_t>(r0 * NCH + chunk_pos<DSUB>(r0, c)) * 16u;
    const __half *s0 = src + static_cast<size_t>(t) * 8;
#pragma unroll
    for (int i = 0; i < CHUNKS / kThreads; ++i)
        cp_async_16(d0 + static_cast<uint32_t>(i * kThreads * 16), s0 + static_cast<size_t>(i) * kThreads * 8);
    cp_async_mbar_arrive(bar);
}

// Eight fp16 values (one 16-byte chunk) as four packed fp32 pairs.
__device__ __forceinline__ void to_f2p4(const uint4 &u, unsigned long long (&f)[4]) {
    f[0] = h2_to_f2p(u.x);
    f[1] = h2_to_f2p(u.y);
    f[2] = h2_to_f2p(u.z);
    f[3] = h2_to_f2p(u.w);
}

// Raw E4M3 slices (one byte per element, rows of DSUB bytes): 16-byte chunk e
// of row k sits at e ^ ((k / 4) & 1) when rows are 32 bytes (the 32-byte TMA
// swizzle: rows k..k+7 read at once cover every bank group), in place when
// they are 16 bytes (one chunk).
template <int DSUB>
__device__ __forceinline__ int e8_pos(int k, int e) {
    if constexpr (DSUB == 32) return e ^ ((k >> 2) & 1);
    else return e;
}

// 8 E4M3 values (two 32-bit words, first value in the lowest byte) as four
// packed fp32 pairs: widened exactly through fp16.
__device__ __forceinline__ void e4m3x8_to_f2p4(uint32_t lo, uint32_t hi, unsigned long long (&f)[4]) {
    const uint32_t w[4] = {lo & 0xffffu, lo >> 16, hi & 0xffffu, hi >> 16};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[j]), __NV_E4M3);
        f[j] = h2_to_f2p(static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16));
    }
}

// Calls fn(c, f) for the 8-element chunks c = 0 .. DSUB/8-1 of codeword row
// `row` of a slice, f = its values as four packed fp32 pairs (in order): fp16
// slices in the swizzled chunk layout, or raw E4M3 slices (two chunks per
// 16-byte load).
template <int DSUB, bool E4M3, typename F>
__device__ __forceinline__ void for_row_chunks(const void *slice, int row, F &&fn) {
    if constexpr (!E4M3) {
        constexpr int NCH = DSUB / 8;
        const uint4 *r = reinterpret_cast<const uint4 *>(slice) + row * NCH;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            unsigned long long f[4];
            to_f2p4(r[chunk_pos<DSUB>(row, c)], f);
            fn(c, f);
        }
    } else {
        constexpr int NE = DSUB / 16;
        const uint4 *r = reinterpret_cast<const uint4 *>(static_cast<const unsigned char *>(slice) + row * DSUB);
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            const uint4 u = r[e8_pos<DSUB>(row, e)];
            unsigned long long f[4];
            e4m3x8_to_f2p4(u.x, u.y, f);
            fn(2 * e, f);
            e4m3x8_to_f2p4(u.z, u.w, f);
            fn(2 * e + 1, f);
        }
    }
}

// A raw E4M3 slice [rows][DSUB] bytes by per-thread 16-byte cp.async copies
// into the e8_pos layout (the TMA copy's fallback); one arrival per thread.
template <int DSUB, int ROWS>
__device__ __forceinline__ void copy_slice_e4m3_raw(unsigned char *dst, const uint8_t *src, uint64_t *bar) {
    constexpr int NE = DSUB / 16, CHUNKS = ROWS * NE;
    for (int q = static_cast<int>(threadIdx.x); q < CHUNKS; q += kThreads) {
        const int row = q / NE, e = q % NE;
        cp_async_16(smem_u32(dst + row * DSUB + e8_pos<DSUB>(row, e) * 16), src + static_cast<size_t>(q) * 16);
    }
    cp_async_mbar_arrive(bar);
}

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

template <int N>
__device__ __forceinline__ void load_vec_u(unsigned (&v)[N], const unsigned *src) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            uint4 t = *reinterpret_cast<const uint4 *>(src + i);
            v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
        }
    } else if constexpr (N == 2) {
        uint2 t = *reinterpret_cast<const uint2 *>(src);
        v[0] = t.x; v[1] = t.y;
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] = src[i];
    }
}

// A compile-time int as a value (slot index of a generic lambda).
template <int N>
struct IntC {
    static constexpr int value = N;
};

// Code bytes of one token: M key codes then M value codes.
template <int M>
struct Codes;
template <>
struct Codes<4> {
    uint2 v;
    __device__ __forceinline__ void load_global(const uint8_t *p) { v = ld_global_na_v2(p); }
    __device__ __forceinline__ void load_shared(const unsigned char *p) { v = *reinterpret_cast<const uint2 *>(p); }
    __device__ __forceinline__ int k(int m) const { return static_cast<int>(__byte_perm(v.x, 0u, 0x4440u | m)); }
    __device__ __forceinline__ int vv(int m) const { return static_cast<int>(__byte_perm(v.y, 0u, 0x4440u | m)); }
};
template <>
struct Codes<8> {
    uint4 v;
    __device__ __forceinline__ void load_global(const uint8_t *p) { v = ld_global_na_v4(p); }
    __device__ __forceinline__ void load_shared(const unsigned char *p) { v = *reinterpret_cast<const uint4 *>(p); }
    __device__ __forceinline__ int k(int m) const {
        return static_cast<int>(__byte_perm(m < 4 ? v.x : v.y, 0u, 0x4440u | (m & 3)));
    }
    __device__ __forceinline__ int vv(int m) const {
        return static_cast<int>(__byte_perm(m < 4 ? v.z : v.w, 0u, 0x4440u | (m & 3)));
    }
};

// One encode step on 8 consecutive dimensions: fp32 squared distance with
// separately rounded subtract / multiply / add, the adds in increasing
// dimension order (the encode decision rule).  Subtracts and squares run as
// packed pairs (each lane rounded as the scalar operation), the running sum
// stays scalar.  x: the new token's sub-vector chunk; f: the codeword chunk as
// four packed pairs.
__device__ __forceinline__ float sqdist8(float d, const float *x, const unsigned long long (&f)[4]) {
    const ulonglong2 xa = *reinterpret_cast<const ulonglong2 *>(x);
    const ulonglong2 xb = *reinterpret_cast<const ulonglong2 *>(x + 4);
    const unsigned long long xv[4] = {xa.x, xa.y, xb.x, xb.y};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const unsigned long long t = f2_sub(xv[e], f[e]);
        const float2 sq = f2_unpack(f2_mul(t, t));
        d = __fadd_rn(d, sq.x);
        d = __fadd_rn(d, sq.y);
    }
    return d;
}


// CTA-wide argmin, lowest index on ties, of one distance per thread (thread =
// codeword): the warp's smallest distance by an integer min-reduction over the
// bit patterns (distances are >= 0, so they order like their values), its
// lowest lane by a ballot, then one 64-bit (distance, index) atomic minimum per
// warp into `slot`, which holds ~0 beforehand.  The code is slot & 0xff once a
// __syncthreads has passed.
__device__ __forceinline__ void warp_argmin_into(float d, unsigned long long *slot) {
    const unsigned db = __float_as_uint(d);
    const unsigned mn = __reduce_min_sync(0xffffffffu, db);
    const unsigned ball = __ballot_sync(0xffffffffu, db == mn);
    if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(ball) - 1))
        atomicMin(slot, (static_cast<unsigned long long>(mn) << 32) | threadIdx.x);
}

// The new token's value codes of the owned subspaces (thread = codeword):
// exact distances to its value sub-vectors xv [MC][DSUB], argmin into
// keys[0..MC) (visible to all threads after the next barrier).
template <int DSUB, int MC, int K, int NCH, bool E4M3 = false>
__device__ __forceinline__ void encode_new_value(const __half *cbv, const float *xv, unsigned long long *keys) {
    const int tid = threadIdx.x;
    float dv[MC];
#pragma unroll
    for (int mi = 0; mi < MC; ++mi) {
        float d = 0.f;
        for_row_chunks<DSUB, E4M3>(cbv, mi * K + tid, [&](int c, const unsigned long long (&f)[4]) {
            d = sqdist8(d, xv + mi * DSUB + c * 8, f);
        });
        dv[mi] = d;
    }
#pragma unroll
    for (int mi = 0; mi < MC; ++mi) warp_argmin_into(dv[mi], &keys[mi]);
}

template <int M, int G, int C, bool APPEND, bool E4M3, bool STREAM>
__global__ void __launch_bounds__(kThreads, kMinBlocks<G, C>) pq_decode_kernel(const __grid_constant__ DecodeParams p) {
    using S = PqCfg<M, G, C>;
    constexpr int D = S::D, K = S::K, P = S::P, DSUB = S::DSUB, MC = S::MC, TPT = S::TPT, NCH = S::NCH;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);   // CK, CV, LUT in, bins in, query
    int *sflag = reinterpret_cast<int *>(smem + S::OFF_MISC);           // [0] local bad, [1] all
    __half *cbk = reinterpret_cast<__half *>(smem + S::OFF_CB);       // K slice
    // V slice: its own buffer, or the K slice's; raw E4M3 slices are half the
    // size, so with a shared buffer the V slice takes its upper half
    constexpr bool SHARED_V = S::SHARED_CB && !E4M3;
    __half *cbv = reinterpret_cast<__half *>(smem + S::OFF_CBV + (S::SHARED_CB && E4M3 ? S::CB_BYTES / 2 : 0));
    float *lut = reinterpret_cast<float *>(smem + S::OFF_LUT);
    float *bins = reinterpret_cast<float *>(smem + S::OFF_BINS);
    float *inc = reinterpret_cast<float *>(smem + S::OFF_INC);
    float *qs = reinterpret_cast<float *>(smem + S::OFF_Q);
    float *red_m = reinterpret_cast<float *>(smem + S::OFF_RED);
    float *red_l = red_m + kWarps * G;
    float *mst = reinterpret_cast<float *>(smem + S::OFF_STAT);        // merged max [G]
    float *lst = mst + G;                                               // merged sum [G]
    float *xnew = reinterpret_cast<float *>(smem + S::OFF_NEW);        // [2][MC][DSUB]
    int *newc = reinterpret_cast<int *>(xnew + 2 * MC * DSUB);          // [2][M]
    float *snew = reinterpret_cast<float *>(newc + 2 * M);              // [G]
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(smem + S::OFF_KEYS);  // [2][MC] argmin slots

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int rank = 0;
    if constexpr (C > 1) rank = static_cast<int>(cluster_ctarank());
    const int split = blockIdx.x / C;
    // blockIdx.y = kv head * 2^head_split_log2 + sub-group: this cluster serves
    // query heads [blockIdx.y * G, +G) of kv head blockIdx.y >> head_split_log2
    const int kvh = static_cast<int>(blockIdx.y >> p.head_split_log2), b = blockIdx.z;
    const int hq0 = p.q_head_base + static_cast<int>(blockIdx.y) * G;
    const int Hq = p.num_q_heads, Hkv = p.num_kv_heads;
    const int S_ = p.num_splits;

    // slices by TMA (one elected thread, hardware swizzle) when the base is
    // 1024-byte aligned and a tensor map was made; else by per-thread 16-byte
    // copies into the same layout (one arrival per thread)
    const bool use_tma = p.cb_map_ok && (smem_u32(smem) & 1023u) == 0;
    // bytes of one slice as copied (E4M3 slices stay one byte per element and
    // are widened by their readers) and of one subspace's box within it
    constexpr uint32_t SLICE_BYTES = E4M3 ? S::CB_BYTES / 2 : S::CB_BYTES;
    constexpr int SUB_BYTES = K * DSUB * (E4M3 ? 1 : 2);
    auto slice_copy = [&](void *dst, int row0, uint64_t *b) {      // rows row0 .. of the codebooks
        if (use_tma) {
            if (tid == 0) {
                mbar_arrive_expect_tx(b, SLICE_BYTES);
#pragma unroll
                for (int mi = 0; mi < MC; ++mi)
                    tma_load_2d(static_cast<unsigned char *>(dst) + mi * SUB_BYTES, &p.cb_map, 0, row0 + mi * K, b);
            }
        } else if constexpr (E4M3) {
            copy_slice_e4m3_raw<DSUB, MC * K>(static_cast<unsigned char *>(dst),
                                              static_cast<const uint8_t *>(p.codebooks) + static_cast<size_t>(row0) * DSUB, b);
        } else {
            copy_slice<DSUB, S::CB_CHUNKS>(static_cast<__half *>(dst),
                                           static_cast<const __half *>(p.codebooks) + static_cast<size_t>(row0) * DSUB, b);
        }
    };
    if (tid == 0) {
        mbar_init(&bar[0], use_tma ? 1 : kThreads);
        mbar_init(&bar[1], use_tma ? 1 : kThreads);
        mbar_init(&bar[2], 1);
        mbar_init(&bar[3], 1);
        mbar_init(&bar[4], 1);
        fence_mbar_init();
        sflag[0] = 0;
    }
    __syncthreads();
    // ---- reads allowed before the preceding kernel on the stream completes
    // (programmatic dependent launch): req_set, seq_lens, the block table, the
    // codebooks and the code pages, which that kernel does not write ---------
    const int share = p.share;
    const int ts = split * p.split_len;
    const int a0 = ts + rank * share;
    const int g = tid % G, jslot = tid / G;
    const int32_t *bt = p.block_table + static_cast<size_t>(b) * p.max_pages;
    const int set = __ldg(p.req_set + b);
    const int L_raw = __ldg(p.seq_lens + b);
    // page ids of this thread's tokens (before the length is known: only
    // entries inside the block-table row are read)
    int pid[TPT];
    {
        const int t_lim = min(a0 + share, p.max_pages * P);
#pragma unroll
        for (int i = 0; i < TPT; ++i) {
            pid[i] = -1;
            if (i * S::TOK_PER_PASS >= share) break;
            const int t = a0 + i * S::TOK_PER_PASS + jslot;
            if (t < t_lim) pid[i] = __ldg(bt + static_cast<unsigned>(t) / P);
        }
    }
    const bool set_ok = set >= 0 && static_cast<int64_t>(set) < p.num_sets;
    // first codebook row of this CTA's K slice (rows of DSUB elements; the V
    // slice is M*K rows further); element offsets are rows * DSUB
    const int rowK = ((set_ok ? set : 0) * Hkv + kvh) * 2 * M * K + rank * MC * K;
    // the K slice now; the V slice too with its own buffer and TMA, else once
    // the K slice has landed (own buffer) or is no longer read (shared buffer)
    if (set_ok) slice_copy(cbk, rowK, &bar[0]);

    // ---- request-level checks: uniform over the cluster ------------------
    int bad0 = 0;
    if (L_raw < 0 || L_raw > p.max_pages * P || L_raw > p.max_seq_len) bad0 |= AQ_DEV_BAD_LENGTH;
    if (!set_ok) bad0 |= AQ_DEV_BAD_SET;
    const int te = bad0 ? ts : min(L_raw, ts + p.split_len);
    if (bad0 || ts >= te) {
        // nothing to stream: NaN for a bad request, zeros / empty partials otherwise
        grid_dependency_wait();
        if (rank == 0) {
            if (bad0 && tid == 0) flag_status(p.status, bad0);
            const float v = bad0 ? __int_as_float(0x7fc00000) : 0.0f;
            for (int i = tid; i < G * D; i += kThreads) {
                const int gg = i / D, d = i % D;
                const size_t bh = static_cast<size_t>(b) * Hq + hq0 + gg;
                if (S_ == 1) p.out[bh * D + d] = v;
                else if (d == 0) {
                    p.part_ml[(bh * S_ + split) * 2 + 0] = bad0 ? v : -INFINITY;
                    p.part_ml[(bh * S_ + split) * 2 + 1] = bad0 ? v : 0.0f;
                }
            }
        }
        if (set_ok) {
            if (!use_tma) cp_async_wait_all();         // this thread's slice copies land first
            else mbar_wait_bounded(&bar[0], 0);        // and the TMA copy
        }
        return;
    }
    const int e0 = min(te, a0 + share);
    // the fused step's new token: position L-1, held by the cluster of its split
    // and streamed by no CTA (it is scored from its fresh codes instead)
    const int new_pos = APPEND ? L_raw - 1 : -1;
    const bool cl_new = APPEND && new_pos >= ts && new_pos < te;
    const bool own_new = cl_new && new_pos >= a0 && new_pos < e0;
    const int eS = own_new ? new_pos : e0;
    const int pg_new = cl_new ? __ldg(bt + new_pos / P) : -1;   // checked where it is used
    if constexpr (C > 1) {
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar[2], (C - 1) * (S::ROW_FLOATS + (cl_new ? MC : 0)) * 4);
            mbar_arrive_expect_tx(&bar[3], (C - 1) * (S::ROW_FLOATS + S::STAT_FLOATS) * 4);
        }
    }
    // ---- this thread's codes, straight to registers --------------------------
    Codes<M> cc[TPT];
    unsigned valid = 0;                                 // bit i: token i is streamed
    bool bad_pg = false;
    const size_t page_stride = static_cast<size_t>(Hkv) * (P * 2 * M);  // one page, all kv heads
    const uint8_t *codes_kvh = p.code_pages + static_cast<size_t>(kvh) * (P * 2 * M);
    const int nslot = (eS - a0 + S::TOK_PER_PASS - 1) / S::TOK_PER_PASS;   // token slots in use
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
        if (i >= nslot) break;
        const int t = a0 + i * S::TOK_PER_PASS + jslot;
        if (t < eS) {
            const int pg = pid[i];
            if (pg >= 0 && static_cast<int64_t>(pg) < p.num_pages) {
                cc[i].load_global(codes_kvh + static_cast<size_t>(pg) * page_stride +
                                  (static_cast<unsigned>(t) % P) * (2 * M));
                valid |= 1u << i;
            } else {
                bad_pg = true;
            }
        }
    }
    // ---- the query and the new token come from the preceding kernel ------------
    grid_dependency_wait();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[4], G * D * 4);
        bulk_g2s(qs, p.q + (static_cast<size_t>(b) * Hq + hq0) * D, G * D * 4,
                 &bar[4]);
    }
    // the new token's owned K and V sub-vector elements, one per thread
    if constexpr (APPEND) {
        if (cl_new && tid < 2 * MC * DSUB) {
            const int w = tid / (MC * DSUB), r = tid % (MC * DSUB);
            xnew[tid] = __half2float(__ldg(reinterpret_cast<const __half *>(p.kv_new) +
                                           ((static_cast<size_t>(b) * p.qo_kv_heads + p.kv_head_base + kvh) * 2 + w) * D +
                                           rank * MC * DSUB + r));
        }
    }
    for (int i = tid; i < S::BIN_WORDS / 4; i += kThreads)
        reinterpret_cast<float4 *>(bins)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < G) snew[tid] = -INFINITY;
    if (tid < S::NKEY) keys[tid] = ~0ull;
    grid_launch_dependents();                          // every read of this CTA is issued
    __syncthreads();                                   // bins, new token, flags visible
    if (bad_pg) atomicOr(&sflag[0], AQ_DEV_BAD_PAGE);
    if constexpr (C > 1) cluster_arrive_relaxed();     // this CTA's barriers are ready for pushes

    // ---- lookup-table rows of the owned subspaces, pushed to the peers; the
    // new token's K and V codes from the same rows --------------------------
    bool tmo = !mbar_wait_limit(&bar[0], 0, p.wait_limit_ns);
    // the V slice into its own buffer once the K slice has landed, so that
    // the K slice, which the table build waits for, has the bandwidth first
    if constexpr (!SHARED_V) slice_copy(cbv, rowK + M * K, &bar[1]);
    tmo |= !mbar_wait_limit(&bar[4], 0, p.wait_limit_ns);
    if constexpr (C > 1) cluster_wait_acquire();       // peers' barriers expect our pushes
    float dkv[MC];
    int vcode[MC];                                     // the new token's V codes, owned subspaces
#pragma unroll
    for (int mi = 0; mi < MC; ++mi) vcode[mi] = -1;
#pragma unroll
    for (int mi = 0; mi < MC; ++mi) {
        const int m = rank * MC + mi;
        const float *qm = qs + m * DSUB;
        unsigned long long acc2[G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) acc2[gg] = 0ull;
        float dk = 0.f;
        for_row_chunks<DSUB, E4M3>(cbk, mi * K + tid, [&](int c, const unsigned long long (&f)[4]) {
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                const ulonglong2 *qv = reinterpret_cast<const ulonglong2 *>(qm + gg * D + c * 8);
                const ulonglong2 qa = qv[0], qb = qv[1];
                unsigned long long a = acc2[gg];
                a = f2_fma(qa.x, f[0], a);
                a = f2_fma(qa.y, f[1], a);
                a = f2_fma(qb.x, f[2], a);
                a = f2_fma(qb.y, f[3], a);
                acc2[gg] = a;
            }
            if (APPEND && cl_new) dk = sqdist8(dk, xnew + mi * DSUB + c * 8, f);
        });
        float acc[G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            const float2 a = f2_unpack(acc2[gg]);
            acc[gg] = (a.x + a.y) * p.scale_log2;
        }
        store_vec<G>(lut + (static_cast<size_t>(m) * K + tid) * G, acc);
        dkv[mi] = dk;
    }
    if constexpr (APPEND) {
        if (cl_new) {
#pragma unroll
            for (int mi = 0; mi < MC; ++mi) warp_argmin_into(dkv[mi], &keys[mi]);
        }
    }
    if constexpr (C > 1) fence_proxy_async_shared();  // the rows, for the bulk copies below
    __syncthreads();                                   // every read of the K slice is done
    if constexpr (SHARED_V) {
        if (use_tma && tid == 0) fence_proxy_async_shared();   // the K slice's reads precede the overwrite
        slice_copy(cbv, rowK + M * K, &bar[1]);
    }
    if constexpr (C > 1) {
        // this CTA's rows to every peer in one bulk copy each; the source is not
        // written again before every peer has received it (each peer scores,
        // and pushes its bins, only once it has)
        if (tid < C - 1) {
            const uint32_t pr = static_cast<uint32_t>(rank + tid + 1) & (C - 1);
            const uint32_t rows = smem_u32(lut + rank * S::ROW_FLOATS);
            bulk_s2cluster(mapa_u32(rows, pr), rows, S::ROW_FLOATS * 4, mapa_u32(smem_u32(&bar[2]), pr));
        }
    }
    if constexpr (APPEND) {
        if (cl_new) {
            if (tid < MC) {                            // K code of subspace rank*MC + tid, to every CTA
                const int m = rank * MC + tid;
                const int code = static_cast<int>(keys[tid] & 0xffu);
                newc[m] = code;
                if constexpr (C > 1) {
                    const uint32_t la = smem_u32(&newc[m]), lb = smem_u32(&bar[2]);
#pragma unroll
                    for (int r = 1; r < C; ++r) {
                        const uint32_t pr = static_cast<uint32_t>(rank + r) & (C - 1);
                        st_async_f32(mapa_u32(la, pr), __int_as_float(code), mapa_u32(lb, pr));
                    }
                }
            }
        }
    }
    if constexpr (C > 1) tmo |= !mbar_wait_limit(&bar[2], 0, p.wait_limit_ns);
    if (tmo) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
    __syncthreads();

    // ---- scores, softmax statistics, value bins --------------------------------
    // Scores by M table gathers stay in registers.  The max of each warp's
    // lanes of head g comes first, the weights relative to it and their sum
    // next; the warps' (max, sum) pairs are merged with one barrier (PAM
    // article §2.2.3 item 1: blockwise statistics merged by rescaling), so the
    // block's max mx and weight sum lsum are known before any weight is
    // binned.  Each weight
    // p = 2^(s - mx) then enters the 256-bin value accumulators as the unsigned
    // fixed-point integer round(p * 2^31 / lsum): the bins of one head sum to
    // 2^31 (plus at most n/2 from rounding and a relative 2^-20 from the
    // approximate exp2), so no bin can overflow 32 bits, and the weight lost to
    // rounding is at most n/2 units of lsum/2^31, a relative n/2^32 of the
    // block's weight (5e-7 at n = 2048 tokens).  Integer shared-memory atomics
    // are exact and fast, and the result does not depend on their order.  The
    // fused step's new token enters the statistics from its fresh codes; its
    // value bin is added after the merge.
    unsigned *ibins = reinterpret_cast<unsigned *>(bins);
    float s_new = -INFINITY;
    if constexpr (APPEND) {
        if (own_new && tid < G) {
            s_new = 0.f;
#pragma unroll
            for (int m = 0; m < M; ++m) s_new += lut[(m * K + newc[m]) * G + tid];
            snew[tid] = s_new;
        }
    }
    // A share of more than one chunk (TPT x TOK_PER_PASS tokens: the codes one
    // thread holds) is streamed twice: pass 1 keeps each thread's (max, sum)
    // online over the tokens, pass 2 re-reads the codes (from L2), recomputes
    // the scores and bins the weights against the block's statistics.
    constexpr int CHUNK = TPT * S::TOK_PER_PASS;
    const int nch = (max(eS - a0, 0) + CHUNK - 1) / CHUNK;
    float mx, lsum, cfac;                              // cfac: integer bin -> weight
    auto score = [&](const Codes<M> &cw) {
        float s = 0.f;
#pragma unroll
        for (int m = 0; m < M; ++m) s += lut[(m * K + cw.k(m)) * G + g];
        return s;
    };
    if (!STREAM || nch <= 1) {
        float sc[TPT];
        float mloc = s_new;
    #pragma unroll
        for (int i = 0; i < TPT; ++i) {
            if (i >= nslot) break;
            if (valid & (1u << i)) {
                float s = 0.f;
    #pragma unroll
                for (int m = 0; m < M; ++m) s += lut[(m * K + cc[i].k(m)) * G + g];
                sc[i] = s;
                mloc = fmaxf(mloc, s);
            }
        }
        // the max over the lanes of head g (one redux for G = 1), this thread's
        // weights relative to it (kept in sc) and their sum over the same lanes
        float mg;
        if constexpr (G == 1) {
            mg = warp_max_f32(mloc);
        } else {
            mg = mloc;
    #pragma unroll
            for (int off = G; off < 32; off <<= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, off));
        }
        float lt = (s_new != -INFINITY) ? fast_exp2(s_new - mg) : 0.f;
    #pragma unroll
        for (int i = 0; i < TPT; ++i) {
            if (i >= nslot) break;
            if (valid & (1u << i)) {
                sc[i] = fast_exp2(sc[i] - mg);
                lt += sc[i];
            }
        }
    #pragma unroll
        for (int off = G; off < 32; off <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
        if (lane < G) {
            red_m[warp * G + lane] = mg;
            red_l[warp * G + lane] = lt;
        }
        __syncthreads();
        if constexpr (G == 1) {
            // lane w < kWarps takes warp w's pair; the same reduction in every
            // warp gives every thread the same (max, sum)
            const float mw = lane < kWarps ? red_m[lane] : -INFINITY;
            mx = warp_max_f32(mw);
            lsum = (mw != -INFINITY) ? red_l[lane] * (mw == mx ? 1.0f : fast_exp2(mw - mx)) : 0.f;
    #pragma unroll
            for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
        } else {
            mx = red_m[g];
    #pragma unroll
            for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, red_m[w * G + g]);
            lsum = 0.f;
    #pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float mw = red_m[w * G + g];
                if (mw != -INFINITY) lsum += red_l[w * G + g] * (mw == mx ? 1.0f : fast_exp2(mw - mx));
            }
        }
        // lsum >= 1 whenever this CTA holds a token of head g (its max weighs 1)
        const float qscale = lsum > 0.f ? __fdividef(2147483648.0f, lsum) : 0.f;
        cfac = lsum * (1.0f / 2147483648.0f);
        {
            // weight relative to mx, in bin units: sc[i] * 2^(mg - mx) * qscale
            const float rq = (mg == -INFINITY) ? 0.f : (mg == mx ? qscale : fast_exp2(mg - mx) * qscale);
    #pragma unroll
            for (int i = 0; i < TPT; ++i) {
                if (i >= nslot) break;
                if (valid & (1u << i)) {
                    const unsigned q = __float2uint_rn(sc[i] * rq);
    #pragma unroll
                    for (int m = 0; m < M; ++m) atomicAdd(&ibins[(m * K + cc[i].vv(m)) * G + g], q);
                }
            }
        }
    } else if constexpr (STREAM) {
        // This thread's tokens in halves of HT slots (half h: tokens
        // a0 + (h*HT + i)*TOK_PER_PASS + jslot), software-pipelined: while
        // half h is scored from one register slot, the codes of half h+1 are
        // in flight into the other and the page ids of the next refill are
        // loading, so neither the block-table nor the code latency is exposed.
        constexpr int HT = TPT / 2;
        const int NH = (max(eS - a0, 0) + HT * S::TOK_PER_PASS - 1) / (HT * S::TOK_PER_PASS);
        int pidn[HT];
        auto tok = [&](int h, int i) { return a0 + (h * HT + i) * S::TOK_PER_PASS + jslot; };
        auto load_pids = [&](int h) {
#pragma unroll
            for (int i = 0; i < HT; ++i) {
                const int t = tok(h, i);
                pidn[i] = (h < NH && t < eS) ? __ldg(bt + static_cast<unsigned>(t) / P) : -2;
            }
        };
        auto issue = [&](auto slot, int h) {                 // codes of half h into slot, from pidn
            constexpr int sl = decltype(slot)::value;
#pragma unroll
            for (int i = 0; i < HT; ++i) {
                valid &= ~(1u << (sl * HT + i));
                const int t = tok(h, i);
                if (h < NH && t < eS) {
                    const int pg = pidn[i];
                    if (pg >= 0 && static_cast<int64_t>(pg) < p.num_pages) {
                        cc[sl * HT + i].load_global(codes_kvh + static_cast<size_t>(pg) * page_stride +
                                                    (static_cast<unsigned>(t) % P) * (2 * M));
                        valid |= 1u << (sl * HT + i);
                    } else {
                        bad_pg = true;
                    }
                }
            }
        };
        // one pass: f(slot, h) consumes half h from its slot, which is then
        // refilled with half h+2 (halves 0 and 1 are in their slots at entry)
        auto pass = [&](auto f) {
            load_pids(2);
            for (int h0 = 0; h0 < NH; h0 += 2) {
                f(IntC<0>{}, h0);
                issue(IntC<0>{}, h0 + 2);
                load_pids(h0 + 3);
                if (h0 + 1 < NH) {
                    f(IntC<1>{}, h0 + 1);
                    issue(IntC<1>{}, h0 + 3);
                    load_pids(h0 + 4);
                }
            }
        };
        // One pass: each half is scored, its block-wide (max, sum) per head
        // merged over the warps (two alternating buffers, one barrier), and its
        // weights binned at once in fixed point against a per-head frame (Mb,
        // Sb): a bin holds sum round(2^(s - Mb) * Sb) over its tokens, Lb =
        // sum 2^(s - Mb) over every token seen.  The frame moves only when a
        // half would take the bins' total Lb * Sb past 2^31: then Mb becomes
        // the running max, Sb = 2^30 / Lb, and the bins already filled are
        // rescaled once (factor <= 1).  So no bin overflows 32 bits, the
        // final resolution is at least 2^-31 of the weight sum (each weight
        // rounded by half a unit, each rescale by half a unit per bin), and
        // the codes are read once (PAM article §2.2.3 item 1: blockwise
        // statistics merged by rescaling).  The new token's weight enters Lb
        // (not the bins: its value bin is added after the merge).
        float Mb = -INFINITY, Lb = 0.f, Sb = 0.f;
        __syncthreads();                               // the new token's score in snew
        {
            const float sn = snew[g];
            if (sn != -INFINITY) {
                Mb = sn;
                Lb = 1.f;
                Sb = 1073741824.0f;
            }
        }
        int hh = 0;                                    // halves consumed (buffer parity)
        pass([&](auto slot, int) {
            constexpr int sl = decltype(slot)::value;
            float sc[HT];
            float mloc = -INFINITY;
#pragma unroll
            for (int i = 0; i < HT; ++i)
                if (valid & (1u << (sl * HT + i))) {
                    sc[i] = score(cc[sl * HT + i]);
                    mloc = fmaxf(mloc, sc[i]);
                }
            float mg;
            if constexpr (G == 1) {
                mg = warp_max_f32(mloc);
            } else {
                mg = mloc;
#pragma unroll
                for (int off = G; off < 32; off <<= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, off));
            }
            float lt = 0.f;
#pragma unroll
            for (int i = 0; i < HT; ++i)
                if (valid & (1u << (sl * HT + i))) {
                    sc[i] = fast_exp2(sc[i] - mg);
                    lt += sc[i];
                }
#pragma unroll
            for (int off = G; off < 32; off <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
            float *rm = red_m + (hh & 1) * 2 * kWarps * G, *rl = rm + kWarps * G;
            if (lane < G) {
                rm[warp * G + lane] = mg;
                rl[warp * G + lane] = lt;
            }
            __syncthreads();
            float hm = -INFINITY, hl = 0.f;
            if constexpr (G == 1) {
                // lane w < kWarps takes warp w's pair; the same reduction in
                // every warp gives every thread the same (max, sum)
                const float mw = lane < kWarps ? rm[lane] : -INFINITY;
                hm = warp_max_f32(mw);
                hl = (mw != -INFINITY) ? rl[lane] * (mw == hm ? 1.0f : fast_exp2(mw - hm)) : 0.f;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) hl += __shfl_xor_sync(0xffffffffu, hl, off);
            } else {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) hm = fmaxf(hm, rm[w * G + g]);
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float mw = rm[w * G + g];
                    if (mw != -INFINITY) hl += rl[w * G + g] * (mw == hm ? 1.0f : fast_exp2(mw - hm));
                }
            }
            bool resc = false;
            float f = 1.f;
            if (hl > 0.f) {
                if (Lb == 0.f) {                       // first weights of head g: the bins are empty
                    Mb = hm;
                    Lb = hl;
                    Sb = __fdividef(1073741824.0f, hl);
                } else {
                    const float add = hl * fast_exp2(hm - Mb);   // this half's weight in the frame (may be inf)
                    if ((Lb + add) * Sb <= 2147483648.0f) {
                        Lb += add;
                    } else {
                        const float Mn = fmaxf(Mb, hm);
                        const float Ln = Lb * fast_exp2(Mb - Mn) + hl * fast_exp2(hm - Mn);
                        const float Sn = __fdividef(1073741824.0f, Ln);
                        f = Sn / Sb * fast_exp2(Mb - Mn);
                        Mb = Mn;
                        Lb = Ln;
                        Sb = Sn;
                        resc = true;
                    }
                }
            }
            AQ_DCHECK(p.status, !(Lb > 0.f) || (Lb * Sb <= 2147483648.0f * 1.001f && f <= 1.0001f));
            bool any = resc;
            if constexpr (G > 1) any = __syncthreads_or(resc);
            if (any) {
                if (resc)                              // this thread's bins: e mod G == g
                    for (int e = tid; e < S::BIN_WORDS; e += kThreads)
                        ibins[e] = __float2uint_rn(static_cast<float>(ibins[e]) * f);
                __syncthreads();
            }
            const float rq = (mg == -INFINITY) ? 0.f : Sb * fast_exp2(mg - Mb);
#pragma unroll
            for (int i = 0; i < HT; ++i)
                if (valid & (1u << (sl * HT + i))) {
                    const Codes<M> &cw = cc[sl * HT + i];
                    const unsigned q = __float2uint_rn(sc[i] * rq);
#pragma unroll
                    for (int m = 0; m < M; ++m) atomicAdd(&ibins[(m * K + cw.vv(m)) * G + g], q);
                }
            ++hh;
        });
        if (bad_pg) atomicOr(&sflag[0], AQ_DEV_BAD_PAGE);
        mx = Mb;
        lsum = Lb;
        cfac = Lb > 0.f ? __fdividef(1.0f, Sb) : 0.f;
    }
    if constexpr (C > 1) fence_proxy_async_shared();  // the bins, for the bulk copies below
    __syncthreads();                                   // every atomic of this CTA is done
#ifdef AQ_DEBUG_CHECKS
    // every token adds the same integer weight to one bin of every subspace:
    // the subspaces' bin sums agree (a streamed share's rescales round each
    // bin by at most half a unit: K/2 per rescale, at most 32 of them), and
    // stay below 2^31 + rounding
    if (tid < M * G) {
        const int m = tid / G, gg = tid % G;
        unsigned long long s0 = 0, sm = 0;
        for (int k = 0; k < K; ++k) {
            s0 += ibins[k * G + gg];
            sm += ibins[(m * K + k) * G + gg];
        }
        const unsigned long long slack = (STREAM && nch > 1) ? 16ull * K : 0ull;
        AQ_DCHECK(p.status, sm <= s0 + slack && s0 <= sm + slack && s0 < 3ull * 1073741824ull);
    }
#endif

    // ---- bins rows (integers, one bulk copy per peer) and statistics to the
    // peers that own them; sender rank lands in slot (rank - pr - 1) mod C ----
    if constexpr (C > 1) {
        const uint32_t lb = smem_u32(&bar[3]);
        // warp r-1 serves peer r: lane 0 the bulk copy, lanes g < G the statistics
        if (warp < C - 1 && lane < G) {                // g == lane here
            const int r = warp + 1;
            const uint32_t pr = static_cast<uint32_t>(rank + r) & (C - 1);
            const uint32_t rslot = smem_u32(inc + (C - r - 1) * S::INC_STRIDE);
            const uint32_t rbar = mapa_u32(lb, pr);
            if (lane == 0)
                bulk_s2cluster(mapa_u32(rslot, pr), smem_u32(ibins + pr * S::ROW_FLOATS), S::ROW_FLOATS * 4, rbar);
            const uint32_t st = mapa_u32(rslot + 4 * S::ROW_FLOATS, pr);
            st_async_f32(st + 4 * lane, mx, rbar);
            st_async_f32(st + 4 * (G + lane), lsum, rbar);
            st_async_f32(st + 4 * (2 * G + lane), snew[lane], rbar);
            st_async_f32(st + 4 * (3 * G + lane), cfac, rbar);
            if (lane == 0) st_async_f32(st + 4 * (4 * G), __int_as_float(sflag[0]), rbar);
        }
    }
    // the new token's V codes (the peers' bins are landing meanwhile: the
    // codes are first needed by the merge, so the encode stays off the path
    // from the table rows to the scores), then its codes into its page slot,
    // its page id checked here
    if constexpr (APPEND) {
        if (cl_new) {
            if (!mbar_wait_limit(&bar[1], 0, p.wait_limit_ns)) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
            encode_new_value<DSUB, MC, K, NCH, E4M3>(cbv, xnew + MC * DSUB, keys + MC);
            __syncthreads();
#pragma unroll
            for (int mi = 0; mi < MC; ++mi) vcode[mi] = static_cast<int>(keys[MC + mi] & 0xffu);
            if (tid == 0) {
                const bool pg_ok = pg_new >= 0 && static_cast<int64_t>(pg_new) < p.num_pages;
                if (pg_ok && !(sflag[0] & AQ_DEV_TIMEOUT)) {   // no codes from data that may not have landed
                    uint8_t *dst = p.code_pages_w +
                                   ((static_cast<size_t>(pg_new) * Hkv + kvh) * P + new_pos % P) * (2 * M);
#pragma unroll
                    for (int mi = 0; mi < MC; ++mi) {
                        dst[rank * MC + mi] = static_cast<uint8_t>(newc[rank * MC + mi]);
                        dst[M + rank * MC + mi] = static_cast<uint8_t>(vcode[mi]);
                    }
                } else {
                    atomicOr(&sflag[0], AQ_DEV_BAD_PAGE);
                }
            }
        }
    }
    if constexpr (C > 1) {
        if (!mbar_wait_limit(&bar[3], 0, p.wait_limit_ns)) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
        cluster_arrive_relaxed();                      // all traffic into this CTA has landed
    }

    // ---- merge: every thread merges the statistics of its head g, then its
    // elements (e = tid + j*kThreads, so e mod G == g) of the owned bin rows --
    // peers by distance d = 1..C-1 from this CTA: the CTA of rank (rank+d) mod C
    // pushed into slot d-1, so every index below is a compile-time constant
    float ms = -INFINITY, ls = 0.f, sn = snew[g];
    float fac[C];                                      // [d]: scale of distance d's rows
    float pscale[C];                                   // [d]: distance d's integer-bin scale
    pscale[0] = cfac;
    {
        float md[C], ld[C];
        md[0] = mx;
        ld[0] = lsum;
#pragma unroll
        for (int d = 1; d < C; ++d) {
            const float *sl = inc + (d - 1) * S::INC_STRIDE + S::ROW_FLOATS;
            md[d] = sl[g];
            ld[d] = sl[G + g];
            sn = fmaxf(sn, sl[2 * G + g]);
            pscale[d] = sl[3 * G + g];
        }
#pragma unroll
        for (int d = 0; d < C; ++d)
            if (ld[d] > 0.f) ms = fmaxf(ms, md[d]);
#pragma unroll
        for (int d = 0; d < C; ++d) {
            const float f = (ld[d] > 0.f) ? fast_exp2(md[d] - ms) : 0.f;
            ls += f * ld[d];
            fac[d] = f * pscale[d];                    // integer bin -> weight relative to ms
        }
    }
    if (tid < G) {
        mst[tid] = ms;
        lst[tid] = ls;
    }
    if (tid == 0) {
        int bb = sflag[0];
#pragma unroll
        for (int d = 1; d < C; ++d) bb |= __float_as_int(inc[(d - 1) * S::INC_STRIDE + S::ROW_FLOATS + 4 * G]);
        sflag[1] = bb;
        if (sflag[0]) flag_status(p.status, sflag[0]);
    }
    float *wtot = lut;                                 // [MC][K][G]; the LUT is no longer read
    {
        const float wnew = (APPEND && cl_new && sn != -INFINITY) ? fast_exp2(sn - ms) : 0.f;
        const unsigned *own = ibins + rank * S::ROW_FLOATS;
#pragma unroll
        for (int mi = 0; mi < MC; ++mi) {
            for (int e1 = tid; e1 < K * G; e1 += kThreads) {   // e1 mod G == g
                const int e = mi * K * G + e1;
                float a = fac[0] * static_cast<float>(own[e]);
#pragma unroll
                for (int d = 1; d < C; ++d)
                    a += fac[d] * static_cast<float>(reinterpret_cast<const unsigned *>(inc)[(d - 1) * S::INC_STRIDE + e]);
                if constexpr (APPEND) {
                    // the new token's value bin
                    if (cl_new && static_cast<unsigned>(e1) / G == static_cast<unsigned>(vcode[mi])) a += wnew;
                }
                wtot[e] = a;
            }
        }
    }
    __syncthreads();
    int bad_all = sflag[1];

    // ---- value codebook product for the owned subspaces -----------------------
    if (!mbar_wait_limit(&bar[1], 0, p.wait_limit_ns)) {
        atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
        bad_all |= AQ_DEV_TIMEOUT;
    }
    // thread = (k slice, 4-dim quad of the owned dims): 8-byte codebook loads,
    // the slices of a warp reduced by shuffles, the warps through shared memory
    float *ored = C > 1 ? inc : bins;                  // [kWarps][MC*DSUB][G]; merged, not in flight
    {
        constexpr int NQ = MC * DSUB / 4, KSQ = kThreads / NQ, KSLQ = K / KSQ;
        constexpr int ROWS128 = 128 / (DSUB * 2);
        static_assert(KSQ % (ROWS128 * NCH) == 0, "row step keeps the swizzle position");
        const int qd = tid % NQ, ks = tid / NQ;
        const int mi = qd / (DSUB / 4), j4 = (qd % (DSUB / 4)) * 4;
        const int cj = j4 / 8, hj = j4 % 8;
        // rows k = kx + i*KSQ, kx = ks ^ (mi * VP_XOR): the rows of one load are
        // bank-conflict-free, and every row of a thread holds chunk cj at the
        // same swizzled position, so all loads are at fixed offsets
        const int kx = ks ^ ((mi * S::VP_XOR) & (KSQ - 1));
        const __half *vrow = cbv + ((mi * K + kx) * NCH + chunk_pos<DSUB>(kx, cj)) * 8 + hj;
        // raw E4M3 slice: the quad's 4 bytes (the rows kx + i*KSQ share kx's chunk position)
        const unsigned char *vrow8 = reinterpret_cast<const unsigned char *>(cbv) + (mi * K + kx) * DSUB +
                                     e8_pos<DSUB>(kx, j4 / 16) * 16 + j4 % 16;
        static_assert(!E4M3 || DSUB == 16 || KSQ % 8 == 0, "row step keeps the E4M3 chunk position");
        const float *wrow = wtot + (static_cast<size_t>(mi) * K + kx) * G;
        unsigned long long acc[G][2];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) acc[gg][0] = acc[gg][1] = 0ull;
#pragma unroll 8
        for (int i = 0; i < KSLQ; ++i) {
            unsigned long long c01, c23;
            if constexpr (E4M3) {
                const uint32_t b4 = *reinterpret_cast<const uint32_t *>(vrow8 + i * KSQ * DSUB);
                const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(b4 & 0xffffu), __NV_E4M3);
                const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(b4 >> 16), __NV_E4M3);
                c01 = h2_to_f2p(static_cast<uint32_t>(h01.x) | (static_cast<uint32_t>(h01.y) << 16));
                c23 = h2_to_f2p(static_cast<uint32_t>(h23.x) | (static_cast<uint32_t>(h23.y) << 16));
            } else {
                const uint2 cv2 = *reinterpret_cast<const uint2 *>(vrow + i * KSQ * NCH * 8);
                c01 = h2_to_f2p(cv2.x);
                c23 = h2_to_f2p(cv2.y);
            }
            float w[G];
            load_vec<G>(w, wrow + i * KSQ * G);
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                const unsigned long long ww = f2_pack(w[gg], w[gg]);
                acc[gg][0] = f2_fma(ww, c01, acc[gg][0]);
                acc[gg][1] = f2_fma(ww, c23, acc[gg][1]);
            }
        }
        float accf[G][4];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            const float2 a01 = f2_unpack(acc[gg][0]), a23 = f2_unpack(acc[gg][1]);
            accf[gg][0] = a01.x; accf[gg][1] = a01.y; accf[gg][2] = a23.x; accf[gg][3] = a23.y;
        }
#pragma unroll
        for (int off = NQ; off < 32; off <<= 1) {
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
#pragma unroll
                for (int e = 0; e < 4; ++e) accf[gg][e] += __shfl_xor_sync(0xffffffffu, accf[gg][e], off);
        }
        if (lane < NQ) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v[G];
#pragma unroll
                for (int gg = 0; gg < G; ++gg) v[gg] = accf[gg][e];
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
            const size_t bh = static_cast<size_t>(b) * Hq + hq0 + gg;
            const float nan = __int_as_float(0x7fc00000);
            if (S_ == 1) {
                const float l = lst[gg];
                p.out[bh * D + d] = bad_all ? nan : (l > 0.f ? __fdividef(o, l) : 0.f);
            } else {
                AQ_DCHECK(p.status, bh < static_cast<size_t>(p.batch) * Hq && split < S_);
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
        cp_async_wait_all();
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
    const size_t bh = static_cast<size_t>(blockIdx.y) * p.num_q_heads + p.q_head_base + blockIdx.x;
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

// ============================================================================
// Whole-split kernel.  One cluster of C CTAs per (request, kv head [, query-
// head sub-group], split); CTA `rank` owns subspaces [rank*M/C, (rank+1)*M/C)
// of both codebooks.  Unlike pq_decode_kernel, every CTA reads the codes of
// all tokens of the split (whole 16-token pages, copied into shared memory;
// the pages come from L2 after the first CTA's read) and scores all of
// them, so every CTA holds the split's softmax statistics itself: only the
// lookup-table rows cross the cluster.  Each CTA then bins the weights by its
// own subspaces' value codes and applies its own value-codebook slice, which
// gives its own output dimensions directly -- no exchange of value bins, no
// merge.  The codebook slices arrive by TMA tensor copies whose hardware
// swizzle places chunk c of row k where chunk_pos() expects it.
//
//  1. TMA: K and V codebook slices; cp.async: the split's code pages; the
//     query group (after the dependency wait);
//  2. LUT rows of the owned subspaces (AQPIM blog §4.1, §5.1 item 3), pushed
//     to the peers; the fused step's new key encoded from the same rows;
//  3. scores of every token of the split, s = sum_m LUT[m][kcode_m]; the
//     split's (max, sum) per head (PAM article §2.2.3 item 1) by an online
//     merge of per-thread pairs and one barrier;
//  4. 256-bin value accumulators of the owned subspaces, fixed point relative
//     to the split's weight sum; o = sum_k W[k] * C^V[k] for the owned dims;
//  5. normalise and store, or store (max, sum, o) partials for the combine.
// ============================================================================
template <int M, int G, int C>
struct AtCfg {
    static constexpr int D = kHeadDim, K = kCodewords, P = kPage;
    static constexpr int DSUB = D / M;
    static constexpr int NCH = DSUB / 8;
    static constexpr int MC = M / C;
    static constexpr int SLICE_BYTES = MC * K * DSUB * 2;   // owned part of one codebook
    static constexpr int LUT_FLOATS = M * K * G;
    static constexpr int ROW_FLOATS = MC * K * G;           // this CTA's LUT rows
    static constexpr int BIN_WORDS = MC * K * G;            // u32 value bins [MC][K][G]
    static constexpr int TOK_PER_PASS = kThreads / G;
    static constexpr int TPT = G == 8 ? 32 : 16;            // scores per thread, in registers
    static constexpr int PAGE_BYTES = P * 2 * M;
    static constexpr int CODE_CAP = 32768;                  // code bytes of one split
    static constexpr int MAX_SPLIT = (TPT * TOK_PER_PASS < CODE_CAP / (2 * M) ? TPT * TOK_PER_PASS
                                                                               : CODE_CAP / (2 * M)) / P * P;
    static constexpr int NOUT = MC * DSUB * G;              // output elements of this CTA
    // layout from the 1024-aligned base
    static constexpr int OFF_CBK = 0;
    static constexpr int OFF_CBV = SLICE_BYTES;
    static constexpr int OFF_LUT = 2 * SLICE_BYTES;
    static constexpr int OFF_BINS = OFF_LUT + LUT_FLOATS * 4;
    static constexpr int OFF_Q = OFF_BINS + BIN_WORDS * 4;
    static constexpr int OFF_PART = OFF_Q + G * D * 4;      // V-product partials [kWarps][NOUT]
    static constexpr int OFF_RED = OFF_PART + kWarps * NOUT * 4;   // red_m, red_l [kWarps][G]
    static constexpr int OFF_STAT = OFF_RED + 2 * kWarps * G * 4;  // mx, lsum, cfac, s_new, qscale [G]
    static constexpr int OFF_NEW = (OFF_STAT + 5 * G * 4 + 15) / 16 * 16;  // xnew [2][MC][DSUB] f32, newc [M]
    static constexpr int OFF_KEYS = (OFF_NEW + 2 * MC * DSUB * 4 + M * 4 + 7) / 8 * 8;  // [2][MC] u64
    static constexpr int OFF_BAR = OFF_KEYS + 2 * MC * 8;   // K, V, codes, q, rows
    static constexpr int OFF_FLAG = OFF_BAR + 5 * 8;
    static constexpr int OFF_PBAD = OFF_FLAG + 16;          // [C] ints
    static constexpr int OFF_CODES = (OFF_PBAD + 4 * C + 15) / 16 * 16;
    static size_t smem(int split_len) { return 1024 + OFF_CODES + static_cast<size_t>(split_len) * 2 * M; }
    static_assert(K == kThreads, "one thread per codeword in the table build");
    static_assert(SLICE_BYTES % 1024 == 0, "slices keep the swizzle alignment");
    static_assert(OFF_LUT % 16 == 0 && OFF_Q % 16 == 0 && OFF_PART % 16 == 0, "alignment");
    static_assert((MC * DSUB / 4) <= 32 && 32 % (MC * DSUB / 4) == 0, "V-product quads within a warp");
    static_assert(ROW_FLOATS % 4 == 0, "bulk copies of whole rows");
    // GQA groups of 4 or more: one thread scores whole tokens for all G heads
    static constexpr bool PER_TOKEN = G >= 4;
    static constexpr int NQ = MC * DSUB / 4;                // value product: 4-dim quads per row
    static constexpr int KSQ = kThreads / NQ;               // its row step
    static constexpr int VPX = (M == 8 && C == 4) ? 2 : 1;  // its k-slice XOR per owned subspace
    // the head permutation of a thread's bin rows is the same across each
    // warp (the lanes differ only in bits of k below the swizzled ones): it
    // is undone where the warps' partials are summed
    static constexpr bool XU = PER_TOKEN && NQ >= (32 >> (5 - (G == 8 ? 3 : 2)));
    static constexpr int TT = MAX_SPLIT / kThreads;         // tokens per thread on that path
    static_assert(!PER_TOKEN || MAX_SPLIT % kThreads == 0, "whole tokens per thread");
};

template <int G>
constexpr int kAtMinBlocks = G == 1 ? 4 : (G == 2 ? 3 : 2);

// Table rows of 8 heads are two 16-byte halves; half h of the row of codeword
// k sits at h ^ ((k >> 2) & 1), so that the rows a warp reads for 32 tokens
// with unrelated codes spread over all eight 16-byte bank groups (without it
// only the even or only the odd groups take a given half).  Rows of 4 heads
// are one 16-byte group already spread by k.
template <int G>
__device__ __forceinline__ int lut_hswz(int k) {
    return G == 8 ? (k >> 2) & 1 : 0;
}

// One table row (G = 4 or 8 floats) as packed pairs, in head order.
template <int G>
__device__ __forceinline__ void lut_row2(const float *lut, int row, unsigned long long (&v)[G / 2]) {
    const ulonglong2 *p = reinterpret_cast<const ulonglong2 *>(lut + static_cast<size_t>(row) * G);
    if constexpr (G == 8) {
        const int h = lut_hswz<G>(row);                 // row = m*K + k with K a multiple of 8
        const ulonglong2 a = p[h], b = p[h ^ 1];
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    } else {
        static_assert(G == 4, "rows of 4 or 8 heads");
        const ulonglong2 a = p[0];
        v[0] = a.x; v[1] = a.y;
    }
}

// Value bins of a GQA group of 4 or 8 filled one token (all G heads) per
// thread: head g of codeword k sits at word g ^ s(k) of its row, s(k) taken
// from the bits of k just above those that pick the bank group of the row,
// so that 32 tokens with unrelated codes adding head g spread over all 32
// banks (unswizzled, rows of 8 words would put them on 4 banks).  s(k) uses
// bits below log2(KSQ) only, the bits that stay fixed along the rows one
// thread reads in the value product (its rows step by KSQ).
template <int G, int KSQ>
__device__ __forceinline__ int bin_wswz(int k) {
    constexpr int LG = G == 8 ? 3 : (G == 4 ? 2 : 0);
    constexpr int SH = 5 - LG;                          // bits of k above the row's bank group
    constexpr int BITS = (KSQ >= 32 ? 5 : (KSQ >= 16 ? 4 : 3)) - SH;
    constexpr int NB = BITS < LG ? (BITS > 0 ? BITS : 0) : LG;
    return (k >> SH) & ((1 << NB) - 1);
}

template <int M, int G, int C, bool APPEND>
__global__ void __launch_bounds__(kThreads, kAtMinBlocks<G>) pq_attend_kernel(const __grid_constant__ DecodeParams p) {
    using S = AtCfg<M, G, C>;
    constexpr int D = S::D, K = S::K, P = S::P, DSUB = S::DSUB, MC = S::MC, TPT = S::TPT, NCH = S::NCH;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __half *cbk = reinterpret_cast<__half *>(smem + S::OFF_CBK);
    __half *cbv = reinterpret_cast<__half *>(smem + S::OFF_CBV);
    float *lut = reinterpret_cast<float *>(smem + S::OFF_LUT);
    unsigned *bins = reinterpret_cast<unsigned *>(smem + S::OFF_BINS);
    float *qs = reinterpret_cast<float *>(smem + S::OFF_Q);
    float *part = reinterpret_cast<float *>(smem + S::OFF_PART);
    float *red_m = reinterpret_cast<float *>(smem + S::OFF_RED);
    float *red_l = red_m + kWarps * G;
    float *st_mx = reinterpret_cast<float *>(smem + S::OFF_STAT);
    float *st_l = st_mx + G, *st_c = st_l + G, *st_sn = st_c + G, *st_qs = st_sn + G;
    float *xnew = reinterpret_cast<float *>(smem + S::OFF_NEW);      // [2][MC][DSUB]
    int *newc = reinterpret_cast<int *>(xnew + 2 * MC * DSUB);        // [M] key codes of the new token
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(smem + S::OFF_KEYS);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);  // K, V, codes, q, rows
    int *sflag = reinterpret_cast<int *>(smem + S::OFF_FLAG);
    int *pbad = reinterpret_cast<int *>(smem + S::OFF_PBAD);          // [C] flags the peers sent with their rows
    const unsigned char *codes = smem + S::OFF_CODES;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int rank = 0;
    if constexpr (C > 1) rank = static_cast<int>(cluster_ctarank());
    const int split = blockIdx.x / C;
    const int kvh = static_cast<int>(blockIdx.y >> p.head_split_log2), b = blockIdx.z;
    const int hq0 = p.q_head_base + static_cast<int>(blockIdx.y) * G;
    const int Hq = p.num_q_heads, Hkv = p.num_kv_heads;
    const int S_ = p.num_splits;

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&bar[i], i == 2 ? kThreads : 1);   // codes: one arrival per thread
        fence_mbar_init();
        sflag[0] = 0;
    }
    __syncthreads();
    // ---- reads allowed before the preceding kernel completes: req_set,
    // seq_lens, the block table, the codebooks and the code pages ------------
    const int set = __ldg(p.req_set + b);
    const int L_raw = __ldg(p.seq_lens + b);
    const bool set_ok = set >= 0 && static_cast<int64_t>(set) < p.num_sets;
    int bad0 = 0;
    if (L_raw < 0 || L_raw > p.max_pages * P || L_raw > p.max_seq_len) bad0 |= AQ_DEV_BAD_LENGTH;
    if (!set_ok) bad0 |= AQ_DEV_BAD_SET;
    const int ts = split * p.split_len;
    const int te = bad0 ? ts : min(L_raw, ts + p.split_len);
    if (bad0 || ts >= te) {
        // nothing to read: NaN for a bad request, zeros / empty partials otherwise
        grid_dependency_wait();
        if (rank == 0) {
            if (bad0 && tid == 0) flag_status(p.status, bad0);
            const float v = bad0 ? __int_as_float(0x7fc00000) : 0.0f;
            for (int i = tid; i < G * D; i += kThreads) {
                const int gg = i / D, d = i % D;
                const size_t bh = static_cast<size_t>(b) * Hq + hq0 + gg;
                if (S_ == 1) p.out[bh * D + d] = v;
                else if (d == 0) {
                    p.part_ml[(bh * S_ + split) * 2 + 0] = bad0 ? v : -INFINITY;
                    p.part_ml[(bh * S_ + split) * 2 + 1] = bad0 ? v : 0.0f;
                }
            }
        }
        return;
    }
    // the fused step's new token (position L-1, the last one) is scored from
    // its fresh codes by every CTA of its split and streamed by none
    const int new_pos = APPEND ? L_raw - 1 : -1;
    const bool cl_new = APPEND && new_pos >= ts && new_pos < te;
    const int ntok = (cl_new ? new_pos : te) - ts;   // streamed tokens [ts, ts + ntok)
    const int32_t *bt = p.block_table + static_cast<size_t>(b) * p.max_pages;
    // the new token's page (written by thread 0 at the end), loaded early
    const int pg_new = (APPEND && cl_new && tid == 0) ? __ldg(bt + new_pos / P) : -1;
    if (tid == 0) {
        // the two codebook slices: one 256-row TMA box per owned subspace
        const int row0 = ((set * Hkv + kvh) * 2) * M * K + rank * MC * K;
        mbar_arrive_expect_tx(&bar[0], S::SLICE_BYTES);
#pragma unroll
        for (int mi = 0; mi < MC; ++mi) tma_load_2d(cbk + mi * K * DSUB, &p.cb_map, 0, row0 + mi * K, &bar[0]);
        mbar_arrive_expect_tx(&bar[1], S::SLICE_BYTES);
#pragma unroll
        for (int mi = 0; mi < MC; ++mi) tma_load_2d(cbv + mi * K * DSUB, &p.cb_map, 0, row0 + M * K + mi * K, &bar[1]);
        if constexpr (C > 1) mbar_arrive_expect_tx(&bar[4], (C - 1) * (S::ROW_FLOATS + (cl_new ? MC : 0) + 1) * 4);
    }
    {
        // the split's code pages, whole pages (16 tokens x 2M codes of this kv
        // head, one line each) into shared memory in token order: 16-byte
        // cp.async chunks, consecutive threads along a page's line, page ids
        // from the block table row (one line per page, so the reads are whole
        // lines even under a shuffled table); one arrival per thread on bar[2]
        constexpr int CPP = S::PAGE_BYTES / 16;          // chunks per page
        const int npg = (ntok + P - 1) / P, pg0 = ts / P;
        const size_t page_stride = static_cast<size_t>(Hkv) * S::PAGE_BYTES;
        const unsigned char *src0 = p.code_pages + static_cast<size_t>(kvh) * S::PAGE_BYTES;
        const uint32_t dst0 = smem_u32(codes);
        bool bad = false;
        for (int q = tid; q < npg * CPP; q += kThreads) {
            const int j = q / CPP, c = q % CPP;
            const int pg = __ldg(bt + pg0 + j);
            if (pg >= 0 && static_cast<int64_t>(pg) < p.num_pages)
                cp_async_16(dst0 + static_cast<uint32_t>(q) * 16u, src0 + static_cast<size_t>(pg) * page_stride + c * 16);
            else
                bad = true;
        }
        cp_async_mbar_arrive(&bar[2]);
        if (bad) atomicOr(&sflag[0], AQ_DEV_BAD_PAGE);
    }
    // ---- the query and the new token come from the preceding kernel ----------
    grid_dependency_wait();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[3], G * D * 4);
        bulk_g2s(qs, p.q + (static_cast<size_t>(b) * Hq + hq0) * D, G * D * 4, &bar[3]);
    }
    if constexpr (APPEND) {
        if (cl_new && tid < 2 * MC * DSUB) {
            const int w = tid / (MC * DSUB), r = tid % (MC * DSUB);
            xnew[tid] = __half2float(__ldg(reinterpret_cast<const __half *>(p.kv_new) +
                                           ((static_cast<size_t>(b) * p.qo_kv_heads + p.kv_head_base + kvh) * 2 + w) * D +
                                           rank * MC * DSUB + r));
        }
    }
    for (int i = tid; i < S::BIN_WORDS / 4; i += kThreads)
        reinterpret_cast<uint4 *>(bins)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < 2 * MC) keys[tid] = ~0ull;
    grid_launch_dependents();                          // every read of this CTA is issued
    __syncthreads();
    if constexpr (C > 1) cluster_arrive_relaxed();     // this CTA's barriers are ready for pushes

    // ---- lookup-table rows of the owned subspaces; the new key's codes -------
    bool tmo = !mbar_wait_limit(&bar[0], 0, p.wait_limit_ns);
    tmo |= !mbar_wait_limit(&bar[3], 0, p.wait_limit_ns);
    // a table built from a slice or query that had not landed reaches the
    // peers too: the flag travels with the rows
    if (tmo) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
    if constexpr (C > 1) cluster_wait_acquire();       // peers' barriers expect our pushes
    {
        float dkv[MC];
#pragma unroll
        for (int mi = 0; mi < MC; ++mi) {
            const int m = rank * MC + mi;
            const float *qm = qs + m * DSUB;
            const uint4 *rowk = reinterpret_cast<const uint4 *>(cbk) + (mi * K + tid) * NCH;
            unsigned long long acc2[G];
#pragma unroll
            for (int gg = 0; gg < G; ++gg) acc2[gg] = 0ull;
            float dk = 0.f;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                unsigned long long f[4];
                to_f2p4(rowk[chunk_pos<DSUB>(tid, c)], f);
#pragma unroll
                for (int gg = 0; gg < G; ++gg) {
                    const ulonglong2 *qv = reinterpret_cast<const ulonglong2 *>(qm + gg * D + c * 8);
                    const ulonglong2 qa = qv[0], qb = qv[1];
                    unsigned long long a = acc2[gg];
                    a = f2_fma(qa.x, f[0], a);
                    a = f2_fma(qa.y, f[1], a);
                    a = f2_fma(qb.x, f[2], a);
                    a = f2_fma(qb.y, f[3], a);
                    acc2[gg] = a;
                }
                if (APPEND && cl_new) dk = sqdist8(dk, xnew + mi * DSUB + c * 8, f);
            }
            float acc[G];
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                const float2 a = f2_unpack(acc2[gg]);
                acc[gg] = (a.x + a.y) * p.scale_log2;
            }
            if constexpr (G == 8) {
                float4 *row = reinterpret_cast<float4 *>(lut + (static_cast<size_t>(m) * K + tid) * G);
                const int h = lut_hswz<G>(tid);
                row[h] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                row[h ^ 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            } else {
                store_vec<G>(lut + (static_cast<size_t>(m) * K + tid) * G, acc);
            }
            dkv[mi] = dk;
        }
        if constexpr (APPEND) {
            if (cl_new) {
#pragma unroll
                for (int mi = 0; mi < MC; ++mi) warp_argmin_into(dkv[mi], &keys[mi]);
            }
        }
    }
    if constexpr (C > 1) fence_proxy_async_shared();  // the rows, for the bulk copies below
    __syncthreads();
    if constexpr (C > 1) {
        // this CTA's rows to every peer, one bulk copy each; the rows are not
        // written again in this launch
        if (tid < C - 1) {
            const uint32_t pr = static_cast<uint32_t>(rank + tid + 1) % C;
            const uint32_t rows = smem_u32(lut + rank * S::ROW_FLOATS);
            const uint32_t rbar = mapa_u32(smem_u32(&bar[4]), pr);
            bulk_s2cluster(mapa_u32(rows, pr), rows, S::ROW_FLOATS * 4, rbar);
            st_async_f32(mapa_u32(smem_u32(&pbad[rank]), pr), __int_as_float(sflag[0]), rbar);
        }
    }
    if constexpr (APPEND) {
        if (cl_new && tid < MC) {                      // the new key's code of subspace rank*MC + tid
            const int m = rank * MC + tid;
            const int code = static_cast<int>(keys[tid] & 0xffu);
            newc[m] = code;
            if constexpr (C > 1) {
                const uint32_t la = smem_u32(&newc[m]), lb = smem_u32(&bar[4]);
#pragma unroll
                for (int r = 1; r < C; ++r) {
                    const uint32_t pr = static_cast<uint32_t>(rank + r) % C;
                    st_async_f32(mapa_u32(la, pr), __int_as_float(code), mapa_u32(lb, pr));
                }
            }
        }
    }
    if constexpr (C > 1) tmo |= !mbar_wait_limit(&bar[4], 0, p.wait_limit_ns);
    tmo |= !mbar_wait_limit(&bar[2], 0, p.wait_limit_ns);
    if (tmo) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
    __syncthreads();                                   // the full table, the new key's codes
    if constexpr (C > 1) cluster_arrive_relaxed();     // everything sent to this CTA has landed

    // ---- scores and the split's softmax statistics ---------------------------
    // Every thread keeps the (max, sum) pair of its tokens online; the pairs
    // are merged over the lanes of head g and then over the warps (PAM article
    // §2.2.3 item 1), so mx and lsum -- the same in every CTA of the cluster --
    // are known before any weight is binned.
    if constexpr (S::PER_TOKEN) {
        // GQA group of 4 or 8: thread tid scores tokens tid, tid + 256, ... for
        // all G heads, one vector read of each table row per subspace.  The
        // max of each head over the warp comes from one redux, each thread's
        // weights are taken relative to it, and the warp's sums per head by a
        // butterfly that halves the heads a lane carries at each step; the
        // warps' (max, sum) pairs merge as on the other path (PAM article
        // §2.2.3 item 1), by the first G threads, between two barriers.
        constexpr int TT = S::TT, LG = G == 8 ? 3 : 2;
        float sc[TT][G];
        float mloc[G], sn[G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) mloc[gg] = sn[gg] = -INFINITY;
        if constexpr (APPEND) {
            if (cl_new && tid == 0) {
                unsigned long long a2[G / 2];
                lut_row2<G>(lut, newc[0], a2);
#pragma unroll
                for (int m = 1; m < M; ++m) {
                    unsigned long long r2[G / 2];
                    lut_row2<G>(lut, m * K + newc[m], r2);
#pragma unroll
                    for (int j = 0; j < G / 2; ++j) a2[j] = f2_add(a2[j], r2[j]);
                }
#pragma unroll
                for (int j = 0; j < G / 2; ++j) {
                    const float2 a = f2_unpack(a2[j]);
                    sn[2 * j] = mloc[2 * j] = a.x;
                    sn[2 * j + 1] = mloc[2 * j + 1] = a.y;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < TT; ++i) {
            const int r = tid + i * kThreads;
            if (r < ntok) {
                Codes<M> cw;
                cw.load_shared(codes + r * 2 * M);
                unsigned long long a2[G / 2];
                lut_row2<G>(lut, cw.k(0), a2);
#pragma unroll
                for (int m = 1; m < M; ++m) {
                    unsigned long long r2[G / 2];
                    lut_row2<G>(lut, m * K + cw.k(m), r2);
#pragma unroll
                    for (int j = 0; j < G / 2; ++j) a2[j] = f2_add(a2[j], r2[j]);
                }
#pragma unroll
                for (int j = 0; j < G / 2; ++j) {
                    const float2 a = f2_unpack(a2[j]);
                    sc[i][2 * j] = a.x;
                    sc[i][2 * j + 1] = a.y;
                }
#pragma unroll
                for (int gg = 0; gg < G; ++gg) mloc[gg] = fmaxf(mloc[gg], sc[i][gg]);
            } else {
#pragma unroll
                for (int gg = 0; gg < G; ++gg) sc[i][gg] = -INFINITY;
            }
        }
        float wmax[G], lw[G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            wmax[gg] = warp_max_f32(mloc[gg]);
            const float ref = wmax[gg] == -INFINITY ? 0.f : wmax[gg];
            float l = fast_exp2(sn[gg] - ref);              // the new token (thread 0), else 0
#pragma unroll
            for (int i = 0; i < TT; ++i) {
                sc[i][gg] = fast_exp2(sc[i][gg] - ref);     // 0 for an empty slot
                l += sc[i][gg];
            }
            lw[gg] = l;
        }
        // warp sums: at offset 16 >> t a lane keeps the upper or the lower half
        // of the heads it carries and adds its partner's copy of that half;
        // after LG steps lane carries head (lane >> (5 - LG)) & (G - 1), summed
        // over the lanes that agree with it in bits 5-LG .. 4
#pragma unroll
        for (int t = 0; t < LG; ++t) {
            const int off = 16 >> t, n = G >> t;
            const bool up = (lane & off) != 0;
#pragma unroll
            for (int j = 0; j < n / 2; ++j) {
                const float send = up ? lw[j] : lw[j + n / 2];
                const float keep = up ? lw[j + n / 2] : lw[j];
                lw[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
#pragma unroll
        for (int off = 16 >> LG; off > 0; off >>= 1) lw[0] += __shfl_xor_sync(0xffffffffu, lw[0], off);
        if (lane == 0) store_vec<G>(red_m + warp * G, wmax);
        if ((lane & ((32 >> LG) - 1)) == 0) red_l[warp * G + ((lane >> (5 - LG)) & (G - 1))] = lw[0];
        __syncthreads();
        if (tid < G) {
            float mx = red_m[tid];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, red_m[w * G + tid]);
            float lsum = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float mw = red_m[w * G + tid];
                if (mw != -INFINITY) lsum += red_l[w * G + tid] * (mw == mx ? 1.0f : fast_exp2(mw - mx));
            }
            // fixed-point value bins: round(p * 2^31 / lsum) per token and head
            st_mx[tid] = mx;
            st_l[tid] = lsum;
            st_c[tid] = lsum * (1.0f / 2147483648.0f);
            st_qs[tid] = lsum > 0.f ? __fdividef(2147483648.0f, lsum) : 0.f;
        }
        if (tid == 0) store_vec<G>(st_sn, sn);
        if constexpr (APPEND) {
            if (cl_new) {
                if (!mbar_wait_limit(&bar[1], 0, p.wait_limit_ns)) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
                encode_new_value<DSUB, MC, K, NCH>(cbv, xnew + MC * DSUB, keys + MC);
            }
        }
        __syncthreads();                               // statistics of every head
        float rq[G];
        {
            float mxv[G], qsv[G];
            load_vec<G>(mxv, st_mx);
            load_vec<G>(qsv, st_qs);
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
                rq[gg] = wmax[gg] == -INFINITY ? 0.f
                                               : (wmax[gg] == mxv[gg] ? qsv[gg] : fast_exp2(wmax[gg] - mxv[gg]) * qsv[gg]);
        }
#pragma unroll
        for (int i = 0; i < TT; ++i) {
            const int r = tid + i * kThreads;
            if (r < ntok) {
                Codes<M> cw;
                cw.load_shared(codes + r * 2 * M);
                unsigned qv[G];
#pragma unroll
                for (int gg = 0; gg < G; ++gg) qv[gg] = __float2uint_rn(sc[i][gg] * rq[gg]);
#pragma unroll
                for (int mi = 0; mi < MC; ++mi) {
                    const int v = cw.vv(rank * MC + mi);
                    const int sw = bin_wswz<G, S::KSQ>(v);
                    unsigned *row = bins + (mi * K + v) * G;
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) atomicAdd(row + (gg ^ sw), qv[gg]);
                }
            }
        }
    } else {
        const int g = tid % G, jslot = tid / G;
        float s_new = -INFINITY;
        if constexpr (APPEND) {
            if (cl_new && tid < G) {
                s_new = 0.f;
#pragma unroll
                for (int m = 0; m < M; ++m) s_new += lut[(m * K + newc[m]) * G + tid];
            }
        }
        const int nslot = (ntok + S::TOK_PER_PASS - 1) / S::TOK_PER_PASS;
        float sc[TPT];
        float mloc = s_new;
#pragma unroll
        for (int i = 0; i < TPT; ++i) {
            if (i >= nslot) break;
            const int r = jslot + i * S::TOK_PER_PASS;
            if (r < ntok) {
                Codes<M> cw;
                cw.load_shared(codes + r * 2 * M);
                float s = 0.f;
#pragma unroll
                for (int m = 0; m < M; ++m) s += lut[(m * K + cw.k(m)) * G + g];
                sc[i] = s;
                mloc = fmaxf(mloc, s);
            }
        }
        float lloc = (s_new != -INFINITY) ? fast_exp2(s_new - mloc) : 0.f;
#pragma unroll
        for (int i = 0; i < TPT; ++i) {
            if (i >= nslot) break;
            if (jslot + i * S::TOK_PER_PASS < ntok) {
                sc[i] = fast_exp2(sc[i] - mloc);
                lloc += sc[i];
            }
        }
        {
            float mt = mloc, lt = lloc;
#pragma unroll
            for (int off = G; off < 32; off <<= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, mt, off);
                const float l2 = __shfl_xor_sync(0xffffffffu, lt, off);
                const float mn = fmaxf(mt, m2);
                lt = (mt == mn ? lt : lt * fast_exp2(mt - mn)) + (m2 == mn ? l2 : l2 * fast_exp2(m2 - mn));
                mt = mn;
            }
            if (lane < G) {
                red_m[warp * G + lane] = mt;
                red_l[warp * G + lane] = lt;
            }
        }
        __syncthreads();
        float mx = red_m[g];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, red_m[w * G + g]);
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float mw = red_m[w * G + g];
            if (mw != -INFINITY) lsum += red_l[w * G + g] * (mw == mx ? 1.0f : fast_exp2(mw - mx));
        }
        // value bins in fixed point: round(p * 2^31 / lsum) per token; the bins of
        // one head sum to 2^31 (plus at most ntok/2 from rounding), and rounding
        // loses at most a relative ntok/2^32 of the weight
        const float qscale = lsum > 0.f ? __fdividef(2147483648.0f, lsum) : 0.f;
        const float cfac = lsum * (1.0f / 2147483648.0f);
        if (tid < G) {
            st_mx[tid] = mx;
            st_l[tid] = lsum;
            st_c[tid] = cfac;
            st_sn[tid] = s_new;
        }
        // the new token's value codes of the owned subspaces
        if constexpr (APPEND) {
            if (cl_new) {
                if (!mbar_wait_limit(&bar[1], 0, p.wait_limit_ns)) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
                float dv[MC];
#pragma unroll
                for (int mi = 0; mi < MC; ++mi) {
                    const uint4 *rowv = reinterpret_cast<const uint4 *>(cbv) + (mi * K + tid) * NCH;
                    float d = 0.f;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        unsigned long long f[4];
                        to_f2p4(rowv[chunk_pos<DSUB>(tid, c)], f);
                        d = sqdist8(d, xnew + (MC + mi) * DSUB + c * 8, f);
                    }
                    dv[mi] = d;
                }
#pragma unroll
                for (int mi = 0; mi < MC; ++mi) warp_argmin_into(dv[mi], &keys[MC + mi]);
            }
        }
        {
            const float rq = (mloc == -INFINITY) ? 0.f : (mloc == mx ? qscale : fast_exp2(mloc - mx) * qscale);
#pragma unroll
            for (int i = 0; i < TPT; ++i) {
                if (i >= nslot) break;
                const int r = jslot + i * S::TOK_PER_PASS;
                if (r < ntok) {
                    Codes<M> cw;
                    cw.load_shared(codes + r * 2 * M);
                    const unsigned qv = __float2uint_rn(sc[i] * rq);
#pragma unroll
                    for (int mi = 0; mi < MC; ++mi) atomicAdd(&bins[(mi * K + cw.vv(rank * MC + mi)) * G + g], qv);
                }
            }
        }
    }
    __syncthreads();                                   // bins, statistics, the new value codes
    int bad_all = sflag[0];
#pragma unroll
    for (int r = 0; r < C; ++r)
        if (r != rank) bad_all |= pbad[r];
    if constexpr (APPEND) {
        if (cl_new && tid == 0) {
            // this CTA's codes of the new token into its page slot
            if (sflag[0] & AQ_DEV_TIMEOUT) {
                // no codes from data that may not have landed
            } else if (pg_new >= 0 && static_cast<int64_t>(pg_new) < p.num_pages) {
                uint8_t *dst = p.code_pages_w + ((static_cast<size_t>(pg_new) * Hkv + kvh) * P + new_pos % P) * (2 * M);
#pragma unroll
                for (int mi = 0; mi < MC; ++mi) {
                    dst[rank * MC + mi] = static_cast<uint8_t>(newc[rank * MC + mi]);
                    dst[M + rank * MC + mi] = static_cast<uint8_t>(keys[MC + mi] & 0xffu);
                }
            } else {
                atomicOr(&sflag[0], AQ_DEV_BAD_PAGE);
                bad_all |= AQ_DEV_BAD_PAGE;
            }
        }
    }
    if (!mbar_wait_limit(&bar[1], 0, p.wait_limit_ns)) {
        atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
        bad_all |= AQ_DEV_TIMEOUT;
    }

    // ---- value codebook product for the owned dims -------------------------------
    {
        constexpr int NQ = MC * DSUB / 4, KSQ = kThreads / NQ, KSLQ = K / KSQ;
        constexpr int ROWS128 = 128 / (DSUB * 2);
        static_assert(KSQ % (ROWS128 * NCH) == 0, "row step keeps the swizzle position");
        const int qd = tid % NQ, ks = tid / NQ;
        const int mi = qd / (DSUB / 4), j4 = (qd % (DSUB / 4)) * 4;
        const int cj = j4 / 8, hj = j4 % 8;
        constexpr int VPX = S::VPX;
        const int kx = ks ^ ((mi * VPX) & (KSQ - 1));
        const __half *vrow = cbv + ((mi * K + kx) * NCH + chunk_pos<DSUB>(kx, cj)) * 8 + hj;
        const unsigned *wrow = bins + (static_cast<size_t>(mi) * K + kx) * G;
        unsigned long long acc[G][2];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) acc[gg][0] = acc[gg][1] = 0ull;
#pragma unroll 8
        for (int i = 0; i < KSLQ; ++i) {
            const uint2 cv2 = *reinterpret_cast<const uint2 *>(vrow + i * KSQ * NCH * 8);
            const unsigned long long c01 = h2_to_f2p(cv2.x), c23 = h2_to_f2p(cv2.y);
            unsigned wu[G];
            load_vec_u<G>(wu, wrow + i * KSQ * G);
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                const float wf = static_cast<float>(wu[gg]);
                const unsigned long long ww = f2_pack(wf, wf);
                acc[gg][0] = f2_fma(ww, c01, acc[gg][0]);
                acc[gg][1] = f2_fma(ww, c23, acc[gg][1]);
            }
        }
        float accf[G][4];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            const float2 a01 = f2_unpack(acc[gg][0]), a23 = f2_unpack(acc[gg][1]);
            accf[gg][0] = a01.x; accf[gg][1] = a01.y; accf[gg][2] = a23.x; accf[gg][3] = a23.y;
        }
        if constexpr (S::PER_TOKEN && !S::XU) {
            // this thread's rows agree in the bits of k below log2(KSQ), so one
            // permutation for all of them: word w of a row holds head w ^ x
            static_assert(KSQ == S::KSQ, "row step of the value product");
            const int x = bin_wswz<G, KSQ>(kx);
#pragma unroll
            for (int bv = 1; bv < G; bv <<= 1) {
                const bool sw = (x & bv) != 0;
#pragma unroll
                for (int gg = 0; gg < G; ++gg) {
                    if (gg & bv) continue;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a = accf[gg][e], c = accf[gg | bv][e];
                        accf[gg][e] = sw ? c : a;
                        accf[gg | bv][e] = sw ? a : c;
                    }
                }
            }
        }
#pragma unroll
        for (int off = NQ; off < 32; off <<= 1) {
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
#pragma unroll
                for (int e = 0; e < 4; ++e) accf[gg][e] += __shfl_xor_sync(0xffffffffu, accf[gg][e], off);
        }
        if (lane < NQ) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v[G];
#pragma unroll
                for (int gg = 0; gg < G; ++gg) v[gg] = accf[gg][e];
                store_vec<G>(part + (static_cast<size_t>(warp) * MC * DSUB + mi * DSUB + j4 + e) * G, v);
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < S::NOUT; i += kThreads) {
        const int gg = i % G, dl = i / G;                 // dl in [0, MC*DSUB)
        float o = 0.f;
        if constexpr (S::XU) {
            // warp w's partials hold head gg at word gg ^ x_w
            const int cx = ((dl / DSUB) * S::VPX) & (S::KSQ - 1);
#pragma unroll
            for (int w = 0; w < kWarps; ++w)
                o += part[static_cast<size_t>(w) * S::NOUT + dl * G + (gg ^ bin_wswz<G, S::KSQ>((w * 32 / S::NQ) ^ cx))];
        } else {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) o += part[static_cast<size_t>(w) * S::NOUT + i];
        }
        o *= st_c[gg];
        if constexpr (APPEND) {
            if (cl_new) {
                // the new token: its weight times its value codeword
                const int mi = dl / DSUB, j = dl % DSUB;
                const int vc = static_cast<int>(keys[MC + mi] & 0xffu);
                const float wn = fast_exp2(st_sn[gg] - st_mx[gg]);
                o += wn * __half2float(cbv[((mi * K + vc) * NCH + chunk_pos<DSUB>(vc, j / 8)) * 8 + j % 8]);
            }
        }
        const int d = rank * MC * DSUB + dl;
        const size_t bh = static_cast<size_t>(b) * Hq + hq0 + gg;
        const float nan = __int_as_float(0x7fc00000);
        if (S_ == 1) {
            const float l = st_l[gg];
            p.out[bh * D + d] = bad_all ? nan : (l > 0.f ? __fdividef(o, l) : 0.f);
        } else {
            p.part_o[(bh * S_ + split) * D + d] = o;
            if (rank == 0 && dl == 0) {
                p.part_ml[(bh * S_ + split) * 2 + 0] = bad_all ? nan : st_mx[gg];
                p.part_ml[(bh * S_ + split) * 2 + 1] = bad_all ? nan : st_l[gg];
            }
        }
    }
    if (tid == 0 && sflag[0]) flag_status(p.status, sflag[0]);
    // A wait that ran out may leave a copy still landing: wait again (bounded)
    // before the shared memory is released.
    if (sflag[0] & AQ_DEV_TIMEOUT) {
        cp_async_wait_all();
        for (int i = 0; i < 4; ++i) mbar_wait_bounded(&bar[i], 0);
        if constexpr (C > 1) mbar_wait_bounded(&bar[4], 0);
    }
    if constexpr (C > 1) cluster_wait_acquire();      // no CTA leaves while a peer may still read its rows
}

template <int M, int G, int C, bool APPEND>
cudaError_t launch_attend(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    using S = AtCfg<M, G, C>;
    auto kern = pq_attend_kernel<M, G, C, APPEND>;
    if (plan.split_len > S::MAX_SPLIT || plan.split_len % kPage) return cudaErrorInvalidValue;
    static SmemAttr attr_state;
    const size_t need = S::smem(plan.split_len);
    if (cudaError_t e = ensure_smem_attr(attr_state, reinterpret_cast<const void *>(kern), S::smem(S::MAX_SPLIT));
        e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C * plan.num_splits),
                       static_cast<unsigned>(p.num_kv_heads) << p.head_split_log2,
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

// ============================================================================
// pq_headsplit_kernel: the whole-split design with the query heads of the
// group, not the table work, divided over the cluster (GQA groups of G >= C,
// G >= 4; qwen-shaped B8 Hq64 Hkv8: C = 4, two query heads per CTA).
//
// One cluster of C CTAs per (request, kv head, split); CTA `rank` owns
// subspaces [rank*MC, (rank+1)*MC) of both codebooks and query heads
// [rank*H, (rank+1)*H), H = G/C:
//  1. table rows q_g[m] . C^K_m[k] for its own subspaces and all G heads (the
//     rows need every head's query, the codebook slice is this CTA's); each
//     peer receives the rows of its own heads only (AQPIM blog §4.1);
//  2. every token of the split scored for its H heads, so the (max, sum) of
//     each of them is complete in this CTA (PAM article §2.2.3 item 1);
//  3. fixed-point value bins of its heads for all M subspaces; each peer
//     receives the bins of the subspaces it owns and the heads' statistics
//     (PAM article §2.2.3 item 3, inside one cluster);
//  4. the value product W . C^V for its own subspaces and all G heads, as in
//     the other kernels; normalise and store, or store split partials.
// Against pq_attend_kernel (every CTA scores every token for all G heads),
// the table reads of the scores and the rows sent fall by C, at the price of
// a second exchange (bins) of MC*256*H words per peer.
// ============================================================================
template <int M, int G, int C>
struct HsCfg {
    static constexpr int D = kHeadDim, K = kCodewords, P = kPage;
    static constexpr int DSUB = D / M;
    static constexpr int NCH = DSUB / 8;
    static constexpr int MC = M / C;
    static constexpr int H = G / C;                         // query heads scored per CTA
    static constexpr int SLICE_BYTES = MC * K * DSUB * 2;
    static constexpr int T_FLOATS = M * K * H;              // table of this CTA's heads [M][K][H]
    static constexpr int SB_FLOATS = MC * K * H;            // rows for one peer [MC][K][H]
    static constexpr int B_WORDS = M * K * H;               // bins of this CTA's heads [M][K][H]
    static constexpr int RB_WORDS = MC * K * H;             // bins of one source [MC][K][H]
    static constexpr int STX_SENT = 4 * H + 1;              // mx, lsum, cfac, s_new of one rank's heads, its flags
    static constexpr int STX = 4 * H + 4;                   // one rank's row (16-byte multiple: vector accesses)
    static constexpr int TT = 4;                            // tokens per thread
    static constexpr int CODE_CAP = 32768;
    static constexpr int MAX_SPLIT = (TT * kThreads < CODE_CAP / (2 * M) ? TT * kThreads : CODE_CAP / (2 * M)) / P * P;
    static constexpr int NOUT = MC * DSUB * G;
    static constexpr int NQ = MC * DSUB / 4, KSQ = kThreads / NQ, KSLQ = K / KSQ;
    static constexpr int VPX = (M == 8 && C == 4) ? 2 : 1;
    // layout from the 1024-aligned base.  The peers' bins land in the key
    // slice (read for the last time before this CTA sends its rows, long
    // before any peer can have bins to send); the value-product partials use
    // the table (read for the last time by the scores).
    static constexpr int OFF_CBK = 0;
    static constexpr int OFF_RB = 0;                        // [C][MC][K][H] u32, slot rank unused
    static constexpr int OFF_CBV = SLICE_BYTES;
    static constexpr int OFF_T = 2 * SLICE_BYTES;
    static constexpr int OFF_PART = OFF_T;                  // [kWarps][NOUT]
    static constexpr int T_BYTES = (T_FLOATS > kWarps * NOUT ? T_FLOATS : kWarps * NOUT) * 4;
    static constexpr int OFF_SB = OFF_T + T_BYTES;          // [C][MC][K][H], slot rank unused
    static constexpr int OFF_B = OFF_SB + C * SB_FLOATS * 4;
    static constexpr int OFF_STX = OFF_B + B_WORDS * 4;     // [C][STX]
    static constexpr int OFF_Q = (OFF_STX + C * STX * 4 + 15) / 16 * 16;
    static constexpr int OFF_RED = OFF_Q + G * D * 4;       // red_m, red_l [kWarps][H]
    static constexpr int OFF_QS = OFF_RED + 2 * kWarps * H * 4;  // qscale [H]
    static constexpr int OFF_NEW = (OFF_QS + H * 4 + 15) / 16 * 16;  // xnew [2][MC][DSUB], newc [M]
    static constexpr int OFF_KEYS = (OFF_NEW + 2 * MC * DSUB * 4 + M * 4 + 7) / 8 * 8;
    static constexpr int OFF_BAR = OFF_KEYS + 2 * MC * 8;   // K, V, codes, q, rows, bins
    static constexpr int OFF_FLAG = OFF_BAR + 6 * 8;
    static constexpr int OFF_PBAD = OFF_FLAG + 16;
    static constexpr int OFF_CODES = (OFF_PBAD + 4 * C + 15) / 16 * 16;
    static size_t smem(int split_len) { return 1024 + OFF_CODES + static_cast<size_t>(split_len) * 2 * M; }
    static_assert(G >= C && G % C == 0 && G >= 4, "the group covers the cluster");
    static_assert(K == kThreads, "one thread per codeword in the table build");
    static_assert(SLICE_BYTES % 1024 == 0, "slices keep the swizzle alignment");
    static_assert(C * RB_WORDS * 4 <= SLICE_BYTES, "the peers' bins fit in the key slice");
    static_assert(OFF_T % 16 == 0 && OFF_SB % 16 == 0 && OFF_B % 16 == 0 && OFF_Q % 16 == 0, "alignment");
    static_assert(NQ <= 32 && 32 % NQ == 0, "V-product quads within a warp");
    static_assert(SB_FLOATS % 4 == 0 && RB_WORDS % 4 == 0, "bulk copies of 16-byte multiples");
    static_assert(MAX_SPLIT % kThreads == 0, "whole tokens per thread");
};

template <int H>
constexpr int kHsMinBlocks = 2;

// bins row of codeword k for the H heads of one CTA: head h at word h ^ s(k)
// (H = 2: s from bit 4 of k, H = 4: bits 3-4), so that the 32 tokens of an
// atomic spread over all banks; s uses bits of k below 5 only, fixed along the
// rows of one thread in the value product when its row step is 32 or more.
template <int H, int KSQ>
__device__ __forceinline__ int hs_bswz(int k) {
    if constexpr (H == 2 && KSQ >= 32) return (k >> 4) & 1;
    else if constexpr (H == 4 && KSQ >= 32) return (k >> 3) & 3;
    else return 0;
}

// An E4M3 slice landed raw (one byte per element, rows of DSUB bytes in the
// e8_pos layout) in the upper half of its fp16 buffer: widened exactly to fp16
// (E4M3 is a subset of fp16) into the buffer's swizzled fp16 layout.  Every
// thread reads its chunks first, a barrier, then writes (the halves overlap).
template <int DSUB, int MC>
__device__ __forceinline__ void widen_e4m3_slice(__half *buf) {
    constexpr int NE = DSUB / 16, NCH = DSUB / 8, ROWS = MC * kCodewords, PER = ROWS * NE / kThreads;
    static_assert(ROWS * NE % kThreads == 0, "whole chunks per thread");
    const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const unsigned char *>(buf) + ROWS * DSUB);
    uint4 raw[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int q = static_cast<int>(threadIdx.x) + i * kThreads, row = q / NE, e = q % NE;
        raw[i] = src[row * NE + e8_pos<DSUB>(row, e)];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int q = static_cast<int>(threadIdx.x) + i * kThreads, row = q / NE, e = q % NE;
        const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
        uint32_t h[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>((w[j / 2] >> (16 * (j % 2))) & 0xffffu), __NV_E4M3);
            h[j] = static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(buf) + row * NCH;
        dst[chunk_pos<DSUB>(row, 2 * e)] = make_uint4(h[0], h[1], h[2], h[3]);
        dst[chunk_pos<DSUB>(row, 2 * e + 1)] = make_uint4(h[4], h[5], h[6], h[7]);
    }
    __syncthreads();
}

template <int M, int G, int C, bool APPEND>
__global__ void __launch_bounds__(kThreads, kHsMinBlocks<G / C>) pq_headsplit_kernel(const __grid_constant__ DecodeParams p) {
    using S = HsCfg<M, G, C>;
    constexpr int D = S::D, K = S::K, P = S::P, DSUB = S::DSUB, MC = S::MC, NCH = S::NCH, H = S::H, TT = S::TT;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __half *cbk = reinterpret_cast<__half *>(smem + S::OFF_CBK);
    __half *cbv = reinterpret_cast<__half *>(smem + S::OFF_CBV);
    unsigned *rb = reinterpret_cast<unsigned *>(smem + S::OFF_RB);
    float *tab = reinterpret_cast<float *>(smem + S::OFF_T);
    float *part = reinterpret_cast<float *>(smem + S::OFF_PART);
    float *sb = reinterpret_cast<float *>(smem + S::OFF_SB);
    unsigned *bins = reinterpret_cast<unsigned *>(smem + S::OFF_B);
    float *stx = reinterpret_cast<float *>(smem + S::OFF_STX);
    float *qs = reinterpret_cast<float *>(smem + S::OFF_Q);
    float *red_m = reinterpret_cast<float *>(smem + S::OFF_RED);
    float *red_l = red_m + kWarps * H;
    float *qsc = reinterpret_cast<float *>(smem + S::OFF_QS);
    float *xnew = reinterpret_cast<float *>(smem + S::OFF_NEW);      // [2][MC][DSUB]
    int *newc = reinterpret_cast<int *>(xnew + 2 * MC * DSUB);        // [M]
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(smem + S::OFF_KEYS);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);  // K, V, codes, q, rows, bins
    int *sflag = reinterpret_cast<int *>(smem + S::OFF_FLAG);
    int *pbad = reinterpret_cast<int *>(smem + S::OFF_PBAD);
    const unsigned char *codes = smem + S::OFF_CODES;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = static_cast<int>(cluster_ctarank());
    const int split = blockIdx.x / C;
    const int kvh = static_cast<int>(blockIdx.y >> p.head_split_log2), b = blockIdx.z;
    const int hq0 = p.q_head_base + static_cast<int>(blockIdx.y) * G;
    const int Hq = p.num_q_heads, Hkv = p.num_kv_heads;
    const int S_ = p.num_splits;

    if (tid == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(&bar[i], i == 2 ? kThreads : 1);
        fence_mbar_init();
        sflag[0] = 0;
    }
    __syncthreads();
    // ---- reads allowed before the preceding kernel completes ----------------
    const int set = __ldg(p.req_set + b);
    const int L_raw = __ldg(p.seq_lens + b);
    const bool set_ok = set >= 0 && static_cast<int64_t>(set) < p.num_sets;
    int bad0 = 0;
    if (L_raw < 0 || L_raw > p.max_pages * P || L_raw > p.max_seq_len) bad0 |= AQ_DEV_BAD_LENGTH;
    if (!set_ok) bad0 |= AQ_DEV_BAD_SET;
    const int ts = split * p.split_len;
    const int te = bad0 ? ts : min(L_raw, ts + p.split_len);
    if (bad0 || ts >= te) {
        grid_dependency_wait();
        if (rank == 0) {
            if (bad0 && tid == 0) flag_status(p.status, bad0);
            const float v = bad0 ? __int_as_float(0x7fc00000) : 0.0f;
            for (int i = tid; i < G * D; i += kThreads) {
                const int gg = i / D, d = i % D;
                const size_t bh = static_cast<size_t>(b) * Hq + hq0 + gg;
                if (S_ == 1) p.out[bh * D + d] = v;
                else if (d == 0) {
                    p.part_ml[(bh * S_ + split) * 2 + 0] = bad0 ? v : -INFINITY;
                    p.part_ml[(bh * S_ + split) * 2 + 1] = bad0 ? v : 0.0f;
                }
            }
        }
        return;
    }
    const int new_pos = APPEND ? L_raw - 1 : -1;
    const bool cl_new = APPEND && new_pos >= ts && new_pos < te;
    const int ntok = (cl_new ? new_pos : te) - ts;
    const int32_t *bt = p.block_table + static_cast<size_t>(b) * p.max_pages;
    const int pg_new = (APPEND && cl_new && tid == 0) ? __ldg(bt + new_pos / P) : -1;
    // E4M3 codebooks: the raw slices (half the bytes) into the upper halves of
    // the fp16 buffers, widened there once they have landed
    const bool e8 = p.codebook_e4m3 != 0;
    if (tid == 0) {
        const int row0 = ((set * Hkv + kvh) * 2) * M * K + rank * MC * K;
        const uint32_t sl_bytes = e8 ? S::SLICE_BYTES / 2 : S::SLICE_BYTES;
        const int row_bytes = e8 ? DSUB : 2 * DSUB;
        unsigned char *kdst = reinterpret_cast<unsigned char *>(cbk) + (e8 ? S::SLICE_BYTES / 2 : 0);
        unsigned char *vdst = reinterpret_cast<unsigned char *>(cbv) + (e8 ? S::SLICE_BYTES / 2 : 0);
        mbar_arrive_expect_tx(&bar[0], sl_bytes);
#pragma unroll
        for (int mi = 0; mi < MC; ++mi) tma_load_2d(kdst + mi * K * row_bytes, &p.cb_map, 0, row0 + mi * K, &bar[0]);
        mbar_arrive_expect_tx(&bar[1], sl_bytes);
#pragma unroll
        for (int mi = 0; mi < MC; ++mi) tma_load_2d(vdst + mi * K * row_bytes, &p.cb_map, 0, row0 + M * K + mi * K, &bar[1]);
        // from each peer: its rows of this CTA's heads, its new-key codes and
        // flag; later its bins of this CTA's subspaces and its heads' statistics
        mbar_arrive_expect_tx(&bar[4], (C - 1) * (S::SB_FLOATS + (cl_new ? MC : 0) + 1) * 4);
        mbar_arrive_expect_tx(&bar[5], (C - 1) * (S::RB_WORDS + S::STX_SENT) * 4);
    }
    {
        // the split's code pages, whole page lines, into shared memory in token
        // order (as in pq_attend_kernel)
        constexpr int PAGE_BYTES = P * 2 * M, CPP = PAGE_BYTES / 16;
        const int npg = (ntok + P - 1) / P, pg0 = ts / P;
        const size_t page_stride = static_cast<size_t>(Hkv) * PAGE_BYTES;
        const unsigned char *src0 = p.code_pages + static_cast<size_t>(kvh) * PAGE_BYTES;
        const uint32_t dst0 = smem_u32(codes);
        bool bad = false;
        for (int q = tid; q < npg * CPP; q += kThreads) {
            const int j = q / CPP, c = q % CPP;
            const int pg = __ldg(bt + pg0 + j);
            if (pg >= 0 && static_cast<int64_t>(pg) < p.num_pages)
                cp_async_16(dst0 + static_cast<uint32_t>(q) * 16u, src0 + static_cast<size_t>(pg) * page_stride + c * 16);
            else
                bad = true;
        }
        cp_async_mbar_arrive(&bar[2]);
        if (bad) atomicOr(&sflag[0], AQ_DEV_BAD_PAGE);
    }
    // ---- the query and the new token come from the preceding kernel ----------
    grid_dependency_wait();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[3], G * D * 4);
        bulk_g2s(qs, p.q + (static_cast<size_t>(b) * Hq + hq0) * D, G * D * 4, &bar[3]);
    }
    if constexpr (APPEND) {
        if (cl_new && tid < 2 * MC * DSUB) {
            const int w = tid / (MC * DSUB), r = tid % (MC * DSUB);
            xnew[tid] = __half2float(__ldg(reinterpret_cast<const __half *>(p.kv_new) +
                                           ((static_cast<size_t>(b) * p.qo_kv_heads + p.kv_head_base + kvh) * 2 + w) * D +
                                           rank * MC * DSUB + r));
        }
    }
    for (int i = tid; i < S::B_WORDS / 4; i += kThreads)
        reinterpret_cast<uint4 *>(bins)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < 2 * MC) keys[tid] = ~0ull;
    grid_launch_dependents();
    __syncthreads();
    cluster_arrive_relaxed();                          // this CTA's barriers are ready for pushes

    // ---- table rows of the owned subspaces for all G heads --------------------
    bool tmo = !mbar_wait_limit(&bar[0], 0, p.wait_limit_ns);
    tmo |= !mbar_wait_limit(&bar[3], 0, p.wait_limit_ns);
    if (tmo) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
    if (e8) widen_e4m3_slice<DSUB, MC>(cbk);
    cluster_wait_acquire();                            // peers' barriers expect our pushes
    // Table rows on the tensor cores: D[k][g] = sum_d C^K_m[k][d] q_g[m][d]
    // for the owned subspaces, codebook rows by ldmatrix from the swizzled
    // slice, the queries as fp16 high and low parts (about 22 significant
    // bits), fp32 accumulation; warp w computes codewords [32w, 32w+32) for
    // all G heads, and each value goes to the CTA that owns its head.
    {
        static_assert(K == 32 * kWarps && DSUB % 16 == 0, "16x16 tiles, 32 codewords per warp");
        constexpr int KS = DSUB / 16, NT = (G + 7) / 8;
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int mi = 0; mi < MC; ++mi) {
            const int m = rank * MC + mi;
            const __half *ks_ = cbk + static_cast<size_t>(mi) * K * DSUB;
            float acc[2][NT][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
#pragma unroll
            for (int kst = 0; kst < KS; ++kst) {
                uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    // head n's query dims 2 tig + {0, 1} and + 8 of this 16-dim step
                    const int n = nt * 8 + gid;
                    float2 x0 = make_float2(0.f, 0.f), x1 = x0;
                    if (n < G) {
                        const float *qn = qs + n * D + m * DSUB + kst * 16 + 2 * tig;
                        x0 = *reinterpret_cast<const float2 *>(qn);
                        x1 = *reinterpret_cast<const float2 *>(qn + 8);
                    }
                    f16x2_split(x0.x, x0.y, bh[nt][0], bl[nt][0]);
                    f16x2_split(x1.x, x1.y, bh[nt][1], bl[nt][1]);
                }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    // rows 32 warp + 16 mt + l%8 (+8 for matrices 1, 3), chunk 2 kst (+1 for matrices 2, 3)
                    const int row = warp * 32 + mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                    const int c = 2 * kst + (lane >> 4);
                    uint32_t a[4];
                    ldsm_x4(smem_u32(ks_ + (row * NCH + chunk_pos<DSUB>(row, c)) * 8), a);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_16816(acc[mt][nt], a, bh[nt][0], bh[nt][1]);
                        mma_16816(acc[mt][nt], a, bl[nt][0], bl[nt][1]);
                    }
                }
            }
            // D fragment: codeword 32 warp + 16 mt + gid (+8), heads nt*8 + 2 tig + {0, 1}
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int k = warp * 32 + mt * 16 + gid + 8 * hf;
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int n = nt * 8 + 2 * tig + e;
                            if (n < G) {
                                const int r = n / H, h = n % H;
                                float *dst = r == rank ? tab + (static_cast<size_t>(m) * K + k) * H + h
                                                       : sb + (static_cast<size_t>(r * MC + mi) * K + k) * H + h;
                                *dst = acc[mt][nt][2 * hf + e] * p.scale_log2;
                            }
                        }
                    }
        }
        // the new key's codes: exact-rule distances, one thread per codeword
        if constexpr (APPEND) {
            if (cl_new) {
#pragma unroll
                for (int mi = 0; mi < MC; ++mi) {
                    float dk = 0.f;
                    for_row_chunks<DSUB, false>(cbk, mi * K + tid, [&](int c, const unsigned long long (&f)[4]) {
                        dk = sqdist8(dk, xnew + mi * DSUB + c * 8, f);
                    });
                    warp_argmin_into(dk, &keys[mi]);
                }
            }
        }
    }
    fence_proxy_async_shared();                        // the staged rows, for the bulk copies below
    __syncthreads();
    if (tid < C - 1) {
        // peer pr's rows (its heads, this CTA's subspaces) into its table
        const uint32_t pr = static_cast<uint32_t>(rank + tid + 1) % C;
        const uint32_t rbar = mapa_u32(smem_u32(&bar[4]), pr);
        bulk_s2cluster(mapa_u32(smem_u32(tab + static_cast<size_t>(rank) * MC * K * H), pr),
                       smem_u32(sb + static_cast<size_t>(pr) * S::SB_FLOATS), S::SB_FLOATS * 4, rbar);
        st_async_f32(mapa_u32(smem_u32(&pbad[rank]), pr), __int_as_float(sflag[0]), rbar);
    }
    if constexpr (APPEND) {
        if (cl_new && tid < MC) {
            const int m = rank * MC + tid;
            const int code = static_cast<int>(keys[tid] & 0xffu);
            newc[m] = code;
            const uint32_t la = smem_u32(&newc[m]), lb = smem_u32(&bar[4]);
#pragma unroll
            for (int r = 1; r < C; ++r) {
                const uint32_t pr = static_cast<uint32_t>(rank + r) % C;
                st_async_f32(mapa_u32(la, pr), __int_as_float(code), mapa_u32(lb, pr));
            }
        }
    }
    // the new token's value codes of the owned subspaces, while the peers' rows land
    bool v_wide = !e8;
    if constexpr (APPEND) {
        if (cl_new) {
            tmo |= !mbar_wait_limit(&bar[1], 0, p.wait_limit_ns);
            if (e8) widen_e4m3_slice<DSUB, MC>(cbv);
            v_wide = true;
            encode_new_value<DSUB, MC, K, NCH>(cbv, xnew + MC * DSUB, keys + MC);
        }
    }
    tmo |= !mbar_wait_limit(&bar[4], 0, p.wait_limit_ns);
    tmo |= !mbar_wait_limit(&bar[2], 0, p.wait_limit_ns);
    if (tmo) atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
    __syncthreads();                                   // the table of this CTA's heads, the new token's codes

    // ---- scores of this CTA's H heads over every token of the split ----------
    constexpr int LH = H == 8 ? 3 : (H == 4 ? 2 : (H == 2 ? 1 : 0));
    float sc[TT][H];
    float mloc[H], sn[H];
#pragma unroll
    for (int h = 0; h < H; ++h) mloc[h] = sn[h] = -INFINITY;
    if constexpr (APPEND) {
        if (cl_new && tid == 0) {
            float a[H];
            load_vec<H>(a, tab + static_cast<size_t>(newc[0]) * H);
#pragma unroll
            for (int m = 1; m < M; ++m) {
                float r[H];
                load_vec<H>(r, tab + (static_cast<size_t>(m) * K + newc[m]) * H);
#pragma unroll
                for (int h = 0; h < H; ++h) a[h] += r[h];
            }
#pragma unroll
            for (int h = 0; h < H; ++h) sn[h] = mloc[h] = a[h];
        }
    }
#pragma unroll
    for (int i = 0; i < TT; ++i) {
        const int r = tid + i * kThreads;
        if (r < ntok) {
            Codes<M> cw;
            cw.load_shared(codes + r * 2 * M);
            float a[H];
            load_vec<H>(a, tab + static_cast<size_t>(cw.k(0)) * H);
#pragma unroll
            for (int m = 1; m < M; ++m) {
                float t[H];
                load_vec<H>(t, tab + (static_cast<size_t>(m) * K + cw.k(m)) * H);
#pragma unroll
                for (int h = 0; h < H; ++h) a[h] += t[h];
            }
#pragma unroll
            for (int h = 0; h < H; ++h) {
                sc[i][h] = a[h];
                mloc[h] = fmaxf(mloc[h], a[h]);
            }
        } else {
#pragma unroll
            for (int h = 0; h < H; ++h) sc[i][h] = -INFINITY;
        }
    }
    // warp max of each head (one redux), weights relative to it, warp sums
    // by a butterfly that halves the heads a lane carries at each step
    float wmax[H], lw[H];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        wmax[h] = warp_max_f32(mloc[h]);
        const float ref = wmax[h] == -INFINITY ? 0.f : wmax[h];
        float l = fast_exp2(sn[h] - ref);                   // the new token (thread 0), else 0
#pragma unroll
        for (int i = 0; i < TT; ++i) {
            sc[i][h] = fast_exp2(sc[i][h] - ref);
            l += sc[i][h];
        }
        lw[h] = l;
    }
#pragma unroll
    for (int t = 0; t < LH; ++t) {
        const int off = 16 >> t, n = H >> t;
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < n / 2; ++j) {
            const float send = up ? lw[j] : lw[j + n / 2];
            const float keep = up ? lw[j + n / 2] : lw[j];
            lw[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int off = 16 >> LH; off > 0; off >>= 1) lw[0] += __shfl_xor_sync(0xffffffffu, lw[0], off);
    if (lane == 0) store_vec<H>(red_m + warp * H, wmax);
    if ((lane & ((32 >> LH) - 1)) == 0) red_l[warp * H + ((lane >> (5 - LH)) & (H - 1))] = lw[0];
    float *st_own = stx + rank * S::STX;               // mx, lsum, cfac, s_new [H] of this CTA's heads
    if (tid == 0) store_vec<H>(st_own + 3 * H, sn);
    __syncthreads();
    if (tid < H) {
        float mx = red_m[tid];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, red_m[w * H + tid]);
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float mw = red_m[w * H + tid];
            if (mw != -INFINITY) lsum += red_l[w * H + tid] * (mw == mx ? 1.0f : fast_exp2(mw - mx));
        }
        // fixed-point value bins: round(p * 2^31 / lsum) per token and head
        const float cf = lsum * (1.0f / 2147483648.0f);
        st_own[tid] = mx;
        st_own[H + tid] = lsum;
        st_own[2 * H + tid] = cf;
        qsc[tid] = lsum > 0.f ? __fdividef(2147483648.0f, lsum) : 0.f;
        const float snv = st_own[3 * H + tid];
        // this CTA's flags as they stand after its waits for the rows and
        // codes, with those the peers sent with their rows, go to every peer
        // with the statistics, and every CTA of the cluster NaNs its outputs
        // when any is set: a CTA whose wait gave up may send its bins early,
        // into a peer's key-slice buffer still being read, so the damage is not
        // confined to the heads of the CTA that flagged
        int fl = sflag[0];
#pragma unroll
        for (int r = 0; r < C; ++r)
            if (r != rank) fl |= pbad[r];
        const uint32_t lbar = smem_u32(&bar[5]);
#pragma unroll
        for (int r = 1; r < C; ++r) {
            const uint32_t pr = static_cast<uint32_t>(rank + r) % C, pb = mapa_u32(lbar, pr);
            st_async_f32(mapa_u32(smem_u32(st_own + tid), pr), mx, pb);
            st_async_f32(mapa_u32(smem_u32(st_own + H + tid), pr), lsum, pb);
            st_async_f32(mapa_u32(smem_u32(st_own + 2 * H + tid), pr), cf, pb);
            st_async_f32(mapa_u32(smem_u32(st_own + 3 * H + tid), pr), snv, pb);
            if (tid == 0) st_async_f32(mapa_u32(smem_u32(st_own + 4 * H), pr), __int_as_float(fl), pb);
        }
    }
    __syncthreads();                                   // statistics of this CTA's heads
    {
        float rq[H];
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const float mx = st_own[h], qv = qsc[h];
            rq[h] = wmax[h] == -INFINITY ? 0.f : (wmax[h] == mx ? qv : fast_exp2(wmax[h] - mx) * qv);
        }
#pragma unroll
        for (int i = 0; i < TT; ++i) {
            const int r = tid + i * kThreads;
            if (r < ntok) {
                Codes<M> cw;
                cw.load_shared(codes + r * 2 * M);
                unsigned qv[H];
#pragma unroll
                for (int h = 0; h < H; ++h) qv[h] = __float2uint_rn(sc[i][h] * rq[h]);
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const int v = cw.vv(m);
                    unsigned *row = bins + (m * K + v) * H;
                    const int sw = hs_bswz<H, S::KSQ>(v);
#pragma unroll
                    for (int h = 0; h < H; ++h) atomicAdd(row + (h ^ sw), qv[h]);
                }
            }
        }
    }
    fence_proxy_async_shared();                        // the bins, for the bulk copies below
    __syncthreads();
#ifdef AQ_DEBUG_CHECKS
    // the bin sums of every subspace agree for each head (each token adds one
    // weight per subspace) and stay below 2^31 + rounding
    if (tid < M * H) {
        const int m = tid / H, hd = tid % H;
        unsigned long long s0 = 0, sm = 0;
        for (int k = 0; k < K; ++k) {
            const int w = hd ^ hs_bswz<H, S::KSQ>(k);
            s0 += bins[k * H + w];
            sm += bins[(m * K + k) * H + w];
        }
        AQ_DCHECK(p.status, sm == s0 && s0 < 3ull * 1073741824ull);
    }
#endif
    if (tid < C - 1) {
        // peer pr's subspaces of this CTA's bins into its slot `rank`
        const uint32_t pr = static_cast<uint32_t>(rank + tid + 1) % C;
        bulk_s2cluster(mapa_u32(smem_u32(rb + static_cast<size_t>(rank) * S::RB_WORDS), pr),
                       smem_u32(bins + static_cast<size_t>(pr) * MC * K * H), S::RB_WORDS * 4,
                       mapa_u32(smem_u32(&bar[5]), pr));
    }
    int bad_all = sflag[0];
#pragma unroll
    for (int r = 0; r < C; ++r)
        if (r != rank) bad_all |= pbad[r];
    if (!mbar_wait_limit(&bar[5], 0, p.wait_limit_ns) || !mbar_wait_limit(&bar[1], 0, p.wait_limit_ns)) {
        atomicOr(&sflag[0], AQ_DEV_TIMEOUT);
        bad_all |= AQ_DEV_TIMEOUT;
    }
#pragma unroll
    for (int r = 0; r < C; ++r)
        if (r != rank) bad_all |= __float_as_int(stx[r * S::STX + 4 * H]);
    cluster_arrive_relaxed();                          // everything sent to this CTA has landed
    if (!v_wide) widen_e4m3_slice<DSUB, MC>(cbv);
    if constexpr (APPEND) {
        if (cl_new && tid == 0) {
            // this CTA's codes of the new token into its page slot
            if (sflag[0] & AQ_DEV_TIMEOUT) {
                // no codes from data that may not have landed
            } else if (pg_new >= 0 && static_cast<int64_t>(pg_new) < p.num_pages) {
                uint8_t *dst = p.code_pages_w + ((static_cast<size_t>(pg_new) * Hkv + kvh) * P + new_pos % P) * (2 * M);
#pragma unroll
                for (int mi = 0; mi < MC; ++mi) {
                    dst[rank * MC + mi] = static_cast<uint8_t>(newc[rank * MC + mi]);
                    dst[M + rank * MC + mi] = static_cast<uint8_t>(keys[MC + mi] & 0xffu);
                }
            } else {
                atomicOr(&sflag[0], AQ_DEV_BAD_PAGE);
                bad_all |= AQ_DEV_BAD_PAGE;
            }
        }
    }

    // ---- value codebook product for the owned dims, all G heads ---------------
    // A dense [dims x 256] . [256 x G] contraction per owned subspace, on the
    // tensor cores: D[d][g] = sum_k C^V[k][d] * W[k][g] / 2^31, C^V read
    // transposed from the swizzled slice by ldmatrix, the fixed-point bins W
    // as fp16 high and low parts (22 significant bits; each bin / 2^31 is at
    // most about 1), fp32 accumulation.  Warp w takes codewords [32w, 32w+32);
    // the warps' partial sums meet in the epilogue.
    {
        static_assert(K == 32 * kWarps, "32 codewords per warp");
        static_assert(DSUB % 16 == 0, "16-dim tiles");
        constexpr int MT = DSUB / 16, NT = (G + 7) / 8;
        const int gid = lane >> 2, tig = lane & 3;
        float acc[MC][MT][NT][4];
#pragma unroll
        for (int mi = 0; mi < MC; ++mi)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[mi][mt][nt][e] = 0.f;
#pragma unroll
        for (int mi = 0; mi < MC; ++mi) {
            const __half *vs = cbv + static_cast<size_t>(mi) * K * DSUB;
#pragma unroll
            for (int kstep = 0; kstep < 2; ++kstep) {
                const int k0 = warp * 32 + kstep * 16;
                uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    // head n's bins of codewords k0 + 2 tig + {0, 1} and + 8
                    const int n = nt * 8 + gid, src = n / H, hh = n % H;
                    const unsigned *wb = src == rank ? bins + static_cast<size_t>(rank * MC + mi) * K * H
                                                     : rb + static_cast<size_t>(src * MC + mi) * K * H;
                    float w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int k = k0 + 2 * tig + (j & 1) + (j >> 1) * 8;
                        w[j] = n < G ? static_cast<float>(wb[k * H + (hh ^ hs_bswz<H, S::KSQ>(k))]) * (1.0f / 2147483648.0f)
                                     : 0.f;
                    }
                    f16x2_split(w[0], w[1], bh[nt][0], bl[nt][0]);
                    f16x2_split(w[2], w[3], bh[nt][1], bl[nt][1]);
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    // rows k0 + l%8 (+8 for matrices 2, 3), 8-dim chunk 2 mt (+1 for matrices 1, 3)
                    const int kr = k0 + (lane & 7) + ((lane >> 4) << 3);
                    const int c = 2 * mt + ((lane >> 3) & 1);
                    uint32_t a[4];
                    ldsm_x4_trans(smem_u32(vs + (kr * NCH + chunk_pos<DSUB>(kr, c)) * 8), a);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_16816(acc[mi][mt][nt], a, bh[nt][0], bh[nt][1]);
                        mma_16816(acc[mi][mt][nt], a, bl[nt][0], bl[nt][1]);
                    }
                }
            }
        }
        // D fragment: (dim gid, heads 2 tig, 2 tig + 1) and (dim gid + 8, same heads)
#pragma unroll
        for (int mi = 0; mi < MC; ++mi)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int n = nt * 8 + 2 * tig;
                    if (n < G) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const int dl = mi * DSUB + mt * 16 + gid + 8 * hf;
                            *reinterpret_cast<float2 *>(part + (static_cast<size_t>(warp) * MC * DSUB + dl) * G + n) =
                                make_float2(acc[mi][mt][nt][2 * hf], acc[mi][mt][nt][2 * hf + 1]);
                        }
                    }
                }
    }
    __syncthreads();
    for (int i = tid; i < S::NOUT; i += kThreads) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) o += part[static_cast<size_t>(w) * S::NOUT + i];
        const int gg = i % G, dl = i / G;                 // dl in [0, MC*DSUB)
        const float *sth = stx + (gg / H) * S::STX;       // statistics of head gg, from its CTA
        const int hh = gg % H;
        const float mxg = sth[hh], lg = sth[H + hh];
        o *= sth[2 * H + hh] * 2147483648.0f;         // the product's bins were scaled by 2^-31
        if constexpr (APPEND) {
            if (cl_new) {
                // the new token: its weight times its value codeword
                const int mi = dl / DSUB, j = dl % DSUB;
                const int vc = static_cast<int>(keys[MC + mi] & 0xffu);
                const float wn = fast_exp2(sth[3 * H + hh] - mxg);
                o += wn * __half2float(cbv[((mi * K + vc) * NCH + chunk_pos<DSUB>(vc, j / 8)) * 8 + j % 8]);
            }
        }
        const int d = rank * MC * DSUB + dl;
        const size_t bh = static_cast<size_t>(b) * Hq + hq0 + gg;
        const float nan = __int_as_float(0x7fc00000);
        if (S_ == 1) {
            p.out[bh * D + d] = bad_all ? nan : (lg > 0.f ? __fdividef(o, lg) : 0.f);
        } else {
            p.part_o[(bh * S_ + split) * D + d] = o;
            if (rank == 0 && dl == 0) {
                p.part_ml[(bh * S_ + split) * 2 + 0] = bad_all ? nan : mxg;
                p.part_ml[(bh * S_ + split) * 2 + 1] = bad_all ? nan : lg;
            }
        }
    }
    if (tid == 0 && sflag[0]) flag_status(p.status, sflag[0]);
    // A wait that ran out may leave a copy still landing: wait again (bounded)
    // before the shared memory is released.
    if (sflag[0] & AQ_DEV_TIMEOUT) {
        cp_async_wait_all();
        for (int i = 0; i < 6; ++i) mbar_wait_bounded(&bar[i], 0);
    }
    cluster_wait_acquire();                            // no CTA leaves while a peer may still read its rows or bins
}

template <int M, int G, int C, bool APPEND>
cudaError_t launch_headsplit(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    using S = HsCfg<M, G, C>;
    auto kern = pq_headsplit_kernel<M, G, C, APPEND>;
    if (plan.split_len > S::MAX_SPLIT || plan.split_len % kPage) return cudaErrorInvalidValue;
    static SmemAttr attr_state;
    const size_t need = S::smem(plan.split_len);
    // Shared memory for two resident CTAs per SM, the rest as L1: the launch
    // is one wave at two per SM, and a third CTA (the next launch's, under
    // programmatic dependent launch) only competes with the running ones
    // (measured on qwen_gqa: 10.5 us per step with three, 9.6 with two).
    constexpr size_t kSmPerSM = 233472;                // 228 KiB
    const int pct = static_cast<int>((2 * (S::smem(S::MAX_SPLIT) + 1024) * 100 + kSmPerSM - 1) / kSmPerSM);
    if (cudaError_t e = ensure_smem_attr(attr_state, reinterpret_cast<const void *>(kern), S::smem(S::MAX_SPLIT),
                                         pct < 100 ? pct : 100);
        e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C * plan.num_splits),
                       static_cast<unsigned>(p.num_kv_heads) << p.head_split_log2,
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

// Groups that cover the cluster (G >= C, G >= 4) split their query heads over
// it (pq_headsplit_kernel); smaller groups score all heads in every CTA.
template <int G, int C>
constexpr bool kHeadSplit = G >= 4 && G >= C;

template <int M, int G, int C, bool APPEND>
cudaError_t attend_one(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    if constexpr (kHeadSplit<G, C>) return launch_headsplit<M, G, C, APPEND>(p, plan, s);
    else if (p.codebook_e4m3) return cudaErrorInvalidValue;   // fp16 slices only
    else return launch_attend<M, G, C, APPEND>(p, plan, s);
}

template <int M, int G, int C>
size_t attend_smem(int split_len) {
    if constexpr (kHeadSplit<G, C>) return HsCfg<M, G, C>::smem(split_len);
    else return AtCfg<M, G, C>::smem(split_len);
}

template <int M, int G, bool APPEND>
cudaError_t attend_c(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    switch (plan.cluster) {
        case 2: return attend_one<M, G, 2, APPEND>(p, plan, s);
        case 4: return attend_one<M, G, 4, APPEND>(p, plan, s);
        case 8:
            if constexpr (M == 8) return attend_one<M, G, 8, APPEND>(p, plan, s);
            else return cudaErrorInvalidConfiguration;
        default: return cudaErrorInvalidConfiguration;
    }
}

template <int M, bool APPEND>
cudaError_t attend_g(const DecodeParams &p, int G, const Plan &plan, cudaStream_t s) {
    switch (G) {
        case 1: return attend_c<M, 1, APPEND>(p, plan, s);
        case 2: return attend_c<M, 2, APPEND>(p, plan, s);
        case 4: return attend_c<M, 4, APPEND>(p, plan, s);
        case 8: return attend_c<M, 8, APPEND>(p, plan, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

// Shares of several chunks stream in two passes; that instantiation exists
// for fp16 codebooks and clusters of 4 or 8 (the planner keeps other shares to
// one chunk).
template <int C, bool E4M3>
constexpr bool kStreams = !E4M3 && C >= 4;

template <int M, int G, int C, bool APPEND, bool E4M3, bool STREAM>
cudaError_t launch_kernel(const DecodeParams &p, const Plan &plan, cudaStream_t s);

template <int M, int G, int C, bool APPEND, bool E4M3>
cudaError_t launch_one(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    using S = PqCfg<M, G, C>;
    if (plan.share % kPage) return cudaErrorInvalidValue;
    if (plan.share > S::MAX_SHARE) {
        if constexpr (kStreams<C, E4M3>) {
            if (plan.share > S::MAX_SHARE * kMaxChunks) return cudaErrorInvalidValue;
            return launch_kernel<M, G, C, APPEND, E4M3, true>(p, plan, s);
        } else {
            return cudaErrorInvalidValue;
        }
    }
    return launch_kernel<M, G, C, APPEND, E4M3, false>(p, plan, s);
}

template <int M, int G, int C, bool APPEND, bool E4M3, bool STREAM>
cudaError_t launch_kernel(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    using S = PqCfg<M, G, C>;
    auto kern = pq_decode_kernel<M, G, C, APPEND, E4M3, STREAM>;
    static SmemAttr attr_state;                    // opt-in dynamic shared memory, per device
    const size_t need = S::smem();
    if (cudaError_t e = ensure_smem_attr(attr_state, reinterpret_cast<const void *>(kern), need); e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C * plan.num_splits),
                       static_cast<unsigned>(p.num_kv_heads) << p.head_split_log2,
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

template <int M, int G, bool APPEND, bool E4M3>
cudaError_t dispatch_c(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    switch (plan.cluster) {
        case 1: return launch_one<M, G, 1, APPEND, E4M3>(p, plan, s);
        case 2: return launch_one<M, G, 2, APPEND, E4M3>(p, plan, s);
        case 4: return launch_one<M, G, 4, APPEND, E4M3>(p, plan, s);
        case 8:                                    // one subspace per CTA
            if constexpr (M == 8) return launch_one<M, G, 8, APPEND, E4M3>(p, plan, s);
            else return cudaErrorInvalidConfiguration;
        default: return cudaErrorInvalidConfiguration;
    }
}

template <int M, bool APPEND, bool E4M3>
cudaError_t dispatch_g(const DecodeParams &p, int G, const Plan &plan, cudaStream_t s) {
    switch (G) {
        case 1: return dispatch_c<M, 1, APPEND, E4M3>(p, plan, s);
        case 2: return dispatch_c<M, 2, APPEND, E4M3>(p, plan, s);
        case 4: return dispatch_c<M, 4, APPEND, E4M3>(p, plan, s);
        case 8: return dispatch_c<M, 8, APPEND, E4M3>(p, plan, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

template <int M>
size_t smem_g(int G, int C) {
#define AQ_SM(GG, CC) \
    if (G == GG && C == CC) return PqCfg<M, GG, CC>::smem();
    AQ_SM(1, 1) AQ_SM(1, 2) AQ_SM(1, 4)
    AQ_SM(2, 1) AQ_SM(2, 2) AQ_SM(2, 4)
    AQ_SM(4, 1) AQ_SM(4, 2) AQ_SM(4, 4)
    AQ_SM(8, 1) AQ_SM(8, 2) AQ_SM(8, 4)
#undef AQ_SM
    if constexpr (M == 8) {
        if (C == 8 && G == 1) return PqCfg<M, 1, 8>::smem();
        if (C == 8 && G == 2) return PqCfg<M, 2, 8>::smem();
        if (C == 8 && G == 4) return PqCfg<M, 4, 8>::smem();
        if (C == 8 && G == 8) return PqCfg<M, 8, 8>::smem();
    }
    return 0;
}

}  // namespace

size_t pq_decode_smem_bytes(int M, int G, int cluster) {
    if (M == 4) return smem_g<4>(G, cluster);
    if (M == 8) return smem_g<8>(G, cluster);
    return 0;
}

size_t pq_attend_smem_bytes(int M, int G, int cluster, int split_len) {
#define AQ_AS(MM, GG, CC) \
    if (M == MM && G == GG && cluster == CC) return attend_smem<MM, GG, CC>(split_len);
    AQ_AS(4, 1, 2) AQ_AS(4, 1, 4) AQ_AS(4, 2, 2) AQ_AS(4, 2, 4) AQ_AS(4, 4, 2) AQ_AS(4, 4, 4) AQ_AS(4, 8, 2) AQ_AS(4, 8, 4)
    AQ_AS(8, 1, 2) AQ_AS(8, 1, 4) AQ_AS(8, 1, 8) AQ_AS(8, 2, 2) AQ_AS(8, 2, 4) AQ_AS(8, 2, 8)
    AQ_AS(8, 4, 2) AQ_AS(8, 4, 4) AQ_AS(8, 4, 8) AQ_AS(8, 8, 2) AQ_AS(8, 8, 4) AQ_AS(8, 8, 8)
#undef AQ_AS
    return 0;
}

int pq_attend_max_split(int M, int G) {
#define AQ_AM(MM, GG) \
    if (M == MM && G == GG) return AtCfg<MM, GG, 2>::MAX_SPLIT;
    AQ_AM(4, 1) AQ_AM(4, 2) AQ_AM(4, 4) AQ_AM(4, 8) AQ_AM(8, 1) AQ_AM(8, 2) AQ_AM(8, 4) AQ_AM(8, 8)
#undef AQ_AM
    return 0;
}

int pq_decode_max_share(int M, int G) {
#define AQ_MS(MM, GG) \
    if (M == MM && G == GG) return PqCfg<MM, GG, 1>::MAX_SHARE;
    AQ_MS(4, 1) AQ_MS(4, 2) AQ_MS(4, 4) AQ_MS(4, 8)
    AQ_MS(8, 1) AQ_MS(8, 2) AQ_MS(8, 4) AQ_MS(8, 8)
#undef AQ_MS
    return 0;
}

cudaError_t launch_pq_decode(const DecodeParams &p, int M, int G, const Plan &plan, cudaStream_t s) {
    cudaError_t e;
    G /= plan.head_split;                          // query heads per cluster
    if (p.codebook_e4m3) return cudaErrorInvalidValue;          // E4M3 codebooks: the fused step only
    if (plan.kernel == 2) e = M == 4 ? attend_g<4, false>(p, G, plan, s) : attend_g<8, false>(p, G, plan, s);
    else if (M == 4) e = dispatch_g<4, false, false>(p, G, plan, s);
    else if (M == 8) e = dispatch_g<8, false, false>(p, G, plan, s);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    if (plan.num_splits > 1) return launch_combine(p, p.num_kv_heads * G * plan.head_split, s);
    return cudaSuccess;
}

cudaError_t launch_pq_decode_step(const DecodeParams &p, int M, int G, const Plan &plan, cudaStream_t s) {
    cudaError_t e;
    G /= plan.head_split;
    if (plan.kernel == 2)           // E4M3 codebooks only in the head-split kernel (the planner's choice)
        e = M == 4 ? attend_g<4, true>(p, G, plan, s) : attend_g<8, true>(p, G, plan, s);
    else if (M == 4) e = p.codebook_e4m3 ? dispatch_g<4, true, true>(p, G, plan, s) : dispatch_g<4, true, false>(p, G, plan, s);
    else if (M == 8) e = p.codebook_e4m3 ? dispatch_g<8, true, true>(p, G, plan, s) : dispatch_g<8, true, false>(p, G, plan, s);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    if (plan.num_splits > 1) return launch_combine(p, p.num_kv_heads * G * plan.head_split, s);
    return cudaSuccess;
}

cudaError_t launch_combine(const DecodeParams &p, int num_q_heads_launch, cudaStream_t s) {
    combine_kernel<<<dim3(static_cast<unsigned>(num_q_heads_launch), static_cast<unsigned>(p.batch)), 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace aq
