// decode_fp16.cu -- the uncompressed comparison point: paged decode attention
// over an fp16 K/V cache (AQPIM blog §2.1 cache layout, B*H*D*2*2 bytes per
// token), with the same split-KV partials and combine as the PQ path (PAM
// article §2.2.3).
//
// One CTA per (request, kv head, split); each of its 8 warps streams whole
// 16-token pages (4 KiB of keys, 4 KiB of values) with 8-byte loads, lane l
// holding dims [4l, 4l+4).  Scores are warp all-reduced dot products; every
// warp keeps its own running (max, sum, acc) per query head of the GQA group;
// the 8 warp states are merged in shared memory at the end.  With APPEND (the
// fp16 heads of a mixed-precision step) the CTA whose split holds position
// seq_lens[b] - 1 writes the new key and value into that page slot and its
// page's warp scores them from kv_new directly.
#include "common.cuh"
#include "internal.h"

namespace aq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float4 h4_to_f4(uint2 u) {
    const float2 a = h2_to_f2(u.x), b = h2_to_f2(u.y);
    return make_float4(a.x, a.y, b.x, b.y);
}

template <int G, bool APPEND>
__global__ void __launch_bounds__(kThreads) fp16_decode_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int D = kHeadDim, P = kPage;
    extern __shared__ __align__(16) unsigned char smem[];
    float *wm = reinterpret_cast<float *>(smem);          // [kWarps][G]
    float *wl = wm + kWarps * G;                          // [kWarps][G]
    float *wacc = wl + kWarps * G;                        // [kWarps][G][D]
    int *sbad = reinterpret_cast<int *>(wacc + kWarps * G * D);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int Hq = p.num_q_heads, Hkv = p.num_kv_heads, S_ = p.num_splits;

    const int L_raw = p.seq_lens[b];
    int bad0 = 0;
    if (L_raw < 0 || L_raw > p.max_pages * P || L_raw > p.max_seq_len) bad0 |= AQ_DEV_BAD_LENGTH;
    const int ts = split * p.split_len;
    const int te = bad0 ? ts : min(L_raw, ts + p.split_len);
    if (bad0 || ts >= te) {
        // launched as a programmatic dependent (mixed step): finish after the
        // preceding kernel, so that stream order holds for what follows
        grid_dependency_wait();
        if (bad0 && tid == 0) flag_status(p.status, bad0);
        const float v = bad0 ? __int_as_float(0x7fc00000) : 0.0f;
        for (int i = tid; i < G * D; i += kThreads) {
            const int g = i / D, d = i % D;
            const size_t bh = static_cast<size_t>(b) * Hq + p.q_head_base + kvh * G + g;
            if (S_ == 1) p.out[bh * D + d] = v;
            else if (d == 0) {
                p.part_ml[(bh * S_ + split) * 2 + 0] = bad0 ? v : -INFINITY;
                p.part_ml[(bh * S_ + split) * 2 + 1] = bad0 ? v : 0.0f;
            }
        }
        return;
    }
    if (tid == 0) *sbad = 0;
    const int32_t *bt = p.block_table + static_cast<size_t>(b) * p.max_pages;
    // the fused step's new token (position L-1), this lane's dims of its key
    // and value; the page slot is written by warp 0 and read by nobody here
    const int new_pos = APPEND ? L_raw - 1 : -1;
    const bool own_new = APPEND && new_pos >= ts && new_pos < te;
    uint2 knew = make_uint2(0u, 0u), vnew = knew;
    if (own_new) {
        const uint2 *src = reinterpret_cast<const uint2 *>(p.kv_new) +
                           (static_cast<size_t>(b) * p.qo_kv_heads + p.kv_head_base + kvh) * 2 * (D / 4);
        knew = src[lane];
        vnew = src[D / 4 + lane];
        const int pgn = bt[new_pos / P];
        if (warp == 0 && pgn >= 0 && static_cast<int64_t>(pgn) < p.num_pages) {
            uint2 *dst = reinterpret_cast<uint2 *>(const_cast<void *>(p.kv_pages)) +
                         ((static_cast<size_t>(pgn) * Hkv + kvh) * 2 * P + static_cast<size_t>(new_pos % P)) * (D / 4);
            dst[lane] = knew;
            dst[static_cast<size_t>(P) * (D / 4) + lane] = vnew;
        }
    }

    // this lane's query slice, pre-scaled into the log2 domain
    float4 qv[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float4 t = *reinterpret_cast<const float4 *>(
            p.q + (static_cast<size_t>(b) * Hq + p.q_head_base + static_cast<size_t>(kvh) * G + g) * D + 4 * lane);
        qv[g] = make_float4(t.x * p.scale_log2, t.y * p.scale_log2, t.z * p.scale_log2,
                            t.w * p.scale_log2);
    }
    float m_w[G], l_w[G];
    float4 acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m_w[g] = -INFINITY;
        l_w[g] = 0.f;
        acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();

    const int pg0 = ts / P, pg1 = (te + P - 1) / P;
    int badpage = 0;
#pragma unroll 1
    for (int pi = pg0 + warp; pi < pg1; pi += kWarps) {
        const int pg = bt[pi];
        if (pg < 0 || static_cast<int64_t>(pg) >= p.num_pages) {
            badpage = 1;
            continue;
        }
        const int n = min(P, te - pi * P);
        const __half *kp = reinterpret_cast<const __half *>(p.kv_pages) +
                           ((static_cast<size_t>(pg) * Hkv + kvh) * 2) * P * D + 4 * lane;
        const __half *vp = kp + static_cast<size_t>(P) * D;
        uint2 kr[P], vr[P];
#pragma unroll
        for (int t = 0; t < P; ++t) {
            kr[t] = ldg_stream_v2(kp + t * D);
            vr[t] = ldg_stream_v2(vp + t * D);
        }
        if (APPEND && own_new && pi == new_pos / P) {
            const int tn = new_pos % P;
#pragma unroll
            for (int t = 0; t < P; ++t)
                if (t == tn) {
                    kr[t] = knew;
                    vr[t] = vnew;
                }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float s[P];
#pragma unroll
            for (int t = 0; t < P; ++t) {
                const float4 k = h4_to_f4(kr[t]);
                float x = qv[g].x * k.x;
                x = fmaf(qv[g].y, k.y, x);
                x = fmaf(qv[g].z, k.z, x);
                x = fmaf(qv[g].w, k.w, x);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
                s[t] = (t < n) ? x : -INFINITY;
            }
            float mx = m_w[g];
#pragma unroll
            for (int t = 0; t < P; ++t) mx = fmaxf(mx, s[t]);
            const float alpha = exp2f(m_w[g] - mx);    // 0 on the first page
            float l = l_w[g] * alpha;
            float4 a = make_float4(acc[g].x * alpha, acc[g].y * alpha, acc[g].z * alpha,
                                   acc[g].w * alpha);
#pragma unroll
            for (int t = 0; t < P; ++t) {
                const float pv = exp2f(s[t] - mx);        // 0 for masked tokens
                const float4 v = h4_to_f4(vr[t]);
                l += pv;
                a.x = fmaf(pv, v.x, a.x);
                a.y = fmaf(pv, v.y, a.y);
                a.z = fmaf(pv, v.z, a.z);
                a.w = fmaf(pv, v.w, a.w);
            }
            m_w[g] = mx;
            l_w[g] = l;
            acc[g] = a;
        }
    }
    if (badpage) atomicOr(sbad, AQ_DEV_BAD_PAGE);
    // ---- merge the warps ----------------------------------------------------
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (lane == 0) {
            wm[warp * G + g] = m_w[g];
            wl[warp * G + g] = l_w[g];
        }
        *reinterpret_cast<float4 *>(wacc + (warp * G + g) * D + 4 * lane) = acc[g];
    }
    __syncthreads();
    grid_dependency_wait();                            // (as above)
    const int bad = *sbad;
    if (bad && tid == 0) flag_status(p.status, bad);
    for (int i = tid; i < G * D; i += kThreads) {
        const int g = i / D, d = i % D;
        float ms = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            if (wl[w * G + g] > 0.f) ms = fmaxf(ms, wm[w * G + g]);
        float o = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float lw = wl[w * G + g];
            if (lw > 0.f) {
                const float f = exp2f(wm[w * G + g] - ms);
                l += f * lw;
                o += f * wacc[(w * G + g) * D + d];
            }
        }
        const size_t bh = static_cast<size_t>(b) * Hq + p.q_head_base + static_cast<size_t>(kvh) * G + g;
        const float nan = __int_as_float(0x7fc00000);
        if (S_ == 1) {
            p.out[bh * D + d] = bad ? nan : (l > 0.f ? o / l : 0.f);
        } else {
            p.part_o[(bh * S_ + split) * D + d] = o;
            if (d == 0) {
                p.part_ml[(bh * S_ + split) * 2 + 0] = bad ? nan : ms;
                p.part_ml[(bh * S_ + split) * 2 + 1] = bad ? nan : l;
            }
        }
    }
}

template <int G, bool APPEND>
cudaError_t launch_g(const DecodeParams &p, const Plan &plan, cudaStream_t s) {
    const size_t smem = (2 * kWarps * G + kWarps * G * kHeadDim) * sizeof(float) + 16;
    auto kern = fp16_decode_kernel<G, APPEND>;
    static SmemAttr attr_state;                    // opt-in dynamic shared memory, per device
    if (cudaError_t e = ensure_smem_attr(attr_state, reinterpret_cast<const void *>(kern), smem); e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.num_splits), static_cast<unsigned>(p.num_kv_heads),
                       static_cast<unsigned>(p.batch));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_fp16_decode(const DecodeParams &p, int G, const Plan &plan, cudaStream_t s) {
    cudaError_t e;
    const bool app = p.kv_new != nullptr;
    switch (G) {
        case 1: e = app ? launch_g<1, true>(p, plan, s) : launch_g<1, false>(p, plan, s); break;
        case 2: e = app ? launch_g<2, true>(p, plan, s) : launch_g<2, false>(p, plan, s); break;
        case 4: e = app ? launch_g<4, true>(p, plan, s) : launch_g<4, false>(p, plan, s); break;
        case 8: e = app ? launch_g<8, true>(p, plan, s) : launch_g<8, false>(p, plan, s); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    if (plan.num_splits > 1) return launch_combine(p, p.num_kv_heads * G, s);
    return cudaSuccess;
}

}  // namespace aq
