// api.cu -- the extern "C" boundary of libaqpq (declared in include/aqpq.h):
// host-side argument checks (before any CUDA call), work planning, dispatch to
// the kernel launchers and mapping of CUDA errors to AQ_ERR_CUDA.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "aqpq.h"
#include "common.cuh"
#include "internal.h"

namespace aq {

namespace {

thread_local char g_last_error[256] = "";

aq_status cuda_fail(cudaError_t e) {
    cudaGetLastError();            // reported here: do not leave it for the next caller
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return AQ_ERR_CUDA;
}

// Device tensors are read with 16-byte vector, cp.async and bulk copies.
bool misaligned(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; }

aq_status check_cfg(const aq_pq_config *cfg, bool need_pq) {
    if (!cfg) return AQ_ERR_INVALID_ARGUMENT;
    if (cfg->head_dim <= 0 || cfg->page_size <= 0) return AQ_ERR_INVALID_ARGUMENT;
    if (cfg->head_dim != kHeadDim || cfg->page_size != kPage) return AQ_ERR_UNSUPPORTED;
    if (!need_pq) return AQ_OK;
    if (cfg->num_subspaces <= 0 || cfg->num_codewords <= 0) return AQ_ERR_INVALID_ARGUMENT;
    if (cfg->head_dim % cfg->num_subspaces != 0) return AQ_ERR_INVALID_ARGUMENT;
    if (cfg->num_codewords > 256) return AQ_ERR_INVALID_ARGUMENT;      // uint8 codes
    if (cfg->num_codewords != kCodewords) return AQ_ERR_UNSUPPORTED;
    if (cfg->num_subspaces != 4 && cfg->num_subspaces != 8) return AQ_ERR_UNSUPPORTED;
    return AQ_OK;
}

bool group_ok(int G) { return G == 1 || G == 2 || G == 4 || G == 8; }

}  // namespace

void record_cuda_error(cudaError_t e) {
    cudaGetLastError();
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
}

namespace {
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitNs};
}  // namespace

unsigned long long decode_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

cudaError_t ensure_smem_attr(SmemAttr &a, const void *func, size_t need, int carveout_pct) {
    auto set = [&]() {
        cudaError_t r = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(need));
        if (r == cudaSuccess && carveout_pct >= 0)
            r = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, carveout_pct);
        return r;
    };
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return set();
    std::lock_guard<std::mutex> lock(a.mu);
    if (a.bytes[dev] >= need) return cudaSuccess;
    e = set();
    if (e == cudaSuccess) a.bytes[dev] = need;
    return e;
}

// The plan is a pure function of the arguments (no device query), so that
// aq_decode_plan and the decode call always agree: it is sized for GB300
// (152 SMs, 227 KiB of opt-in shared memory per CTA).
constexpr int kPlanSMs = 152;
constexpr size_t kPlanSmemCap = 232448;

// Work plan of a decode call.  Host-only arithmetic; `sms` is the SM count.
//   PQ:   cluster C = 4 CTAs per split when M >= 4 (each owns M/C subspaces of
//         both codebooks, so every codebook byte is read once and a split's
//         tokens spread over 4 SMs), smaller if shared memory does not fit.
//         When C = 4 would give many waves of CTAs anyway (a long ragged
//         batch), C = 2: the per-(request, kv head) work -- table build, the
//         new token's encode, value product -- then runs with half the
//         exchanges and per-CTA overhead, and the GPU is still full.
//         Splits are added only when (request, kv head) clusters cannot fill
//         the GPU and each split keeps >= 1024 tokens, since every split
//         re-reads the codebooks.
//         With M = 8 and a request long enough for several splits, clusters
//         of 8 (one subspace per CTA) halve the splits.
//         A GQA group is split over several clusters (query heads per
//         cluster G / head_split) before any KV split when the (request, kv
//         head) clusters alone would not fill the GPU.
//   fp16: splits so that (request, kv head, split) CTAs reach 2 per SM, each
//         keeping >= 256 tokens.
constexpr int kManyWaves = 8;          // waves of 4 CTAs per SM

// Returns false when the request is too long for this kernel: a CTA holds at
// most share_max tokens and a call runs at most kMaxSplits splits.
constexpr int kMaxSplits = 4096;

static bool split_plan(int C, int share_max, bool fp16, int64_t units, int max_seq_len, int req, int sms, int P,
                       Plan *pl) {
    const int max_pages_needed = (max_seq_len + P - 1) / P;
    int S = req;
    if (S <= 0) {
        const int64_t target = 2ll * sms;
        const int min_tok = fp16 ? 256 : 1024;
        const int64_t per_split_ctas = units * C;
        S = 1;
        if (per_split_ctas > 0 && per_split_ctas < target) {
            const int64_t want = (target + per_split_ctas - 1) / per_split_ctas;
            const int64_t cap = max_seq_len / min_tok;
            S = static_cast<int>(want < cap ? want : cap);
            if (S < 1) S = 1;
        }
    }
    if (!fp16) {
        // each CTA of a cluster holds at most share_max tokens
        const int64_t need = (static_cast<int64_t>(max_seq_len) + static_cast<int64_t>(C) * share_max - 1) /
                             (static_cast<int64_t>(C) * share_max);
        if (need > kMaxSplits) return false;
        if (S < need) S = static_cast<int>(need);
    }
    if (S > kMaxSplits) S = kMaxSplits;
    if (max_pages_needed == 0) S = 1;
    // split length: page multiple; recompute S so no trailing split is empty
    int split_pages = (max_pages_needed + S - 1) / S;
    if (split_pages < 1) split_pages = 1;
    S = (max_pages_needed + split_pages - 1) / split_pages;
    if (S < 1) S = 1;
    pl->num_splits = S;
    pl->cluster = C;
    pl->split_len = split_pages * P;
    pl->share = ((pl->split_len + C - 1) / C + P - 1) / P * P;
    return true;
}

// Which PQ kernel: AQPQ_DECODE_KERNEL=1 or 2 in the environment forces one
// (for comparing them); otherwise the planner chooses.
static int forced_kernel() {
    const char *e = std::getenv("AQPQ_DECODE_KERNEL");
    if (!e) return 0;
    return (e[0] == '1' || e[0] == '2') && e[1] == 0 ? e[0] - '0' : 0;
}

// Whole-split plan (pq_attend_kernel): clusters of C CTAs, one subspace each
// (M = 4: C = 4; M = 8: C = 8), every CTA holding the codes of the whole
// split.  Splits only as many as the split capacity requires, more when the
// clusters would not give about one CTA per SM; each split keeps >= 512
// tokens, since every split reads the codebooks again.
static bool attend_plan(int M, int G, int64_t units, int max_seq_len, int req, int sms, int P,
                        size_t smem_cap, Plan *pl) {
    const int C = M;                                   // one subspace per CTA
    const int cap = pq_attend_max_split(M, G);
    if (cap <= 0) return false;
    const int pages = (max_seq_len + P - 1) / P;
    int S = req;
    if (S <= 0) {
        S = (max_seq_len + cap - 1) / cap;
        if (S < 1) S = 1;
        const int64_t ctas = units * C * S;
        if (ctas < sms && max_seq_len >= 1024) {
            int want = static_cast<int>((sms + units * C - 1) / (units * C));
            const int most = max_seq_len / 512;
            if (want > most) want = most;
            if (want > S) S = want;
        }
    }
    if (S > kMaxSplits) S = kMaxSplits;
    if (pages == 0) S = 1;
    int split_pages = (pages + S - 1) / S;
    if (split_pages < 1) split_pages = 1;
    if (split_pages * P > cap) return false;
    S = (pages + split_pages - 1) / split_pages;
    if (S < 1) S = 1;
    const size_t smem = pq_attend_smem_bytes(M, G, C, split_pages * P);
    if (smem == 0 || smem > smem_cap) return false;
    pl->kernel = 2;
    pl->num_splits = S;
    pl->cluster = C;
    pl->split_len = split_pages * P;
    pl->share = pl->split_len;
    pl->head_split = 1;
    pl->smem = smem;
    return true;
}

static aq_status share_plan(const aq_pq_config *cfg, int batch, int Hq, int Hkv, int max_seq_len,
                            int req, bool fp16, int sms, size_t smem_cap, Plan *pl, bool stream);

// The plan of a decode call.  PQ: the whole-split kernel for GQA groups of 4
// or more query heads per kv head when a split of at most two fits its
// capacity (with E4M3 codebooks only its head-split form) -- there the table and value product
// per query head dominate and scoring every token in each CTA is cheap
// (measured: B8 Hq64 Hkv8 L1000 13.3 -> 12.9 us) -- else the token-share
// kernel, whose split of the token work across the cluster is cheaper when
// each kv head serves one or two query heads (B4 H32 L2048: 7.9 us against
// 9.3 us).  The workspace reported covers both, so a caller that
// sizes it with aq_decode_plan (which does not know the codebook format) has
// enough for either.
static aq_status make_plan(const aq_pq_config *cfg, int batch, int Hq, int Hkv, int max_seq_len,
                           int req, bool fp16, int sms, size_t smem_cap, Plan *pl, bool e4m3 = false,
                           bool allow_attend = true) {
    // the token-share plan for this codebook format, and for the other one (an
    // E4M3 call streams no multi-chunk shares, so it may split more)
    Plan p1{}, p1x{};
    aq_status st = share_plan(cfg, batch, Hq, Hkv, max_seq_len, req, fp16, sms, smem_cap, &p1, !e4m3);
    if (st != AQ_OK) return st;
    // the other format's plan only widens the workspace; a length it cannot
    // take is refused when a call of that format asks for it
    if (share_plan(cfg, batch, Hq, Hkv, max_seq_len, req, fp16, sms, smem_cap, &p1x, e4m3) == AQ_OK &&
        p1x.workspace > p1.workspace)
        p1.workspace = p1x.workspace;
    Plan p2{};
    const int64_t units = static_cast<int64_t>(batch) * Hkv;
    const int forced = forced_kernel();
    if (!fp16 && allow_attend && forced != 1 && (forced == 2 || Hq / Hkv >= 4) &&
        attend_plan(cfg->num_subspaces, Hq / Hkv, units, max_seq_len, req, sms, cfg->page_size, smem_cap, &p2) &&
        (forced == 2 || p2.num_splits <= 2)) {
        p2.workspace = p2.num_splits > 1
                           ? static_cast<size_t>(batch) * Hq * p2.num_splits * (kHeadDim + 2) * sizeof(float)
                           : 0;
        const size_t ws = p2.workspace > p1.workspace ? p2.workspace : p1.workspace;
        // E4M3 codebooks: the head-split kernel (the group covers the cluster of
        // one subspace per CTA) widens its slices; the whole-split one reads fp16
        const int G = Hq / Hkv, M = cfg->num_subspaces;
        *pl = (e4m3 && !(G >= 4 && G >= M)) ? p1 : p2;
        pl->workspace = ws;
        return AQ_OK;
    }
    *pl = p1;
    return AQ_OK;
}

static aq_status share_plan(const aq_pq_config *cfg, int batch, int Hq, int Hkv, int max_seq_len,
                            int req, bool fp16, int sms, size_t smem_cap, Plan *pl, bool stream) {
    const int P = cfg->page_size;
    const int G = Hq / Hkv;
    const int64_t units = static_cast<int64_t>(batch) * Hkv;
    pl->kernel = 1;
    if (fp16) {
        split_plan(1, 0, true, units, max_seq_len, req, sms, P, pl);
        pl->head_split = 1;
        pl->smem = 0;
    } else {
        const int M = cfg->num_subspaces;
        // a GQA group's query heads over several clusters while (request, kv
        // head) clusters of 4 would not give 2 CTAs per SM: each cluster builds
        // the table, scores and takes the value product for its heads only, so
        // only the codebook and code reads (from L2 after the first) and the
        // new token's encode repeat -- much cheaper than more KV splits
        int nsub = 1;
        while (nsub < G && units * 4 * nsub < 2ll * sms) nsub *= 2;
        const int Gs = G / nsub;
        int C = 0;
        for (int c = 4; c >= 1; c /= 2)
            if (c <= M && pq_decode_smem_bytes(M, Gs, c) <= smem_cap) { C = c; break; }
        if (C == 0) return AQ_ERR_UNSUPPORTED;
        const int chunk = pq_decode_max_share(M, Gs) / P * P;
        if (chunk <= 0) return AQ_ERR_UNSUPPORTED;
        // shares of several chunks (streamed in two passes) for clusters of 4 or 8
        auto share_max = [&](int c) { return stream && c >= 4 ? chunk * kMaxStreamChunks : chunk; };
        const int64_t clusters = units * nsub;         // per split
        if (!split_plan(C, share_max(C), false, clusters, max_seq_len, req, sms, P, pl))
            return AQ_ERR_UNSUPPORTED;
        const int64_t ctas = clusters * pl->num_splits * C;
        // a re-plan replaces the first one only where it exists
        Plan alt = *pl;
        if (C == 4 && ctas >= static_cast<int64_t>(kManyWaves) * sms * 4 &&
            pq_decode_smem_bytes(M, Gs, 2) <= smem_cap) {
            if (split_plan(2, share_max(2), false, clusters, max_seq_len, req, sms, P, &alt)) *pl = alt;
        } else if (C == 4 && M == 8 && pl->num_splits >= 2 && pq_decode_smem_bytes(M, Gs, 8) > 0 &&
                   pq_decode_smem_bytes(M, Gs, 8) <= smem_cap) {
            // a long request with 8 subspaces: clusters of 8, one subspace per
            // CTA, half the splits and so half the per-split fixed work
            if (split_plan(8, share_max(8), false, clusters, max_seq_len, req, sms, P, &alt)) *pl = alt;
        }
        pl->head_split = nsub;
        pl->smem = pq_decode_smem_bytes(M, Gs, pl->cluster);
    }
    pl->workspace = pl->num_splits > 1
                        ? static_cast<size_t>(batch) * Hq * pl->num_splits * (kHeadDim + 2) * sizeof(float)
                        : 0;
    return AQ_OK;
}

}  // namespace aq

namespace aq {
namespace {

// The device address of page-locked host memory the device can reach (pinned
// with cudaHostAlloc / cudaMallocHost or registered), or null for any other
// pointer (pageable memory, device memory).
void *mapped_host(const void *h) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// The step's query and new K/V from mapped host memory into the device
// staging, 16 bytes per thread over the NVLink-C2C link: the host-to-device
// copy of a step without a DMA set-up, ahead of the step, which starts as its
// programmatic dependent and reads the staging after it completes.
__global__ void __launch_bounds__(256) host_gather_kernel(const uint4 *q_h, uint4 *q_d, size_t nq, const uint4 *kv_h,
                                                          uint4 *kv_d, size_t nkv) {
    grid_launch_dependents();
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t j = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < nq + nkv; j += stride) {
        if (j < nq) q_d[j] = q_h[j];
        else kv_d[j - nq] = kv_h[j - nq];
    }
}

}  // namespace
}  // namespace aq

using namespace aq;

extern "C" {

const char *aq_status_string(aq_status s) {
    switch (s) {
        case AQ_OK: return "AQ_OK";
        case AQ_ERR_INVALID_ARGUMENT: return "AQ_ERR_INVALID_ARGUMENT";
        case AQ_ERR_UNSUPPORTED: return "AQ_ERR_UNSUPPORTED";
        case AQ_ERR_WORKSPACE_TOO_SMALL: return "AQ_ERR_WORKSPACE_TOO_SMALL";
        case AQ_ERR_CUDA: return "AQ_ERR_CUDA";
        default: return "AQ_ERR_UNKNOWN";
    }
}

const char *aq_last_error_message(void) { return aq::g_last_error; }

const char *aq_version(void) { return "aqpq 0.2 sm_103a"; }

uint64_t aq_set_wait_limit_ns(uint64_t ns) {
    constexpr uint64_t kMax = 1000000000ull;           // 1 s
    return aq::g_wait_limit_ns.exchange(ns > kMax ? kMax : ns);
}

aq_status aq_fit_codebooks(const aq_pq_config *cfg, int64_t num_units, int32_t n_samples,
                           int32_t iters, const void *samples_f16, void *codebooks_f16,
                           int32_t *assign_out, aq_stream_t stream) {
    aq_status st = check_cfg(cfg, true);
    if (st != AQ_OK) return st;
    if (num_units < 0 || n_samples < 1 || iters < 1 || iters > 1000) return AQ_ERR_INVALID_ARGUMENT;
    if (n_samples > 1024) return AQ_ERR_UNSUPPORTED;
    if (num_units > 0 && (!samples_f16 || !codebooks_f16)) return AQ_ERR_INVALID_ARGUMENT;
    if (misaligned(samples_f16) || misaligned(codebooks_f16)) return AQ_ERR_INVALID_ARGUMENT;
    if (num_units > 2147483647ll) return AQ_ERR_UNSUPPORTED;
    if (num_units == 0) return AQ_OK;
    FitParams p{};
    p.samples = samples_f16;
    p.codebooks = codebooks_f16;
    p.assign = assign_out;
    p.num_units = num_units;
    p.n_samples = n_samples;
    p.iters = iters;
    cudaError_t e = launch_fit(p, cfg->num_subspaces, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AQ_OK : cuda_fail(e);
}

aq_status aq_refine_codebooks(const aq_pq_config *cfg, int64_t num_units, int32_t n_samples,
                              int32_t iters, const void *samples_f16, void *codebooks_f16,
                              int32_t *assign_out, aq_stream_t stream) {
    aq_status st = check_cfg(cfg, true);
    if (st != AQ_OK) return st;
    if (num_units < 0 || n_samples < 1 || iters < 1 || iters > 1000) return AQ_ERR_INVALID_ARGUMENT;
    if (n_samples > 1024) return AQ_ERR_UNSUPPORTED;
    if (num_units > 0 && (!samples_f16 || !codebooks_f16)) return AQ_ERR_INVALID_ARGUMENT;
    if (misaligned(samples_f16) || misaligned(codebooks_f16)) return AQ_ERR_INVALID_ARGUMENT;
    if (num_units > 2147483647ll) return AQ_ERR_UNSUPPORTED;
    if (num_units == 0) return AQ_OK;
    FitParams p{};
    p.samples = samples_f16;
    p.cb_init = codebooks_f16;
    p.codebooks = codebooks_f16;
    p.assign = assign_out;
    p.num_units = num_units;
    p.n_samples = n_samples;
    p.iters = iters;
    cudaError_t e = launch_fit(p, cfg->num_subspaces, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AQ_OK : cuda_fail(e);
}

aq_status aq_codebooks_to_e4m3(int64_t n, const void *src_f16, uint8_t *dst_e4m3, aq_stream_t stream) {
    if (n < 0) return AQ_ERR_INVALID_ARGUMENT;
    if (n == 0) return AQ_OK;
    if (!src_f16 || !dst_e4m3 || misaligned(src_f16) || misaligned(dst_e4m3)) return AQ_ERR_INVALID_ARGUMENT;
    cudaError_t e = launch_to_e4m3(n, src_f16, dst_e4m3, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AQ_OK : cuda_fail(e);
}

aq_status aq_codebooks_from_e4m3(int64_t n, const uint8_t *src_e4m3, void *dst_f16, aq_stream_t stream) {
    if (n < 0) return AQ_ERR_INVALID_ARGUMENT;
    if (n == 0) return AQ_OK;
    if (!src_e4m3 || !dst_f16 || misaligned(src_e4m3) || misaligned(dst_f16)) return AQ_ERR_INVALID_ARGUMENT;
    cudaError_t e = launch_from_e4m3(n, src_e4m3, dst_f16, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AQ_OK : cuda_fail(e);
}

aq_status aq_kmeans_step(const aq_pq_config *cfg, int64_t num_units, int32_t n_samples,
                         const void *samples_f16, const float *centroids_in, float *centroids_out,
                         int32_t *assign_out, aq_stream_t stream) {
    aq_status st = check_cfg(cfg, true);
    if (st != AQ_OK) return st;
    if (num_units < 0 || n_samples < 1) return AQ_ERR_INVALID_ARGUMENT;
    if (n_samples > 1024) return AQ_ERR_UNSUPPORTED;
    if (num_units > 0 && (!samples_f16 || !centroids_in || !centroids_out || !assign_out))
        return AQ_ERR_INVALID_ARGUMENT;
    if (misaligned(samples_f16) || misaligned(centroids_in) || misaligned(centroids_out))
        return AQ_ERR_INVALID_ARGUMENT;
    if (num_units > 2147483647ll) return AQ_ERR_UNSUPPORTED;
    if (num_units == 0) return AQ_OK;
    FitParams p{};
    p.samples = samples_f16;
    p.cent_in = centroids_in;
    p.cent_out = centroids_out;
    p.assign = assign_out;
    p.num_units = num_units;
    p.n_samples = n_samples;
    p.iters = 1;
    cudaError_t e = launch_fit(p, cfg->num_subspaces, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AQ_OK : cuda_fail(e);
}

aq_status aq_encode_append(const aq_pq_config *cfg, int32_t num_tokens, int32_t num_kv_heads,
                           const void *kv_f16, const int32_t *token_set, const int64_t *slot_mapping,
                           const void *codebooks_f16, int64_t num_sets, uint8_t *code_pages,
                           int64_t num_pages, int32_t *device_status, aq_stream_t stream) {
    aq_status st = check_cfg(cfg, true);
    if (st != AQ_OK) return st;
    if (num_tokens < 0 || num_kv_heads < 1 || num_kv_heads > 65535 || num_sets < 0 || num_pages < 0)
        return AQ_ERR_INVALID_ARGUMENT;
    if (num_tokens == 0) return AQ_OK;
    if (!kv_f16 || !token_set || !slot_mapping || !codebooks_f16 || !code_pages)
        return AQ_ERR_INVALID_ARGUMENT;
    if (misaligned(kv_f16) || misaligned(codebooks_f16) || misaligned(code_pages))
        return AQ_ERR_INVALID_ARGUMENT;
    EncodeParams p{};
    p.kv = kv_f16;
    p.token_set = token_set;
    p.slot_mapping = slot_mapping;
    p.codebooks = codebooks_f16;
    p.code_pages = code_pages;
    p.status = device_status;
    p.num_tokens = num_tokens;
    p.num_kv_heads = num_kv_heads;
    p.num_sets = num_sets;
    p.num_pages = num_pages;
    cudaError_t e = launch_encode(p, cfg->num_subspaces, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AQ_OK : cuda_fail(e);
}

// TMA view of the codebooks [S][Hkv][2][M][K][Dsub] fp16 as rows of Dsub
// elements, one 256-row box per subspace, with the 64-byte (Dsub 32) or
// 32-byte (Dsub 16) swizzle that places 16-byte chunk c of row k at
// c ^ ((k / (128 / row bytes)) mod chunks per row) -- the kernels' layout.
static cudaError_t codebook_tensor_map(CUtensorMap *map, const void *codebooks, int64_t num_sets, int Hkv, int M,
                                       bool e4m3 = false) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            fn = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }();
    if (!encode) return cudaErrorNotSupported;
    const int dsub = kHeadDim / M;
    const cuuint64_t rows = static_cast<cuuint64_t>(num_sets > 0 ? num_sets : 1) * Hkv * 2 * M * kCodewords;
    if (rows >= (1ull << 31)) return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(dsub), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(dsub) * (e4m3 ? 1 : 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(dsub), static_cast<cuuint32_t>(kCodewords)};
    const cuuint32_t estr[2] = {1, 1};
    // fp16 rows of 64 / 32 bytes: the 64B / 32B swizzle; E4M3 rows of 32 bytes:
    // the 32B swizzle, of 16 bytes: none (one chunk per row)
    const CUtensorMapSwizzle swz = e4m3 ? (dsub == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE)
                                        : (dsub == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    const CUresult r = encode(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                              const_cast<void *>(codebooks), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static aq_status check_decode_common(const aq_pq_config *cfg, bool need_pq, int32_t batch, int32_t Hq,
                                     int32_t Hkv, int32_t max_pages, int32_t max_seq_len,
                                     int32_t num_splits) {
    aq_status st = check_cfg(cfg, need_pq);
    if (st != AQ_OK) return st;
    if (batch < 0 || Hq < 1 || Hkv < 1 || max_pages < 0 || max_seq_len < 0 || num_splits < 0)
        return AQ_ERR_INVALID_ARGUMENT;
    if (Hq % Hkv != 0) return AQ_ERR_INVALID_ARGUMENT;
    if (!group_ok(Hq / Hkv)) return AQ_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages) * cfg->page_size)
        return AQ_ERR_INVALID_ARGUMENT;
    if (batch > 65535 || Hkv > 65535) return AQ_ERR_UNSUPPORTED;
    return AQ_OK;
}

aq_status aq_decode_plan(const aq_pq_config *cfg, int32_t batch, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t max_seq_len, int32_t num_splits_req,
                         int32_t fp16, int32_t *num_splits, int32_t *cluster_size,
                         size_t *workspace_bytes) {
    const int P = cfg ? cfg->page_size : 1;
    aq_status st = check_decode_common(cfg, !fp16, batch, num_q_heads, num_kv_heads,
                                       P > 0 ? (max_seq_len + P - 1) / P : 0, max_seq_len,
                                       num_splits_req);
    if (st != AQ_OK) return st;
    Plan pl{};
    st = make_plan(cfg, batch, num_q_heads, num_kv_heads, max_seq_len, num_splits_req, fp16 != 0,
                   kPlanSMs, kPlanSmemCap, &pl);
    if (st != AQ_OK) return st;
    if (num_splits) *num_splits = pl.num_splits;
    if (cluster_size) *cluster_size = pl.cluster;
    if (workspace_bytes) *workspace_bytes = pl.workspace;
    return AQ_OK;
}

static aq_status decode_impl(const aq_pq_config *cfg, bool fp16, int32_t batch, int32_t Hq, int32_t Hkv,
                             const float *q, const uint8_t *code_pages, const void *kv_pages,
                             const void *kv_new, uint8_t *code_pages_w, int32_t flags,
                             int64_t num_pages, const void *codebooks, int64_t num_sets,
                             const int32_t *req_set, const int32_t *block_table, int32_t max_pages,
                             const int32_t *seq_lens, int32_t max_seq_len, float scale,
                             int32_t num_splits, float *out, void *ws, size_t ws_bytes,
                             int32_t *device_status, aq_stream_t stream, bool check_only = false) {
    aq_status st = check_decode_common(cfg, !fp16, batch, Hq, Hkv, max_pages, max_seq_len, num_splits);
    if (st != AQ_OK) return st;
    if (!std::isfinite(scale)) return AQ_ERR_INVALID_ARGUMENT;
    if (num_pages < 0 || num_sets < 0) return AQ_ERR_INVALID_ARGUMENT;
    if (batch == 0) return AQ_OK;
    if (!q || !out || !block_table || !seq_lens) return AQ_ERR_INVALID_ARGUMENT;
    if (fp16 ? !kv_pages : (!code_pages || !codebooks || !req_set)) return AQ_ERR_INVALID_ARGUMENT;
    if (kv_new && !code_pages_w) return AQ_ERR_INVALID_ARGUMENT;
    if (misaligned(q) || misaligned(out) || misaligned(code_pages) || misaligned(kv_pages) ||
        misaligned(kv_new) || misaligned(code_pages_w) || misaligned(codebooks) || misaligned(ws))
        return AQ_ERR_INVALID_ARGUMENT;
    if (flags & ~(AQ_STEP_OVERLAP | AQ_STEP_E4M3)) return AQ_ERR_INVALID_ARGUMENT;
    if ((flags & AQ_STEP_E4M3) && (fp16 || !kv_new)) return AQ_ERR_INVALID_ARGUMENT;
    if (max_pages == 0 && max_seq_len > 0) return AQ_ERR_INVALID_ARGUMENT;
    Plan pl{};
    st = make_plan(cfg, batch, Hq, Hkv, max_seq_len, num_splits, fp16, kPlanSMs, kPlanSmemCap, &pl,
                   (flags & AQ_STEP_E4M3) != 0);
    if (st != AQ_OK) return st;
    if (pl.workspace > 0 && (!ws || ws_bytes < pl.workspace)) return AQ_ERR_WORKSPACE_TOO_SMALL;
    if (check_only) return AQ_OK;
    DecodeParams p{};
    // a TMA view of the codebooks (fp16 or E4M3) for the kernels' slice copies
    p.cb_map_ok = !fp16 && codebook_tensor_map(&p.cb_map, codebooks, num_sets, Hkv, cfg->num_subspaces,
                                               (flags & AQ_STEP_E4M3) != 0) == cudaSuccess;
    if (pl.kernel == 2 && !p.cb_map_ok) {
        // no TMA view of these codebooks (too many rows): the token-share kernel
        const size_t ws_need = pl.workspace;
        st = make_plan(cfg, batch, Hq, Hkv, max_seq_len, num_splits, fp16, kPlanSMs, kPlanSmemCap, &pl, true, false);
        if (st != AQ_OK) return st;
        pl.workspace = ws_need > pl.workspace ? ws_need : pl.workspace;
    }
    p.q = q;
    p.code_pages = code_pages;
    p.codebooks = codebooks;
    p.kv_pages = kv_pages;
    p.req_set = req_set;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = out;
    if (pl.num_splits > 1) {
        p.part_o = static_cast<float *>(ws);
        p.part_ml = p.part_o + static_cast<size_t>(batch) * Hq * pl.num_splits * kHeadDim;
    }
    p.status = device_status;
    p.batch = batch;
    p.num_q_heads = Hq;
    p.num_kv_heads = Hkv;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.num_sets = num_sets;
    p.max_seq_len = max_seq_len;
    p.num_splits = pl.num_splits;
    p.split_len = pl.split_len;
    p.share = pl.share;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.kv_new = kv_new;
    p.code_pages_w = code_pages_w;
    p.overlap = (flags & AQ_STEP_OVERLAP) ? 1 : 0;
    p.codebook_e4m3 = (flags & AQ_STEP_E4M3) ? 1 : 0;
    p.q_head_base = 0;
    p.kv_head_base = 0;
    p.qo_kv_heads = Hkv;
    p.wait_limit_ns = decode_wait_limit_ns();
    p.head_split_log2 = 0;
    while ((1 << p.head_split_log2) < pl.head_split) ++p.head_split_log2;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = fp16     ? launch_fp16_decode(p, Hq / Hkv, pl, s)
                    : kv_new ? launch_pq_decode_step(p, cfg->num_subspaces, Hq / Hkv, pl, s)
                             : launch_pq_decode(p, cfg->num_subspaces, Hq / Hkv, pl, s);
    return e == cudaSuccess ? AQ_OK : cuda_fail(e);
}

aq_status aq_decode_attention(const aq_pq_config *cfg, int32_t batch, int32_t num_q_heads,
                              int32_t num_kv_heads, const float *q, const uint8_t *code_pages,
                              int64_t num_pages, const void *codebooks_f16, int64_t num_sets,
                              const int32_t *req_set, const int32_t *block_table, int32_t max_pages,
                              const int32_t *seq_lens, int32_t max_seq_len, float scale,
                              int32_t num_splits, float *out, void *workspace, size_t workspace_bytes,
                              int32_t *device_status, aq_stream_t stream) {
    return decode_impl(cfg, false, batch, num_q_heads, num_kv_heads, q, code_pages, nullptr, nullptr, nullptr, 0,
                       num_pages, codebooks_f16, num_sets, req_set, block_table, max_pages, seq_lens,
                       max_seq_len, scale, num_splits, out, workspace, workspace_bytes, device_status, stream);
}

aq_status aq_decode_step(const aq_pq_config *cfg, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                         const float *q, const void *kv_new_f16, uint8_t *code_pages, int64_t num_pages,
                         const void *codebooks_f16, int64_t num_sets, const int32_t *req_set,
                         const int32_t *block_table, int32_t max_pages, const int32_t *seq_lens,
                         int32_t max_seq_len, float scale, int32_t num_splits, int32_t flags, float *out,
                         void *workspace, size_t workspace_bytes, int32_t *device_status, aq_stream_t stream) {
    if (batch > 0 && !kv_new_f16) return AQ_ERR_INVALID_ARGUMENT;
    return decode_impl(cfg, false, batch, num_q_heads, num_kv_heads, q, code_pages, nullptr, kv_new_f16,
                       code_pages, flags, num_pages, codebooks_f16, num_sets, req_set, block_table, max_pages,
                       seq_lens, max_seq_len, scale, num_splits, out, workspace, workspace_bytes,
                       device_status, stream);
}

size_t aq_decode_step_host_staging(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads) {
    const size_t q = static_cast<size_t>(batch) * num_q_heads * kHeadDim * sizeof(float);
    const size_t kv = static_cast<size_t>(batch) * num_kv_heads * 2 * kHeadDim * 2;
    return (q + 255) / 256 * 256 + (kv + 255) / 256 * 256 + (q + 255) / 256 * 256;
}

aq_status aq_decode_step_host(const aq_pq_config *cfg, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                              const float *q_host, const void *kv_new_host, uint8_t *code_pages, int64_t num_pages,
                              const void *codebooks_f16, int64_t num_sets, const int32_t *req_set,
                              const int32_t *block_table, int32_t max_pages, const int32_t *seq_lens,
                              int32_t max_seq_len, float scale, int32_t num_splits, int32_t flags, float *out_host,
                              void *staging, size_t staging_bytes, void *workspace, size_t workspace_bytes,
                              int32_t *device_status, aq_stream_t stream) {
    if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1) return AQ_ERR_INVALID_ARGUMENT;
    if (batch > 0 && (!q_host || !kv_new_host || !out_host || !staging)) return AQ_ERR_INVALID_ARGUMENT;
    if (misaligned(staging)) return AQ_ERR_INVALID_ARGUMENT;
    if (staging_bytes < aq_decode_step_host_staging(batch, num_q_heads, num_kv_heads))
        return AQ_ERR_WORKSPACE_TOO_SMALL;
    if (flags & ~(AQ_STEP_OVERLAP | AQ_STEP_E4M3)) return AQ_ERR_INVALID_ARGUMENT;
    const size_t qb = static_cast<size_t>(batch) * num_q_heads * kHeadDim * sizeof(float);
    const size_t kvb = static_cast<size_t>(batch) * num_kv_heads * 2 * kHeadDim * 2;
    unsigned char *st = static_cast<unsigned char *>(staging);
    float *q_d = reinterpret_cast<float *>(st);
    void *kv_d = st + (qb + 255) / 256 * 256;
    float *out_d = reinterpret_cast<float *>(st + (qb + 255) / 256 * 256 + (kvb + 255) / 256 * 256);
    // every argument of the step is checked before anything is enqueued, so a
    // rejected call leaves the stream and the staging buffer untouched
    const aq_status chk = decode_impl(cfg, false, batch, num_q_heads, num_kv_heads, q_d, code_pages, nullptr, kv_d,
                                      code_pages, flags & ~AQ_STEP_OVERLAP, num_pages, codebooks_f16, num_sets,
                                      req_set, block_table, max_pages, seq_lens, max_seq_len, scale, num_splits,
                                      out_d, workspace, workspace_bytes, device_status, stream, true);
    if (chk != AQ_OK || batch == 0) return chk;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // page-locked buffers the device can reach: the inputs by a gather kernel,
    // the output written by the step straight into host memory
    void *q_m = misaligned(q_host) ? nullptr : mapped_host(q_host);
    void *kv_m = q_m && !misaligned(kv_new_host) ? mapped_host(kv_new_host) : nullptr;
    void *out_m = kv_m && !misaligned(out_host) ? mapped_host(out_host) : nullptr;
    if (out_m) {
        const size_t nq = qb / 16, nkv = kvb / 16;
        size_t blocks = (nq + nkv + 255) / 256;
        if (blocks > 4 * static_cast<size_t>(kPlanSMs)) blocks = 4 * static_cast<size_t>(kPlanSMs);
        host_gather_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            static_cast<const uint4 *>(q_m), reinterpret_cast<uint4 *>(q_d), nq, static_cast<const uint4 *>(kv_m),
            static_cast<uint4 *>(kv_d), nkv);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
        // the step as a programmatic dependent of the gather, which writes none
        // of its early inputs (codebooks, req_set, seq_lens, block table, pages)
        return aq_decode_step(cfg, batch, num_q_heads, num_kv_heads, q_d, kv_d, code_pages, num_pages, codebooks_f16,
                              num_sets, req_set, block_table, max_pages, seq_lens, max_seq_len, scale, num_splits,
                              (flags & ~AQ_STEP_OVERLAP) | AQ_STEP_OVERLAP, static_cast<float *>(out_m), workspace,
                              workspace_bytes, device_status, stream);
    }
    // otherwise DMA copies, which precede the step in stream order; no
    // programmatic overlap with a preceding kernel
    cudaError_t e = cudaMemcpyAsync(q_d, q_host, qb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(kv_d, kv_new_host, kvb, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    aq_status r = aq_decode_step(cfg, batch, num_q_heads, num_kv_heads, q_d, kv_d, code_pages, num_pages,
                                 codebooks_f16, num_sets, req_set, block_table, max_pages, seq_lens, max_seq_len, scale,
                                 num_splits, flags & ~AQ_STEP_OVERLAP, out_d, workspace, workspace_bytes,
                                 device_status, stream);
    if (r != AQ_OK) return r;
    e = cudaMemcpyAsync(out_host, out_d, qb, cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? AQ_OK : cuda_fail(e);
}

aq_status aq_decode_attention_fp16(const aq_pq_config *cfg, int32_t batch, int32_t num_q_heads,
                                   int32_t num_kv_heads, const float *q, const void *kv_pages_f16,
                                   int64_t num_pages, const int32_t *block_table, int32_t max_pages,
                                   const int32_t *seq_lens, int32_t max_seq_len, float scale,
                                   int32_t num_splits, float *out, void *workspace,
                                   size_t workspace_bytes, int32_t *device_status, aq_stream_t stream) {
    return decode_impl(cfg, true, batch, num_q_heads, num_kv_heads, q, nullptr, kv_pages_f16, nullptr, nullptr, 0,
                       num_pages, nullptr, 0, nullptr, block_table, max_pages, seq_lens, max_seq_len, scale,
                       num_splits, out, workspace, workspace_bytes, device_status, stream);
}

static size_t part_bytes(int32_t batch, int32_t Hq, int32_t splits) {
    return splits > 1 ? static_cast<size_t>(batch) * Hq * splits * (kHeadDim + 2) * sizeof(float) : 0;
}

// Plans of the two parts of a mixed-precision step: the fp16 heads' attention
// and the PQ heads' step, each over its own heads, with split partials in its
// own part of the workspace (indexed by the full query-head numbering).
static aq_status mixed_plans(const aq_pq_config *cfg, int32_t batch, int32_t Hq, int32_t Hkv, int32_t n16,
                             int32_t max_seq_len, bool e4m3, Plan *p16, Plan *ppq, size_t *ws) {
    const int G = Hq / Hkv;
    *ws = 0;
    if (n16 > 0) {
        aq_status st = make_plan(cfg, batch, n16 * G, n16, max_seq_len, 0, true, kPlanSMs, kPlanSmemCap, p16);
        if (st != AQ_OK) return st;
        *ws += part_bytes(batch, Hq, p16->num_splits);
    }
    if (n16 < Hkv) {
        aq_status st = make_plan(cfg, batch, (Hkv - n16) * G, Hkv - n16, max_seq_len, 0, false, kPlanSMs,
                                 kPlanSmemCap, ppq, e4m3);
        if (st != AQ_OK) return st;
        // the workspace covers the plan of either codebook format (the size
        // query does not know the format) and the token-share plan that
        // replaces the head-split one when the codebooks get no TMA view
        // (a length one of those cannot take is refused by the call that needs it)
        Plan other{}, share{};
        int s = ppq->num_splits;
        if (make_plan(cfg, batch, (Hkv - n16) * G, Hkv - n16, max_seq_len, 0, false, kPlanSMs, kPlanSmemCap,
                      &other, !e4m3) == AQ_OK &&
            other.num_splits > s)
            s = other.num_splits;
        if (make_plan(cfg, batch, (Hkv - n16) * G, Hkv - n16, max_seq_len, 0, false, kPlanSMs, kPlanSmemCap,
                      &share, true, false) == AQ_OK &&
            share.num_splits > s)
            s = share.num_splits;
        *ws += part_bytes(batch, Hq, s);
    }
    return AQ_OK;
}

aq_status aq_decode_step_mixed_workspace(const aq_pq_config *cfg, int32_t batch, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t num_fp16_heads, int32_t max_seq_len,
                                         size_t *workspace_bytes) {
    const int P = cfg ? cfg->page_size : 1;
    aq_status st = check_decode_common(cfg, true, batch, num_q_heads, num_kv_heads,
                                       P > 0 ? (max_seq_len + P - 1) / P : 0, max_seq_len, 0);
    if (st != AQ_OK) return st;
    if (num_fp16_heads < 0 || num_fp16_heads > num_kv_heads) return AQ_ERR_INVALID_ARGUMENT;
    Plan a{}, b{};
    size_t ws = 0;
    st = mixed_plans(cfg, batch, num_q_heads, num_kv_heads, num_fp16_heads, max_seq_len, false, &a, &b, &ws);
    if (st != AQ_OK) return st;
    if (workspace_bytes) *workspace_bytes = ws;
    return AQ_OK;
}

aq_status aq_decode_step_mixed(const aq_pq_config *cfg, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t num_fp16_heads, const float *q, const void *kv_new_f16,
                               void *kv_pages_f16, int64_t num_fp16_pages, uint8_t *code_pages, int64_t num_pages,
                               const void *codebooks, int64_t num_sets, const int32_t *req_set,
                               const int32_t *block_table, int32_t max_pages, const int32_t *seq_lens,
                               int32_t max_seq_len, float scale, int32_t flags, float *out, void *workspace,
                               size_t workspace_bytes, int32_t *device_status, aq_stream_t stream) {
    aq_status st = check_decode_common(cfg, true, batch, num_q_heads, num_kv_heads, max_pages, max_seq_len, 0);
    if (st != AQ_OK) return st;
    const int Hkv = num_kv_heads, Hq = num_q_heads, G = Hq / Hkv, n16 = num_fp16_heads;
    if (n16 < 0 || n16 > Hkv) return AQ_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(scale) || num_pages < 0 || num_fp16_pages < 0 || num_sets < 0) return AQ_ERR_INVALID_ARGUMENT;
    if (flags & ~(AQ_STEP_OVERLAP | AQ_STEP_E4M3)) return AQ_ERR_INVALID_ARGUMENT;
    if (batch == 0) return AQ_OK;
    if (!q || !out || !kv_new_f16 || !block_table || !seq_lens) return AQ_ERR_INVALID_ARGUMENT;
    if (n16 > 0 && !kv_pages_f16) return AQ_ERR_INVALID_ARGUMENT;
    if (n16 < Hkv && (!code_pages || !codebooks || !req_set)) return AQ_ERR_INVALID_ARGUMENT;
    if (misaligned(q) || misaligned(out) || misaligned(kv_new_f16) || misaligned(kv_pages_f16) ||
        misaligned(code_pages) || misaligned(codebooks) || misaligned(workspace))
        return AQ_ERR_INVALID_ARGUMENT;
    if (max_pages == 0 && max_seq_len > 0) return AQ_ERR_INVALID_ARGUMENT;
    Plan p16{}, ppq{};
    size_t ws = 0;
    st = mixed_plans(cfg, batch, Hq, Hkv, n16, max_seq_len, (flags & AQ_STEP_E4M3) != 0, &p16, &ppq, &ws);
    if (st != AQ_OK) return st;
    if (ws > 0 && (!workspace || workspace_bytes < ws)) return AQ_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float *wsp = static_cast<float *>(workspace);
    DecodeParams base{};
    base.q = q;
    base.out = out;
    base.block_table = block_table;
    base.seq_lens = seq_lens;
    base.kv_new = kv_new_f16;
    base.status = device_status;
    base.batch = batch;
    base.num_q_heads = Hq;
    base.max_pages = max_pages;
    base.max_seq_len = max_seq_len;
    base.scale_log2 = scale * 1.4426950408889634f;
    base.qo_kv_heads = Hkv;
    base.wait_limit_ns = decode_wait_limit_ns();
    if (n16 < Hkv) {
        // the PQ heads: one fused step over their pools
        DecodeParams p = base;
        p.code_pages = code_pages;
        p.code_pages_w = code_pages;
        p.codebooks = codebooks;
        p.req_set = req_set;
        p.num_pages = num_pages;
        p.num_sets = num_sets;
        p.num_kv_heads = Hkv - n16;
        p.kv_head_base = n16;
        p.q_head_base = n16 * G;
        p.num_splits = ppq.num_splits;
        p.split_len = ppq.split_len;
        p.share = ppq.share;
        p.overlap = (flags & AQ_STEP_OVERLAP) ? 1 : 0;
        p.codebook_e4m3 = (flags & AQ_STEP_E4M3) ? 1 : 0;
        p.cb_map_ok = codebook_tensor_map(&p.cb_map, codebooks, num_sets, Hkv - n16, cfg->num_subspaces,
                                          p.codebook_e4m3 != 0) == cudaSuccess;
        if (ppq.kernel == 2 && !p.cb_map_ok) {
            st = make_plan(cfg, batch, (Hkv - n16) * G, Hkv - n16, max_seq_len, 0, false, kPlanSMs, kPlanSmemCap,
                           &ppq, true, false);
            if (st != AQ_OK) return st;
            p.num_splits = ppq.num_splits;                 // within the workspace: mixed_plans covers this plan
            p.split_len = ppq.split_len;
            p.share = ppq.share;
        }
        p.head_split_log2 = 0;
        while ((1 << p.head_split_log2) < ppq.head_split) ++p.head_split_log2;
        if (ppq.num_splits > 1) {
            p.part_o = wsp;
            p.part_ml = p.part_o + static_cast<size_t>(batch) * Hq * ppq.num_splits * kHeadDim;
            wsp += static_cast<size_t>(batch) * Hq * ppq.num_splits * (kHeadDim + 2);
        }
        cudaError_t e = launch_pq_decode_step(p, cfg->num_subspaces, G, ppq, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (n16 > 0) {
        // the fp16 heads: the new tokens into their pages, then the attention
        DecodeParams p = base;
        p.kv_pages = kv_pages_f16;
        p.num_pages = num_fp16_pages;
        p.num_kv_heads = n16;
        p.kv_head_base = 0;
        p.q_head_base = 0;
        p.num_splits = p16.num_splits;
        p.split_len = p16.split_len;
        p.share = p16.share;
        if (p16.num_splits > 1) {
            p.part_o = wsp;
            p.part_ml = p.part_o + static_cast<size_t>(batch) * Hq * p16.num_splits * kHeadDim;
        }
        // one kernel appends the new tokens and attends (fp16_decode_kernel's
        // APPEND form); after the PQ step it starts as that step's programmatic
        // dependent: it reads none of the step's outputs, and the step lets
        // dependents start only once it has passed its own dependency wait, so
        // the kernels before the step are complete.  It finishes after the step.
        p.overlap = n16 < Hkv ? 1 : 0;
        cudaError_t e = launch_fp16_decode(p, G, p16, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return AQ_OK;
}

}  // extern "C"
