// internal.h -- launch parameters and launcher entry points shared between the
// C-ABI layer (api.cu) and the kernel translation units.  Not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace aq {

struct DecodeParams {
    // TMA view of the codebooks as rows of Dsub fp16 elements
    // ([S * Hkv * 2 * M * K] rows), swizzled like the shared-memory slices
    // (PQ kernel with whole-split scoring)
    CUtensorMap cb_map;
    const float *q;             // [B][Hq][D]
    const uint8_t *code_pages;  // [NP][Hkv][P][2][M]
    const void *codebooks;      // fp16 [S][Hkv][2][M][K][Dsub]
    const void *kv_pages;       // fp16 [NP][Hkv][2][P][D] (fp16 path)
    const int32_t *req_set;     // [B]
    const int32_t *block_table; // [B][max_pages]
    const int32_t *seq_lens;    // [B]
    float *out;                 // [B][Hq][D]
    float *part_o;              // [B][Hq][S][D]   (num_splits > 1)
    float *part_ml;             // [B][Hq][S][2]   (num_splits > 1)
    int32_t *status;
    int32_t batch, num_q_heads, num_kv_heads, max_pages;
    int64_t num_pages, num_sets;
    int32_t max_seq_len, num_splits, split_len;  // split_len: tokens, multiple of P
    int32_t share;                               // tokens per cluster CTA, multiple of P
    const void *kv_new;     // fp16 [B][Hkv][2][D]: the token appended by a fused decode step
    uint8_t *code_pages_w;  // writable alias of code_pages (fused decode step)
    int32_t overlap;        // launched as a programmatic dependent of the previous kernel
    int32_t head_split_log2;  // PQ: 2^this clusters per kv head, each for Hq/Hkv >> this query heads
    int32_t codebook_e4m3;    // PQ step: codebooks are FP8 E4M3 codes, same layout
    int32_t cb_map_ok;        // cb_map describes the codebooks (fp16, TMA-addressable)
    // Head numbering of q / out / kv_new when a launch covers only some kv
    // heads (a mixed-precision step): launch kv head h is kv head
    // kv_head_base + h of those arrays, which hold qo_kv_heads kv heads and
    // num_q_heads query heads; its first query head is q_head_base + h * G.
    // Pages, codebooks and the grid use num_kv_heads (this launch's heads).
    int32_t q_head_base, kv_head_base, qo_kv_heads;
    // limit of the decode kernels' waits on their own copies before the
    // drain (aq_set_wait_limit_ns); the drain before exit keeps the default
    unsigned long long wait_limit_ns;
    float scale_log2;                            // scale * log2(e)
};

struct EncodeParams {
    const void *kv;            // fp16 [T][Hkv][2][D]
    const int32_t *token_set;  // [T]
    const int64_t *slot_mapping;
    const void *codebooks;     // fp16 [S][Hkv][2][M][K][Dsub]
    uint8_t *code_pages;       // [NP][Hkv][P][2][M]
    int32_t *status;
    int32_t num_tokens, num_kv_heads;
    int64_t num_sets, num_pages;
};

struct FitParams {
    const void *samples;       // fp16 [U][N][D]
    const float *cent_in;      // fp32 [U][M][K][Dsub] (step) or nullptr (fit)
    const void *cb_init;       // fp16 [U][M][K][Dsub] starting centroids (refine) or nullptr
    float *cent_out;           // fp32 [U][M][K][Dsub] (step) or nullptr
    void *codebooks;           // fp16 [U][M][K][Dsub] (fit) or nullptr
    int32_t *assign;           // [U][N][M] or nullptr
    int64_t num_units;
    int32_t n_samples, iters;
};

struct Plan {
    int32_t kernel;       // PQ: 1 = per-CTA token shares with merged bins, 2 = whole-split scoring
    int32_t num_splits;
    int32_t cluster;      // CTAs per split
    int32_t split_len;    // tokens per split (multiple of the page size)
    int32_t share;        // tokens per CTA of a cluster (multiple of the page size)
    int32_t head_split;   // PQ: query-head sub-groups per kv head, each its own cluster
    size_t workspace;     // bytes
    size_t smem;          // dynamic shared memory per CTA
};

// Returns cudaSuccess or the launch error.
cudaError_t launch_pq_decode(const DecodeParams &p, int M, int G, const Plan &plan,
                             cudaStream_t s);
// Fused decode step: append each request's new token (at position seq_len-1)
// into the code cache, then the PQ decode attention that includes it.
cudaError_t launch_pq_decode_step(const DecodeParams &p, int M, int G, const Plan &plan,
                                  cudaStream_t s);
cudaError_t launch_fp16_decode(const DecodeParams &p, int G, const Plan &plan, cudaStream_t s);
// Combine of split partials for this launch's query heads (num_q_heads_launch
// of them, from q_head_base on).
cudaError_t launch_combine(const DecodeParams &p, int num_q_heads_launch, cudaStream_t s);
// Copy each request's new fp16 key and value (kv_new) into its page slot of an
// fp16 cache, for this launch's kv heads.
cudaError_t launch_encode(const EncodeParams &p, int M, cudaStream_t s);
cudaError_t launch_to_e4m3(int64_t n, const void *src_f16, uint8_t *dst, cudaStream_t s);
cudaError_t launch_from_e4m3(int64_t n, const uint8_t *src, void *dst_f16, cudaStream_t s);
cudaError_t launch_fit(const FitParams &p, int M, cudaStream_t s);

// Shared-memory bytes a PQ decode CTA needs for (M, G, cluster).
size_t pq_decode_smem_bytes(int M, int G, int cluster);
// Whole-split kernel: shared-memory bytes for a split of `split_len` tokens
// (0 for an unsupported (M, G, cluster)), and the most tokens one split may
// hold (its codes in shared memory, its scores in registers).
size_t pq_attend_smem_bytes(int M, int G, int cluster, int split_len);
int pq_attend_max_split(int M, int G);
// Tokens of one chunk of a token-share CTA (its codes live in registers, a
// fixed number per thread); 0 for an unsupported (M, G).  A CTA of a cluster
// of 4 or 8 with fp16 codebooks streams up to kMaxStreamChunks chunks in two
// passes; other CTAs hold one chunk.
int pq_decode_max_share(int M, int G);
constexpr int kMaxStreamChunks = 16;
size_t fit_smem_bytes(int M, int n_samples);
// The current limit of the decode kernels' waits (aq_set_wait_limit_ns).
unsigned long long decode_wait_limit_ns();
// Record a CUDA error for aq_last_error_message() and clear the runtime's
// last-error state.
void record_cuda_error(cudaError_t e);

// Opt-in dynamic shared memory already granted to one kernel, per device
// ordinal: cudaFuncSetAttribute acts on the current device's context only, so
// a size set while device 0 was current says nothing about device 1.
constexpr int kMaxDevices = 64;
struct SmemAttr {
    std::mutex mu;
    size_t bytes[kMaxDevices] = {};
};
// Make sure `func` may launch with `need` bytes of dynamic shared memory on the
// current device (sets the attribute the first time a larger size is asked
// for on that device; thread-safe).  carveout_pct >= 0 also sets the
// preferred shared-memory carveout (percent of the SM's shared memory; the
// rest serves as L1) at that point.
cudaError_t ensure_smem_attr(SmemAttr &a, const void *func, size_t need, int carveout_pct = -1);

}  // namespace aq
