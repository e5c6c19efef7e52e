/*
 * aqpq.h -- C ABI of libaqpq: product-quantised (PQ) KV-cache decode attention
 * for NVIDIA GB300 (sm_103a).
 *
 * The method (AQPIM blog, devpress.csdn.net, "当大模型推理撞上内存墙"):
 *   - each head_dim-D key and value vector is split into M contiguous
 *     sub-vectors of Dsub = D / M dims (§3.1 step 1);
 *   - each sub-vector is stored as the 8-bit index of its nearest codeword in a
 *     K = 256-entry codebook kept per request, layer, kv head and K-or-V
 *     (§3.1 steps 2-3, §3.2 item 1);
 *   - codebooks are fitted online from the first tokens of the sequence by a
 *     quick k-means (§3.2 item 2, §5.2 item 1);
 *   - attention scores are computed by the fused "index -> codebook lookup ->
 *     sub-vector dot product -> accumulate" flow without writing decoded
 *     vectors to memory (§4.1, §5.1 item 3);
 * with the online, split-KV softmax whose per-block (max, sum) statistics are
 * merged by a reduction (PAM article, maplevalley.com.cn,
 * "大语言模型KV缓存优化与PAM架构实践", §2.2.3) and a paged cache addressed by a
 * block table (PAM article §2.2.2; AQPIM blog §5.1 item 4).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; arrays are
 *     contiguous and row-major with the shapes given below.  libaqpq never
 *     allocates device memory and keeps no state between calls.
 *   - The fp16, fp32 and uint8 tensors (vectors, codebooks, code pages,
 *     queries, outputs, workspace) start on a 16-byte boundary, as every CUDA
 *     allocation does; a misaligned one returns AQ_ERR_INVALID_ARGUMENT.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *     legacy default stream).  A status other than AQ_OK from argument checks
 *     means nothing was launched.
 *   - Argument checks (host side, before any CUDA call) return
 *     AQ_ERR_INVALID_ARGUMENT or AQ_ERR_UNSUPPORTED; a launch failure returns
 *     AQ_ERR_CUDA (aq_last_error_message() names the CUDA error).
 *   - Data errors that only the device can see (a page id outside the pool, a
 *     sequence length beyond the block table, a codebook-set index outside the
 *     codebook array) never fault or trap: the kernels OR AQ_DEV_* bits into
 *     the caller-zeroed int32 `device_status` word and skip the offending
 *     element; attention outputs of an affected request are set to NaN.
 *   - Kernels never wait on another launch.  Their only waits are on their own
 *     asynchronous copies, bounded in time (aq_set_wait_limit_ns); a wait that
 *     runs out sets AQ_DEV_TIMEOUT, and the affected outputs become NaN.
 *
 * Layouts (D = head_dim, M = num_subspaces, Dsub = D / M, K = num_codewords,
 * P = page_size, S = number of codebook sets, NP = number of pages):
 *   codebooks_f16  fp16 [S][Hkv][2][M][K][Dsub]; [2] is K then V; a "set" is
 *                  one request (and layer): its codebooks for every kv head.
 *   code_pages     uint8 [NP][Hkv][P][2][M]; for each token slot the M key
 *                  codes then the M value codes.
 *   kv_pages_f16   fp16 [NP][Hkv][2][P][D] (uncompressed comparison cache).
 *   block_table    int32 [B][max_pages]; token t of request b is in page
 *                  block_table[b][t / P], slot t % P.
 *   GQA: query head h reads kv head h / (Hq / Hkv) (Near-memory computing
 *   ch.1, zsc.github.io, §1.4.3).
 */
#ifndef AQPQ_H
#define AQPQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t aq_status;
#define AQ_OK                      0
#define AQ_ERR_INVALID_ARGUMENT    1
#define AQ_ERR_UNSUPPORTED         2
#define AQ_ERR_WORKSPACE_TOO_SMALL 3
#define AQ_ERR_CUDA                4

/* Bits ORed into *device_status by the kernels. */
#define AQ_DEV_BAD_PAGE    1  /* block-table entry or slot outside [0, num_pages)  */
#define AQ_DEV_BAD_LENGTH  2  /* seq_len < 0, > max_pages * P or > max_seq_len     */
#define AQ_DEV_BAD_SET     4  /* req_set / token_set outside [0, num_sets)         */
#define AQ_DEV_TIMEOUT     8  /* an asynchronous copy did not land in time         */
#define AQ_DEV_INVARIANT  16  /* builds with AQ_DEBUG_CHECKS only: an internal
                                 invariant of a kernel failed (never set otherwise) */

typedef struct CUstream_st *aq_stream_t;   /* == cudaStream_t */

typedef struct {
    int32_t head_dim;        /* D: 128                                  */
    int32_t num_subspaces;   /* M: 4 or 8 (Dsub = 32 or 16)             */
    int32_t num_codewords;   /* K: 256 (codes are uint8)                */
    int32_t page_size;       /* P: 16 tokens per page                   */
} aq_pq_config;

/* Human-readable name of a status code (static string). */
const char *aq_status_string(aq_status s);

/* Text of the last CUDA error seen by this thread's libaqpq call ("" if none). */
const char *aq_last_error_message(void);

/* Library version, e.g. "aqpq 0.2 sm_103a". */
const char *aq_version(void);

/* Limit, in nanoseconds, of the decode kernels' waits on their own
 * asynchronous copies (aq_decode_attention, aq_decode_step, the PQ part of
 * aq_decode_step_mixed); default AQ_DEFAULT_WAIT_LIMIT_NS (200 ms), at most
 * 1 s.  A wait that runs out sets AQ_DEV_TIMEOUT, the outputs it affects
 * become NaN, and a fused step writes no new codes from that CTA.  Whatever
 * the limit, a kernel waits (up to 200 ms) for every copy into its shared
 * memory to land before it exits.  Meant for testing the timeout path; it
 * applies to launches made after the call, from any thread, and returns the
 * previous limit.  No pages describe this: it is a property of this
 * library's kernels. */
#define AQ_DEFAULT_WAIT_LIMIT_NS 200000000ull
uint64_t aq_set_wait_limit_ns(uint64_t ns);

/* ---------------------------------------------------------------------------
 * aq_fit_codebooks -- codebook fit by Lloyd k-means (AQPIM blog §3.2 item 2,
 * §5.2 item 1: codebooks initialised from the first tokens of each sequence
 * with a quick k-means on a small sample set).
 *
 * For each unit u in [0, num_units) (one set, kv head and K-or-V; the unit
 * order matches codebooks_f16 with u = (set * Hkv + kvh) * 2 + kv) and each
 * subspace m: centroid k starts as sample (k mod n_samples); then `iters`
 * steps of {assign every sample to its nearest centroid (squared Euclidean
 * distance summed in fp32 over j = 0..Dsub-1 without fused multiply-add, ties
 * to the lowest index); move every centroid with members to their mean
 * (exact sum, double-precision division); a centroid without members keeps its
 * value}.  The codebook is the final centroids rounded to fp16 (nearest even).
 *
 *   samples_f16   in   fp16 [U][N][D]
 *   codebooks_f16 out  fp16 [U][M][K][Dsub]
 *   assign_out    out  int32 [U][N][M], the assignment of the last step, or NULL
 * Requires 1 <= n_samples <= 1024, 1 <= iters <= 1000.
 * ------------------------------------------------------------------------- */
aq_status aq_fit_codebooks(const aq_pq_config *cfg, int64_t num_units,
                           int32_t n_samples, int32_t iters,
                           const void *samples_f16, void *codebooks_f16,
                           int32_t *assign_out, aq_stream_t stream);

/* ---------------------------------------------------------------------------
 * aq_refine_codebooks -- periodic codebook update (AQPIM blog §6.1 item 3:
 * every so many generated tokens, e.g. 64, fine-tune the codebooks with a few
 * k-means iterations on the most recent K/V vectors).
 *
 * The same `iters` Lloyd steps as aq_fit_codebooks, but centroid k starts as
 * row k of the given codebook instead of a sample; the result replaces the
 * codebook in place (a centroid that never gains members keeps its fp16
 * value bit for bit).  Codes already in the cache keep pointing at the moved
 * rows; the recent tokens used as samples are re-encoded by calling
 * aq_encode_append with the refined codebooks.
 *
 *   samples_f16   in      fp16 [U][N][D] (the recent vectors of each unit)
 *   codebooks_f16 in/out  fp16 [U][M][K][Dsub], same unit order as the fit
 *   assign_out    out     int32 [U][N][M], the assignment of the last step, or NULL
 * Requires 1 <= n_samples <= 1024, 1 <= iters <= 1000.
 * ------------------------------------------------------------------------- */
aq_status aq_refine_codebooks(const aq_pq_config *cfg, int64_t num_units,
                              int32_t n_samples, int32_t iters,
                              const void *samples_f16, void *codebooks_f16,
                              int32_t *assign_out, aq_stream_t stream);

/* ---------------------------------------------------------------------------
 * FP8 E4M3 codebook storage (AQPIM blog §4.2: codebooks kept in a
 * low-precision float such as FP8).  E4M3 (OCP): sign, 4 exponent bits with
 * bias 7, 3 fraction bits, subnormals m * 2^-9, no infinities, S.1111.111 =
 * NaN, largest magnitude 448.
 *
 * aq_codebooks_to_e4m3: n fp16 values -> n E4M3 codes, nearest with ties to
 *   the even fraction; magnitudes beyond 448 and infinities become +-448; NaN
 *   stays NaN.
 * aq_codebooks_from_e4m3: n E4M3 codes -> their exact fp16 values.  Encoding
 *   (aq_encode_append) against the widened codebook decides exactly as against
 *   the E4M3 one.
 * Both arrays are device memory, 16-byte aligned; n = 0 does nothing.
 * ------------------------------------------------------------------------- */
aq_status aq_codebooks_to_e4m3(int64_t n, const void *src_f16, uint8_t *dst_e4m3,
                               aq_stream_t stream);
aq_status aq_codebooks_from_e4m3(int64_t n, const uint8_t *src_e4m3, void *dst_f16,
                                 aq_stream_t stream);

/* One Lloyd step from given fp32 centroids (the step of aq_fit_codebooks,
 * exposed for step-by-step checking).
 *   centroids_in   in  fp32 [U][M][K][Dsub]
 *   centroids_out  out fp32 [U][M][K][Dsub] (member mean rounded to fp32, or
 *                      the input value for a centroid without members)
 *   assign_out     out int32 [U][N][M]                                     */
aq_status aq_kmeans_step(const aq_pq_config *cfg, int64_t num_units,
                         int32_t n_samples, const void *samples_f16,
                         const float *centroids_in, float *centroids_out,
                         int32_t *assign_out, aq_stream_t stream);

/* ---------------------------------------------------------------------------
 * aq_encode_append -- encode new K/V vectors and write their codes into the
 * paged code cache (AQPIM blog §3.1 step 3 and §5.2 item 2: the index of the
 * nearest codeword per subspace; §5.1 item 2: the cache stores indices).
 *
 * Token i uses codebook set token_set[i] and is written to page
 * slot_mapping[i] / P, slot slot_mapping[i] % P, for every kv head.  The
 * nearest codeword is decided exactly as in aq_fit_codebooks (fp32 squared
 * distance, plain order, lowest index on ties).  A negative slot_mapping entry
 * skips the token.  Out-of-range slots or sets set AQ_DEV_BAD_PAGE /
 * AQ_DEV_BAD_SET and skip the token.
 *
 *   kv_f16        in   fp16 [T][Hkv][2][D] (key then value of each token)
 *   token_set     in   int32 [T]
 *   slot_mapping  in   int64 [T]
 *   codebooks_f16 in   fp16 [num_sets][Hkv][2][M][K][Dsub]
 *   code_pages    out  uint8 [num_pages][Hkv][P][2][M] (only the named slots)
 *   device_status out  int32, ORed
 * ------------------------------------------------------------------------- */
aq_status aq_encode_append(const aq_pq_config *cfg, int32_t num_tokens,
                           int32_t num_kv_heads, const void *kv_f16,
                           const int32_t *token_set, const int64_t *slot_mapping,
                           const void *codebooks_f16, int64_t num_sets,
                           uint8_t *code_pages, int64_t num_pages,
                           int32_t *device_status, aq_stream_t stream);

/* ---------------------------------------------------------------------------
 * aq_decode_plan -- host-only: the split count and workspace a decode call
 * with these arguments will use (no CUDA call).  A split is one block of the
 * blockwise softmax of PAM article §2.2.3: its (max, sum, output) partials go
 * to the workspace and the combine merges them; how many blocks, and how many
 * CTAs share one, is this library's choice for the GPU, not the page's.
 *   num_splits_req  0 = choose automatically, else the requested count
 *   *num_splits     out: splits per (request, kv head)  (may be NULL)
 *   *cluster_size   out: CTAs cooperating on one split (may be NULL)
 *   *workspace_bytes out: bytes the call needs in `workspace` (may be NULL)
 * `fp16` selects the plan of aq_decode_attention_fp16.
 * Two PQ kernels exist: one whose cluster CTAs split the tokens and merge
 * their value bins, and one whose CTAs each score every token of their split
 * (used for GQA groups of 4 or more query heads per kv head).
 * A call runs at most 4096 splits and a CTA holds a bounded share of tokens,
 * so a PQ call has a longest request it can take: beyond it this function
 * and the decode calls return AQ_ERR_UNSUPPORTED (before any CUDA call).
 * With M = 4 and one query head per kv head that is 2^29 tokens with fp16
 * codebooks and 2^25 with E4M3 codebooks (which are not streamed); larger
 * groups hold fewer tokens per CTA.  The fp16 comparison call has no such
 * bound.  The
 * environment variable AQPQ_DECODE_KERNEL=1 or =2 forces the first or, where
 * its split fits, the second (read at every call; results agree within
 * rounding).
 * ------------------------------------------------------------------------- */
aq_status aq_decode_plan(const aq_pq_config *cfg, int32_t batch,
                         int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t max_seq_len, int32_t num_splits_req, int32_t fp16,
                         int32_t *num_splits, int32_t *cluster_size,
                         size_t *workspace_bytes);

/* ---------------------------------------------------------------------------
 * aq_decode_attention -- single-token PQ decode attention over the paged code
 * cache.
 *
 * For request b (codebook set req_set[b], seq_lens[b] cached tokens) and query
 * head h (kv head h / G, G = Hq / Hkv):
 *   LUT[m][k] = q[b][h][m*Dsub .. +Dsub) . C^K_m[k]          (per-query table)
 *   s_t       = scale * sum_m LUT[m][kcode(t, m)]
 *   p         = softmax(s) over t < seq_lens[b]
 *   out[b][h][m*Dsub + j] = sum_k ( sum_{t: vcode(t,m) = k} p_t ) * C^V_m[k][j]
 * i.e. exactly softmax attention over the reconstructed keys and values
 * (AQPIM blog §4 / §4.1 decomposition; PAM article §2.2.3 for the blockwise
 * softmax merged over splits).  seq_lens[b] == 0 gives the zero vector.
 * The current token must already be appended (aq_encode_append).
 *
 *   q             in   fp32 [B][Hq][D]
 *   code_pages    in   uint8 [num_pages][Hkv][P][2][M]
 *   codebooks_f16 in   fp16 [num_sets][Hkv][2][M][K][Dsub]
 *   req_set       in   int32 [B]
 *   block_table   in   int32 [B][max_pages]
 *   seq_lens      in   int32 [B]   (device)
 *   max_seq_len   host upper bound of seq_lens, <= max_pages * P; work is
 *                 planned for it, longer device lengths set AQ_DEV_BAD_LENGTH
 *   scale         softmax scale (1/sqrt(D) for standard attention)
 *   num_splits    0 = automatic, else splits per (request, kv head)
 *   out           out  fp32 [B][Hq][D]
 *   workspace     device scratch of >= the planned workspace_bytes (may be
 *                 NULL when that is 0); contents need no initialisation
 *   device_status out  int32, ORed
 * ------------------------------------------------------------------------- */
aq_status aq_decode_attention(const aq_pq_config *cfg, int32_t batch,
                              int32_t num_q_heads, int32_t num_kv_heads,
                              const float *q, const uint8_t *code_pages,
                              int64_t num_pages, const void *codebooks_f16,
                              int64_t num_sets, const int32_t *req_set,
                              const int32_t *block_table, int32_t max_pages,
                              const int32_t *seq_lens, int32_t max_seq_len,
                              float scale, int32_t num_splits, float *out,
                              void *workspace, size_t workspace_bytes,
                              int32_t *device_status, aq_stream_t stream);

/* ---------------------------------------------------------------------------
 * aq_decode_step -- one fused decode step: append each request's new token to
 * the PQ code cache, then the decode attention that includes it, in a single
 * launch that reads every codebook once (aq_encode_append followed by
 * aq_decode_attention read them twice).
 *
 * The new token of request b is the one at position seq_lens[b] - 1: its key
 * and value kv_new_f16[b] are encoded exactly as aq_encode_append does (AQPIM
 * blog §3.1 step 3) against set req_set[b] and written to page
 * block_table[b][(seq_lens[b]-1) / P], slot (seq_lens[b]-1) % P; the output is
 * aq_decode_attention's over all seq_lens[b] tokens.
 *
 *   kv_new_f16    in   fp16 [B][Hkv][2][D]
 *   code_pages    in/out (only the new tokens' slots are written)
 *   flags         AQ_STEP_OVERLAP: the call may start reading the codebooks,
 *                 req_set, seq_lens, block_table and code_pages before the
 *                 preceding kernel on `stream` has finished (programmatic
 *                 dependent launch); q and kv_new_f16 are read, and out,
 *                 code_pages, workspace and device_status written, only after
 *                 it.  Set it only when that kernel writes none of the five
 *                 inputs read early -- not, for example, right after another
 *                 aq_decode_step on the same code_pages.  0: plain stream
 *                 order.
 *                 AQ_STEP_E4M3: codebooks_f16 holds FP8 E4M3 codes (uint8,
 *                 same [S][Hkv][2][M][K][Dsub] layout, from
 *                 aq_codebooks_to_e4m3) instead of fp16 values: half the
 *                 codebook bytes.  The kernel widens them exactly to fp16, so
 *                 the step equals the fp16 step on the widened codebooks (and
 *                 the new token's codes equal aq_encode_append's on them).
 *   other arguments as aq_decode_attention.
 * ------------------------------------------------------------------------- */
#define AQ_STEP_OVERLAP 1
#define AQ_STEP_E4M3    2
aq_status aq_decode_step(const aq_pq_config *cfg, int32_t batch,
                         int32_t num_q_heads, int32_t num_kv_heads,
                         const float *q, const void *kv_new_f16,
                         uint8_t *code_pages, int64_t num_pages,
                         const void *codebooks_f16, int64_t num_sets,
                         const int32_t *req_set, const int32_t *block_table,
                         int32_t max_pages, const int32_t *seq_lens,
                         int32_t max_seq_len, float scale, int32_t num_splits,
                         int32_t flags, float *out, void *workspace,
                         size_t workspace_bytes, int32_t *device_status,
                         aq_stream_t stream);

/* ---------------------------------------------------------------------------
 * aq_decode_step_host -- aq_decode_step with the query, the new K/V and the
 * output in host memory (a serving loop's view: one call per step).  An
 * interface convenience of this library; the pages describe the step itself.
 *
 * Enqueues on `stream` the transfer of q_host [B][Hq][D] fp32 and kv_new_host
 * [B][Hkv][2][D] fp16 into the caller's device `staging`, the fused step, and
 * the transfer of the output into out_host [B][Hq][D] fp32.  Returns once they
 * are enqueued; out_host holds the step's output when the stream has passed
 * this point.  When all three buffers are page-locked host memory the device
 * can address (cudaHostAlloc / cudaMallocHost / cudaHostRegister) and all
 * three are 16-byte aligned, a gather kernel reads the inputs over
 * the host link into `staging`, the step starts as its programmatic dependent
 * and writes its output directly into out_host (no DMA copies); otherwise the
 * inputs and the output move by cudaMemcpyAsync (pageable buffers make those
 * copies synchronous).  Either way the host must not rewrite the inputs or
 * read the output until the stream has passed the step.  Every argument, the
 * step's included, is checked before anything is enqueued: a call that
 * returns an error has enqueued nothing and left `staging` untouched.
 *   staging        device memory of >= aq_decode_step_host_staging() bytes,
 *                  16-byte aligned, owned by the caller (no allocation here)
 *   flags          AQ_STEP_E4M3 only (AQ_STEP_OVERLAP is ignored: the step
 *                  follows its own input transfer)
 *   other arguments as aq_decode_step.
 * ------------------------------------------------------------------------- */
size_t aq_decode_step_host_staging(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads);
aq_status aq_decode_step_host(const aq_pq_config *cfg, int32_t batch, int32_t num_q_heads,
                              int32_t num_kv_heads, const float *q_host,
                              const void *kv_new_host, uint8_t *code_pages,
                              int64_t num_pages, const void *codebooks_f16,
                              int64_t num_sets, const int32_t *req_set,
                              const int32_t *block_table, int32_t max_pages,
                              const int32_t *seq_lens, int32_t max_seq_len, float scale,
                              int32_t num_splits, int32_t flags, float *out_host,
                              void *staging, size_t staging_bytes, void *workspace,
                              size_t workspace_bytes, int32_t *device_status,
                              aq_stream_t stream);

/* ---------------------------------------------------------------------------
 * aq_decode_attention_fp16 -- the uncompressed comparison point: the same
 * paged decode attention over an fp16 K/V cache (AQPIM blog §2.1 cache).
 * Only cfg->head_dim and cfg->page_size are used.
 *
 *   kv_pages_f16  in   fp16 [num_pages][Hkv][2][P][D]
 *   other arguments as aq_decode_attention.
 * ------------------------------------------------------------------------- */
aq_status aq_decode_attention_fp16(const aq_pq_config *cfg, int32_t batch,
                                   int32_t num_q_heads, int32_t num_kv_heads,
                                   const float *q, const void *kv_pages_f16,
                                   int64_t num_pages, const int32_t *block_table,
                                   int32_t max_pages, const int32_t *seq_lens,
                                   int32_t max_seq_len, float scale,
                                   int32_t num_splits, float *out,
                                   void *workspace, size_t workspace_bytes,
                                   int32_t *device_status, aq_stream_t stream);

/* ---------------------------------------------------------------------------
 * aq_decode_step_mixed -- one fused decode step over a cache kept at two
 * precisions, by kv head (AQPIM blog §6.1 item 4: keep the full-precision
 * cache for the most important heads, here kv heads [0, num_fp16_heads) and
 * their query heads; every other kv head is product-quantised).
 *
 * For kv head h < num_fp16_heads: the new key and value kv_new_f16[b][h] are
 * written into kv_pages_f16 at position seq_lens[b] - 1 and the attention is
 * aq_decode_attention_fp16's over the fp16 cache.  For kv head h >=
 * num_fp16_heads: aq_decode_step's over the PQ cache, whose pools hold only
 * those heads (pool head h - num_fp16_heads).  Both caches are addressed by
 * the same block table (a page id indexes either pool).  Query head j reads
 * kv head j / (Hq / Hkv) as everywhere.
 *
 *   q             in      fp32 [B][Hq][D]
 *   kv_new_f16    in      fp16 [B][Hkv][2][D]
 *   kv_pages_f16  in/out  fp16 [num_fp16_pages][num_fp16_heads][2][P][D]
 *   code_pages    in/out  uint8 [num_pages][Hkv - num_fp16_heads][P][2][M]
 *   codebooks     in      fp16 (or E4M3 codes with AQ_STEP_E4M3)
 *                         [num_sets][Hkv - num_fp16_heads][2][M][K][Dsub]
 *   out           out     fp32 [B][Hq][D]
 *   workspace     device scratch of >= aq_decode_step_mixed_workspace() bytes
 *   flags         AQ_STEP_OVERLAP (applies to the PQ heads' launch, with
 *                 aq_decode_step's contract), AQ_STEP_E4M3
 *   other arguments as aq_decode_step.  0 <= num_fp16_heads <= Hkv; with 0 the
 *   fp16 arguments may be NULL, with Hkv the PQ ones.  Up to four launches:
 *   the PQ step (+ its combine), the fp16 append, the fp16 attention (+ its
 *   combine).
 * ------------------------------------------------------------------------- */
aq_status aq_decode_step_mixed(const aq_pq_config *cfg, int32_t batch, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t num_fp16_heads,
                               const float *q, const void *kv_new_f16,
                               void *kv_pages_f16, int64_t num_fp16_pages,
                               uint8_t *code_pages, int64_t num_pages,
                               const void *codebooks, int64_t num_sets,
                               const int32_t *req_set, const int32_t *block_table,
                               int32_t max_pages, const int32_t *seq_lens,
                               int32_t max_seq_len, float scale, int32_t flags,
                               float *out, void *workspace, size_t workspace_bytes,
                               int32_t *device_status, aq_stream_t stream);

/* Host-only: the workspace bytes aq_decode_step_mixed needs for these
 * arguments (either codebook format). */
aq_status aq_decode_step_mixed_workspace(const aq_pq_config *cfg, int32_t batch,
                                         int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t num_fp16_heads, int32_t max_seq_len,
                                         size_t *workspace_bytes);

/* ---------------------------------------------------------------------------
 * aq_decode_attention_noalloc -- aq_decode_attention for callers that cannot
 * allocate device memory.  (The pages describe no such variant: it is an
 * interface convenience of this library.)
 *
 * Splitting long sequences needs device scratch for the per-split (max, sum,
 * output) partials, which aq_decode_attention takes from the caller.  A
 * caller that is handed only the call's tensors (a plugin or operator that
 * must not draw on the host framework's memory pool), whose device memory is
 * fully reserved elsewhere, or that runs where allocation is not allowed (it
 * can synchronise the device and can fail) uses this entry point instead: the
 * partials live in one fixed 4 MiB array owned by the library, which every GPU
 * that loads the library holds until the process exits.
 *
 * Arguments, layouts and results are those of aq_decode_attention without the
 * workspace.  A call whose planned scratch exceeds 4 MiB (batch * Hq * splits *
 * (D + 2) * 4 bytes) returns AQ_ERR_WORKSPACE_TOO_SMALL before any launch; no
 * call allocates or frees memory.  The array's device address is looked up
 * once per device by the first call made with that device current, so make
 * that first call before any stream capture.  The address is kept for the
 * life of the process: after cudaDeviceReset on a device it is stale, and this
 * entry point must not be called on that device again.  All calls share the
 * array: two calls whose kernels overlap on the GPU (other streams, other host
 * threads) race on it.  Nothing in it needs clearing between calls.
 * ------------------------------------------------------------------------- */
aq_status aq_decode_attention_noalloc(const aq_pq_config *cfg, int32_t batch,
                                      int32_t num_q_heads, int32_t num_kv_heads,
                                      const float *q, const uint8_t *code_pages,
                                      int64_t num_pages, const void *codebooks_f16,
                                      int64_t num_sets, const int32_t *req_set,
                                      const int32_t *block_table, int32_t max_pages,
                                      const int32_t *seq_lens, int32_t max_seq_len,
                                      float scale, int32_t num_splits, float *out,
                                      int32_t *device_status, aq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* AQPQ_H */
