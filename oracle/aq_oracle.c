/*
 * aq_oracle.c -- plain, slow CPU oracle for product-quantised (PQ) KV-cache
 * decode attention.  TEST INFRASTRUCTURE ONLY: it is compiled into
 * oracle/_build/liboracle.so and may be loaded only by tests/, by
 * __graft_entry__.smoke() and by the cpu_baseline and --impl reference legs
 * of bench.py.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * Sources (cited by page title and section):
 *   "AQPIM blog" = devpress.csdn.net, "当大模型推理撞上内存墙" (adaptive product
 *                  quantisation + processing-in-memory)
 *   "PAM article" = maplevalley.com.cn, "大语言模型KV缓存优化与PAM架构实践"
 *   "NMC ch.1"    = zsc.github.io near_memory_computing, chapter 1
 *
 * Precision: every floating-point result is computed in double from the exact
 * fp16 / fp32 inputs, except where a float decides an integer (the nearest
 * codeword in encode and in the k-means assignment).  There the squared
 * distance is accumulated in float in the plain order j = 0..Dsub-1, which is
 * the precision the GPU kernels decide in; the relative gap to the runner-up is
 * reported so that tests compare indices only outside the near-tie band.
 *
 * Layouts (row-major, contiguous), with D = head_dim, M = subspaces,
 * Dsub = D / M, K = codewords per subspace, P = tokens per page:
 *   codebooks  [S][Hkv][2][M][K][Dsub]   (the [2] axis is K then V)
 *   code_pages [NP][Hkv][P][2][M]        (uint8 codes, K codes then V codes)
 *   kv_pages   [NP][Hkv][2][P][D]        (raw fp16 cache, as double here)
 *   block_table[B][max_pages], token t of request b sits in page
 *   block_table[b][t / P], slot t % P.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Nearest codeword.  AQPIM blog §3.1 (step 3, "which classic paragraph is it
 * closest to") and §5.2 item 2 (encode = find the nearest codeword).  Squared
 * Euclidean distance, accumulated in float; ties go to the lowest index.
 * The gap is (d2 - d1) / d2, where d2 is the smallest distance among codewords
 * whose (float) vector differs from the winner's vector; +inf when there is no
 * such codeword or d2 == 0.                                                 */
static int nearest_codeword(int K, int Dsub, const float *x, const float *cb,
                            float *gap_out) {
    int best = 0;
    float d1 = INFINITY;
    for (int k = 0; k < K; ++k) {
        float d = 0.0f;
        for (int j = 0; j < Dsub; ++j) {
            float e = x[j] - cb[(size_t)k * Dsub + j];
            d = d + e * e;
        }
        if (d < d1) { d1 = d; best = k; }
    }
    if (gap_out) {
        float d2 = INFINITY;
        const float *w = cb + (size_t)best * Dsub;
        for (int k = 0; k < K; ++k) {
            const float *c = cb + (size_t)k * Dsub;
            if (memcmp(c, w, sizeof(float) * (size_t)Dsub) == 0) continue;
            float d = 0.0f;
            for (int j = 0; j < Dsub; ++j) {
                float e = x[j] - c[j];
                d = d + e * e;
            }
            if (d < d2) d2 = d;
        }
        *gap_out = (isinf(d2) || d2 <= 0.0f) ? INFINITY : (d2 - d1) / d2;
    }
    return best;
}

/* Encode a batch of vectors against one codebook [M][K][Dsub]: AQPIM blog
 * §3.1 (split into M contiguous sub-vectors; index of the nearest codeword). */
void oracle_pq_encode(int64_t n, int D, int M, int K, const float *x,
                      const float *cb, int32_t *codes, float *gap) {
    const int Dsub = D / M;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        for (int m = 0; m < M; ++m) {
            float g;
            codes[i * M + m] = nearest_codeword(
                K, Dsub, x + i * D + (size_t)m * Dsub,
                cb + (size_t)m * K * Dsub, gap ? &g : NULL);
            if (gap) gap[i * M + m] = g;
        }
    }
}

/* Encode-and-append: token i (request set token_set[i], every kv head, K and V)
 * is encoded and its codes written to page slot slot_mapping[i] (= page * P +
 * slot).  AQPIM blog §5.1 item 2 (the quantised cache stores integer indices)
 * and PAM article §2.2.2 (paged KV cache, global block table).
 *   kv        [T][Hkv][2][D]  (exact fp16 values, as float)
 *   codebooks [S][Hkv][2][M][K][Dsub] (exact fp16 values, as float)
 *   code_pages[NP][Hkv][P][2][M] (written; untouched elsewhere)
 *   gap       [T][Hkv][2][M] or NULL
 * A negative slot marks a padding token: it is skipped (its gap entries are
 * left as they were).                                                      */
void oracle_encode_append(int T, int Hkv, int D, int M, int K, int P,
                          const float *kv, const int32_t *token_set,
                          const int64_t *slot_mapping, const float *codebooks,
                          uint8_t *code_pages, float *gap) {
    const int Dsub = D / M;
    const size_t cb_stride = (size_t)M * K * Dsub;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        if (slot_mapping[t] < 0) continue;        /* padding token: nothing to store */
        const int64_t page = slot_mapping[t] / P, slot = slot_mapping[t] % P;
        for (int h = 0; h < Hkv; ++h) {
            for (int w = 0; w < 2; ++w) {
                const float *x = kv + (((size_t)t * Hkv + h) * 2 + w) * D;
                const float *cb = codebooks +
                    (((size_t)token_set[t] * Hkv + h) * 2 + w) * cb_stride;
                for (int m = 0; m < M; ++m) {
                    float g;
                    int c = nearest_codeword(K, Dsub, x + (size_t)m * Dsub,
                                             cb + (size_t)m * K * Dsub, &g);
                    code_pages[(((size_t)page * Hkv + h) * P + slot) * 2 * M +
                               (size_t)w * M + m] = (uint8_t)c;
                    if (gap) gap[(((size_t)t * Hkv + h) * 2 + w) * M + m] = g;
                }
            }
        }
    }
}

/* FP8 E4M3 codebook storage (AQPIM blog §4.2: codebooks kept in a low-precision
 * float such as FP8).  The OCP E4M3 format: 1 sign bit, 4 exponent bits (bias
 * 7), 3 fraction bits; exponent field 0 holds the subnormals m * 2^-9; no
 * infinities; S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 * 2^8 = 448.
 * Value of one code.                                                         */
static double e4m3_value(uint8_t b) {
    const int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest code, ties to the even fraction, magnitudes beyond 448 (and
 * infinities) saturated to 448; NaN gives 0x7F.                              */
static uint8_t e4m3_round(double x) {
    if (isnan(x)) return 0x7F;
    const uint8_t s = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a == 0.0) return s;        /* +0 / -0 */
    if (a >= 448.0) return s | 0x7E;
    int e;
    frexp(a, &e);                  /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                        /* a in [2^e, 2^(e+1)) */
    if (e < -6) e = -6;            /* subnormal spacing below 2^-6 */
    double q = nearbyint(ldexp(a, 3 - e));   /* units of 2^(e-3), half to even */
    if (q >= 16.0) { q = 8.0; e += 1; }      /* rounded up into the next binade */
    if (e == -6 && q < 8.0) return s | (uint8_t)q;          /* subnormal (or zero) */
    const int code = ((e + 7) << 3) | ((int)q - 8);
    if (code > 0x7E) return s | 0x7E;        /* 480 would be the NaN pattern */
    return s | (uint8_t)code;
}

void oracle_e4m3_from_float(int64_t n, const float *x, uint8_t *codes) {
    for (int64_t i = 0; i < n; ++i) codes[i] = e4m3_round((double)x[i]);
}

void oracle_e4m3_to_float(int64_t n, const uint8_t *codes, float *x) {
    for (int64_t i = 0; i < n; ++i) x[i] = (float)e4m3_value(codes[i]);
}

/* Reconstruction: x̂[m*Dsub + j] = C_m[c_m][j].  AQPIM blog §3.1 ("take the
 * codeword each index points to and concatenate").                          */
void oracle_pq_reconstruct(int64_t n, int D, int M, int K, const double *cb,
                           const uint8_t *codes, double *out) {
    const int Dsub = D / M;
    for (int64_t i = 0; i < n; ++i)
        for (int m = 0; m < M; ++m)
            for (int j = 0; j < Dsub; ++j)
                out[i * D + (size_t)m * Dsub + j] =
                    cb[((size_t)m * K + codes[i * M + m]) * Dsub + j];
}

/* Textbook single-pass softmax attention for one query:
 *   s_t = scale * <q, k_t>,  p = softmax(s),  out = sum_t p_t v_t.
 * NMC ch.1 §1.1.2 (Q·K^T, softmax, Score·V for one decode token).
 * L == 0 yields the zero vector (empty sum; a convention shared with the
 * kernels).                                                                 */
void oracle_attention_dense(int L, int D, const double *q, const double *Kx,
                            const double *Vx, double scale, double *out) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (L <= 0) return;
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    double mx = -INFINITY;
    for (int t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * Kx[(size_t)t * D + d];
        s[t] = scale * acc;
        if (s[t] > mx) mx = s[t];
    }
    double z = 0.0;
    for (int t = 0; t < L; ++t) { s[t] = exp(s[t] - mx); z += s[t]; }
    for (int t = 0; t < L; ++t)
        for (int d = 0; d < D; ++d) out[d] += s[t] * Vx[(size_t)t * D + d];
    for (int d = 0; d < D; ++d) out[d] /= z;
    free(s);
}

/* Blockwise online softmax with (max, sum) statistics per block, merged by a
 * reduction: PAM article §2.2.3 item 1 (PAMattention), NMC ch.1 §1.5.2
 * (FlashAttention blocks).  bounds[0..nsplit] are the token boundaries; a
 * block may be empty.  Used only to pin the single-pass result above.       */
void oracle_attention_split_merge(int L, int D, const double *q,
                                  const double *Kx, const double *Vx,
                                  double scale, int nsplit,
                                  const int32_t *bounds, double *out) {
    double *m = (double *)malloc(sizeof(double) * (size_t)nsplit);
    double *l = (double *)malloc(sizeof(double) * (size_t)nsplit);
    double *o = (double *)calloc((size_t)nsplit * D, sizeof(double));
    for (int sp = 0; sp < nsplit; ++sp) {
        m[sp] = -INFINITY;
        l[sp] = 0.0;
        for (int t = bounds[sp]; t < bounds[sp + 1]; ++t) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += q[d] * Kx[(size_t)t * D + d];
            if (scale * acc > m[sp]) m[sp] = scale * acc;
        }
        for (int t = bounds[sp]; t < bounds[sp + 1]; ++t) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += q[d] * Kx[(size_t)t * D + d];
            double p = exp(scale * acc - m[sp]);
            l[sp] += p;
            for (int d = 0; d < D; ++d) o[(size_t)sp * D + d] += p * Vx[(size_t)t * D + d];
        }
    }
    double gm = -INFINITY;
    for (int sp = 0; sp < nsplit; ++sp) if (m[sp] > gm) gm = m[sp];
    double z = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int sp = 0; sp < nsplit; ++sp) {
        if (l[sp] == 0.0) continue;            /* empty block contributes 0 */
        double w = exp(m[sp] - gm);
        z += w * l[sp];
        for (int d = 0; d < D; ++d) out[d] += w * o[(size_t)sp * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] = (z > 0.0) ? out[d] / z : 0.0;
    free(m); free(l); free(o);
}

/* PQ decode attention over a paged code cache, decompress-then-compute (the
 * plain flow of AQPIM blog §4 steps 1-3): for each request b and query head h
 * with kv head h / (Hq / Hkv) (GQA, NMC ch.1 §1.4.3), reconstruct every cached
 * key and value from its codes and the request's codebook set req_set[b], then
 * run textbook softmax attention.
 *   q          [B][Hq][D]
 *   code_pages [NP][Hkv][P][2][M]
 *   codebooks  [S][Hkv][2][M][K][Dsub]  (exact fp16 values, as double)
 *   out        [B][Hq][D]                                                  */
void oracle_decode_attention(int B, int Hq, int Hkv, int D, int M, int K, int P,
                             const double *q, const uint8_t *code_pages,
                             const double *codebooks, const int32_t *req_set,
                             const int32_t *block_table, int max_pages,
                             const int32_t *seq_lens, double scale, double *out) {
    const int G = Hq / Hkv, Dsub = D / M;
    const size_t cb_stride = (size_t)M * K * Dsub;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            const int kvh = h / G, L = seq_lens[b];
            double *Kx = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
            double *Vx = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
            const double *cbK = codebooks + (((size_t)req_set[b] * Hkv + kvh) * 2 + 0) * cb_stride;
            const double *cbV = codebooks + (((size_t)req_set[b] * Hkv + kvh) * 2 + 1) * cb_stride;
            for (int t = 0; t < L; ++t) {
                const size_t page = (size_t)block_table[(size_t)b * max_pages + t / P];
                const uint8_t *c = code_pages + ((page * Hkv + kvh) * P + t % P) * 2 * M;
                oracle_pq_reconstruct(1, D, M, K, cbK, c, Kx + (size_t)t * D);
                oracle_pq_reconstruct(1, D, M, K, cbV, c + M, Vx + (size_t)t * D);
            }
            oracle_attention_dense(L, D, q + ((size_t)b * Hq + h) * D, Kx, Vx,
                                   scale, out + ((size_t)b * Hq + h) * D);
            free(Kx); free(Vx);
        }
    }
}

/* The uncompressed comparison point: the same attention over raw fp16 K/V
 * pages.  AQPIM blog §2.1 (the fp16 KV cache).
 *   kv_pages [NP][Hkv][2][P][D] (exact fp16 values, as double)             */
void oracle_decode_attention_fp16(int B, int Hq, int Hkv, int D, int P,
                                  const double *q, const double *kv_pages,
                                  const int32_t *block_table, int max_pages,
                                  const int32_t *seq_lens, double scale,
                                  double *out) {
    const int G = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            const int kvh = h / G, L = seq_lens[b];
            double *Kx = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
            double *Vx = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
            for (int t = 0; t < L; ++t) {
                const size_t page = (size_t)block_table[(size_t)b * max_pages + t / P];
                for (int d = 0; d < D; ++d) {
                    Kx[(size_t)t * D + d] = kv_pages[(((page * Hkv + kvh) * 2 + 0) * P + t % P) * D + d];
                    Vx[(size_t)t * D + d] = kv_pages[(((page * Hkv + kvh) * 2 + 1) * P + t % P) * D + d];
                }
            }
            oracle_attention_dense(L, D, q + ((size_t)b * Hq + h) * D, Kx, Vx,
                                   scale, out + ((size_t)b * Hq + h) * D);
            free(Kx); free(Vx);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Lloyd k-means for one subspace of one unit.  AQPIM blog §3.2 item 2 and
 * §5.2 item 1 (codebooks initialised online from the first tokens of the
 * sequence with a quick k-means on a small sample set).
 *   x      [N][D] sample vectors (exact fp16 values, as float); this
 *          subspace's coordinates are x[n][off .. off + Dsub)
 *   cent   [K][Dsub] double, in: current centroids, out: updated centroids
 *   assign [N] out: nearest centroid of each sample (decided in float on the
 *          float-rounded centroids, ties to the lowest index)
 *   gap    [N] out (may be NULL): relative runner-up gap of each decision
 * One step = assign every sample, then move each centroid to the mean of its
 * members; a centroid with no member keeps its value.                      */
static void kmeans_one_step(int N, int D, int off, int K, int Dsub,
                            const float *x, double *cent, int32_t *assign,
                            float *gap, float *xs, float *cf, double *sum,
                            int64_t *cnt) {
    for (int k = 0; k < K * Dsub; ++k) cf[k] = (float)cent[k];
    for (int n = 0; n < N; ++n) {
        for (int j = 0; j < Dsub; ++j) xs[j] = x[(size_t)n * D + off + j];
        float g;
        assign[n] = nearest_codeword(K, Dsub, xs, cf, gap ? &g : NULL);
        if (gap) gap[n] = g;
    }
    for (int k = 0; k < K * Dsub; ++k) sum[k] = 0.0;
    for (int k = 0; k < K; ++k) cnt[k] = 0;
    for (int n = 0; n < N; ++n) {
        cnt[assign[n]] += 1;
        for (int j = 0; j < Dsub; ++j)
            sum[(size_t)assign[n] * Dsub + j] += (double)x[(size_t)n * D + off + j];
    }
    for (int k = 0; k < K; ++k)
        if (cnt[k] > 0)
            for (int j = 0; j < Dsub; ++j)
                cent[(size_t)k * Dsub + j] = sum[(size_t)k * Dsub + j] / (double)cnt[k];
}

/* Run `iters` Lloyd steps for every unit u and subspace m.  With
 * from_samples, centroid k starts as sample (k mod N); otherwise it starts as
 * the value already in `centroids`.                                          */
static void kmeans_run(int64_t U, int D, int M, int K, int N, int iters, int from_samples,
                       const float *samples, double *centroids, int32_t *assign,
                       float *min_gap) {
    const int Dsub = D / M;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t u = 0; u < U; ++u) {
        for (int m = 0; m < M; ++m) {
            const float *x = samples + (size_t)u * N * D;
            double *cent = centroids + ((size_t)u * M + m) * K * Dsub;
            float *xs = (float *)malloc(sizeof(float) * (size_t)Dsub);
            float *cf = (float *)malloc(sizeof(float) * (size_t)K * Dsub);
            double *sum = (double *)malloc(sizeof(double) * (size_t)K * Dsub);
            int64_t *cnt = (int64_t *)malloc(sizeof(int64_t) * (size_t)K);
            int32_t *a = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
            float *g = (float *)malloc(sizeof(float) * (size_t)N);
            if (from_samples)
                for (int k = 0; k < K; ++k)
                    for (int j = 0; j < Dsub; ++j)
                        cent[(size_t)k * Dsub + j] = (double)x[(size_t)(k % N) * D + (size_t)m * Dsub + j];
            float mg = INFINITY;
            for (int it = 0; it < iters; ++it) {
                kmeans_one_step(N, D, m * Dsub, K, Dsub, x, cent, a, g, xs, cf, sum, cnt);
                for (int n = 0; n < N; ++n) if (g[n] < mg) mg = g[n];
            }
            for (int n = 0; n < N; ++n) assign[((size_t)u * N + n) * M + m] = a[n];
            if (min_gap) min_gap[(size_t)u * M + m] = mg;
            free(xs); free(cf); free(sum); free(cnt); free(a); free(g);
        }
    }
}

/* Codebook fit: for every unit u (one request/layer, kv head, K-or-V) and every
 * subspace m, initialise centroid k to sample (k mod N) and run `iters` Lloyd
 * steps.
 *   samples   [U][N][D]   (exact fp16 values, as float)
 *   centroids [U][M][K][Dsub] out, double (the caller rounds to fp16)
 *   assign    [U][N][M] out: the assignment of the last step (iters >= 1)
 *   min_gap   [U][M] out (may be NULL): smallest relative runner-up gap met
 *             in any assignment decision of any step                       */
void oracle_kmeans_fit(int64_t U, int D, int M, int K, int N, int iters,
                       const float *samples, double *centroids,
                       int32_t *assign, float *min_gap) {
    kmeans_run(U, D, M, K, N, iters, 1, samples, centroids, assign, min_gap);
}

/* Codebook refresh (AQPIM blog §6.1 item 3: a few k-means iterations on the
 * recent vectors, starting from the codebook in use): the fit's steps with
 * centroid k starting at row k of the given codebook.
 *   centroids [U][M][K][Dsub] double, in: the codebook (exact fp16 values),
 *             out: the refined centroids (the caller rounds to fp16)
 * other arguments as for oracle_kmeans_fit.                                 */
void oracle_kmeans_refine(int64_t U, int D, int M, int K, int N, int iters,
                          const float *samples, double *centroids,
                          int32_t *assign, float *min_gap) {
    kmeans_run(U, D, M, K, N, iters, 0, samples, centroids, assign, min_gap);
}

/* One Lloyd step from given float centroids (the step-parity check).
 *   centroids_in  [U][M][K][Dsub] float
 *   assign        [U][N][M] out;  gap [U][N][M] out (may be NULL)
 *   centroids_out [U][M][K][Dsub] double out                               */
void oracle_kmeans_step(int64_t U, int D, int M, int K, int N,
                        const float *samples, const float *centroids_in,
                        int32_t *assign, double *centroids_out, float *gap) {
    const int Dsub = D / M;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t u = 0; u < U; ++u) {
        for (int m = 0; m < M; ++m) {
            const float *x = samples + (size_t)u * N * D;
            double *cent = centroids_out + ((size_t)u * M + m) * K * Dsub;
            const float *cin = centroids_in + ((size_t)u * M + m) * K * Dsub;
            float *xs = (float *)malloc(sizeof(float) * (size_t)Dsub);
            float *cf = (float *)malloc(sizeof(float) * (size_t)K * Dsub);
            double *sum = (double *)malloc(sizeof(double) * (size_t)K * Dsub);
            int64_t *cnt = (int64_t *)malloc(sizeof(int64_t) * (size_t)K);
            int32_t *a = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
            float *g = (float *)malloc(sizeof(float) * (size_t)N);
            for (int k = 0; k < K * Dsub; ++k) cent[k] = (double)cin[k];
            kmeans_one_step(N, D, m * Dsub, K, Dsub, x, cent, a, g, xs, cf, sum, cnt);
            for (int n = 0; n < N; ++n) {
                assign[((size_t)u * N + n) * M + m] = a[n];
                if (gap) gap[((size_t)u * N + n) * M + m] = g[n];
            }
            free(xs); free(cf); free(sum); free(cnt); free(a); free(g);
        }
    }
}

/* Mean squared quantisation error of samples against centroids (the k-means
 * objective), in double; used by the monotonicity pin.                      */
double oracle_kmeans_distortion(int N, int D, int M, int K, int m,
                                const float *x, const double *cent) {
    const int Dsub = D / M;
    double tot = 0.0;
    for (int n = 0; n < N; ++n) {
        double best = INFINITY;
        for (int k = 0; k < K; ++k) {
            double d = 0.0;
            for (int j = 0; j < Dsub; ++j) {
                double e = (double)x[(size_t)n * D + (size_t)m * Dsub + j] - cent[(size_t)k * Dsub + j];
                d += e * e;
            }
            if (d < best) best = d;
        }
        tot += best;
    }
    return tot / N;
}
