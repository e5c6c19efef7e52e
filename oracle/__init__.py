"""CPU oracle for PQ-compressed KV-cache decode attention.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product (``decode_attention_product_gb300``) never imports it and
the two share no code: this module wraps ``aq_oracle.c`` (plain C loops, fp64)
with numpy marshalling and nothing else.

What each function computes, and the passage it follows, is stated in
``aq_oracle.c``:

* ``pq_encode`` / ``encode_append``: nearest codeword per subspace (AQPIM blog
  §3.1, §5.2 item 2), decided in float, ties to the lowest index, with the
  relative runner-up gap.
* ``pq_reconstruct``: concatenation of the indexed codewords (AQPIM blog §3.1).
* ``attention_dense`` / ``attention_split_merge``: single-pass softmax
  attention and the blockwise (max, sum) merge (PAM article §2.2.3).
* ``decode_attention`` / ``decode_attention_fp16``: paged PQ (resp. fp16)
  decode attention, decompress-then-compute (AQPIM blog §4).
* ``decode_attention_mixed``: fp16 attention for the first kv heads, PQ for
  the rest (AQPIM blog §6.1 item 4).
* ``kmeans_fit`` / ``kmeans_step``: Lloyd k-means codebook fit (AQPIM blog
  §3.2 item 2, §5.2 item 1); ``kmeans_distortion``: its objective.
* ``kmeans_refine``: the periodic refresh, Lloyd steps on recent vectors
  seeded from the codebook in use (AQPIM blog §6.1 item 3).
* ``e4m3_from_float`` / ``e4m3_to_float``: FP8 E4M3 codebook storage, nearest
  with ties to even, saturating at 448 (AQPIM blog §4.2).

Floating-point inputs given as fp16 are widened exactly; results come back in
float64 (``kmeans_fit`` also returns the fp16 round-to-nearest-even codebook).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "aq_oracle.c")

_lib = None


def build(force: bool = False) -> str:
    """Compile aq_oracle.c into oracle/_build/liboracle.so with gcc (+OpenMP).

    -ffp-contract=off keeps the float distance sums free of fused
    multiply-adds, so the decision arithmetic is the same on x86 and Arm.
    """
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    # a temporary of this process's own, renamed into place at once: builds
    # in parallel processes never write the same file
    tmp = f"{_SO}.{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        sig = {
            "oracle_num_threads": ([], ctypes.c_int),
            "oracle_set_num_threads": ([ctypes.c_int], None),
            "oracle_pq_encode": ([i64, i32, i32, i32, P, P, P, P], None),
            "oracle_encode_append": ([i32, i32, i32, i32, i32, i32, P, P, P, P, P, P], None),
            "oracle_pq_reconstruct": ([i64, i32, i32, i32, P, P, P], None),
            "oracle_attention_dense": ([i32, i32, P, P, P, dbl, P], None),
            "oracle_attention_split_merge": ([i32, i32, P, P, P, dbl, i32, P, P], None),
            "oracle_decode_attention": ([i32] * 7 + [P, P, P, P, P, i32, P, dbl, P], None),
            "oracle_decode_attention_fp16": ([i32] * 5 + [P, P, P, i32, P, dbl, P], None),
            "oracle_kmeans_fit": ([i64, i32, i32, i32, i32, i32, P, P, P, P], None),
            "oracle_kmeans_refine": ([i64, i32, i32, i32, i32, i32, P, P, P, P], None),
            "oracle_kmeans_step": ([i64, i32, i32, i32, i32, P, P, P, P, P], None),
            "oracle_kmeans_distortion": ([i32, i32, i32, i32, i32, P, P], dbl),
            "oracle_e4m3_from_float": ([i64, P, P], None),
            "oracle_e4m3_to_float": ([i64, P, P], None),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def pq_encode(x, codebook, *, with_gap=False):
    """Codes [n][M] (int32) of vectors x [n][D] against codebook [M][K][Dsub]."""
    x = _c(x, np.float32)
    cb = _c(codebook, np.float32)
    M, K, Dsub = cb.shape
    n, D = x.shape
    assert D == M * Dsub
    codes = np.zeros((n, M), np.int32)
    gap = np.zeros((n, M), np.float32) if with_gap else None
    _load().oracle_pq_encode(n, D, M, K, _p(x), _p(cb), _p(codes), _p(gap))
    return (codes, gap) if with_gap else codes


def encode_append(kv, token_set, slot_mapping, codebooks, code_pages, page_size):
    """Encode kv [T][Hkv][2][D] into code_pages [NP][Hkv][P][2][M] (in place).

    Returns the relative gaps [T][Hkv][2][M].
    """
    kv = _c(kv, np.float32)
    cbs = _c(codebooks, np.float32)
    T, Hkv, _, D = kv.shape
    _, _, _, M, K, Dsub = cbs.shape
    assert code_pages.dtype == np.uint8 and code_pages.flags.c_contiguous
    gap = np.zeros((T, Hkv, 2, M), np.float32)
    _load().oracle_encode_append(
        T, Hkv, D, M, K, page_size, _p(kv), _p(_c(token_set, np.int32)),
        _p(_c(slot_mapping, np.int64)), _p(cbs), _p(code_pages), _p(gap))
    return gap


def pq_reconstruct(codebook, codes):
    cb = _c(codebook, np.float64)
    M, K, Dsub = cb.shape
    codes = _c(codes, np.uint8)
    out = np.zeros((codes.shape[0], M * Dsub), np.float64)
    _load().oracle_pq_reconstruct(codes.shape[0], M * Dsub, M, K, _p(cb), _p(codes), _p(out))
    return out


def attention_dense(q, k, v, scale):
    q = _c(q, np.float64); k = _c(k, np.float64); v = _c(v, np.float64)
    out = np.zeros(q.shape[0], np.float64)
    _load().oracle_attention_dense(k.shape[0], q.shape[0], _p(q), _p(k), _p(v), scale, _p(out))
    return out


def attention_split_merge(q, k, v, scale, bounds):
    q = _c(q, np.float64); k = _c(k, np.float64); v = _c(v, np.float64)
    b = _c(bounds, np.int32)
    out = np.zeros(q.shape[0], np.float64)
    _load().oracle_attention_split_merge(k.shape[0], q.shape[0], _p(q), _p(k), _p(v),
                                         scale, len(b) - 1, _p(b), _p(out))
    return out


def decode_attention(q, code_pages, codebooks, req_set, block_table, seq_lens, scale,
                     page_size):
    """PQ decode attention; returns float64 [B][Hq][D]."""
    q = _c(q, np.float64)
    B, Hq, D = q.shape
    cp = _c(code_pages, np.uint8)
    cbs = _c(codebooks, np.float64)
    _, Hkv, _, M, K, Dsub = cbs.shape
    bt = _c(block_table, np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    _load().oracle_decode_attention(
        B, Hq, Hkv, D, M, K, page_size, _p(q), _p(cp), _p(cbs), _p(_c(req_set, np.int32)),
        _p(bt), bt.shape[1], _p(_c(seq_lens, np.int32)), scale, _p(out))
    return out


def decode_attention_fp16(q, kv_pages, block_table, seq_lens, scale):
    """fp16-cache decode attention; kv_pages [NP][Hkv][2][P][D]."""
    q = _c(q, np.float64)
    B, Hq, D = q.shape
    kvp = _c(kv_pages, np.float64)
    _, Hkv, _, P, _ = kvp.shape
    bt = _c(block_table, np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    _load().oracle_decode_attention_fp16(
        B, Hq, Hkv, D, P, _p(q), _p(kvp), _p(bt), bt.shape[1],
        _p(_c(seq_lens, np.int32)), scale, _p(out))
    return out


def decode_attention_mixed(q, kv_pages_f16, code_pages, codebooks, req_set, block_table, seq_lens,
                           scale, page_size, num_fp16_heads):
    """Decode attention over a cache kept at two precisions by kv head (AQPIM
    blog §6.1 item 4: the full-precision cache kept for the most important
    heads): kv heads [0, num_fp16_heads) attend over their fp16 pages
    kv_pages_f16 [NP][n16][2][P][D] exactly as decode_attention_fp16, the
    others over their PQ cache (pools of Hkv - n16 heads) exactly as
    decode_attention.  Query head j reads kv head j / G.  float64 [B][Hq][D].
    """
    q = np.asarray(q)
    B, Hq, D = q.shape
    n16 = int(num_fp16_heads)
    Hpq = codebooks.shape[1] if codebooks is not None else 0
    Hkv = n16 + Hpq
    assert Hq % Hkv == 0
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), np.float64)
    if n16 > 0:
        out[:, :n16 * G] = decode_attention_fp16(q[:, :n16 * G], kv_pages_f16, block_table, seq_lens, scale)
    if Hpq > 0:
        out[:, n16 * G:] = decode_attention(q[:, n16 * G:], code_pages, codebooks, req_set, block_table,
                                            seq_lens, scale, page_size)
    return out


def e4m3_from_float(x):
    """FP8 E4M3 codes (uint8, same shape) of x: nearest, ties to even, |x| > 448
    saturated, NaN -> 0x7F."""
    x = np.asarray(x, np.float32)
    xc = _c(x.reshape(-1), np.float32)
    out = np.zeros(xc.shape, np.uint8)
    _load().oracle_e4m3_from_float(xc.size, _p(xc), _p(out))
    return out.reshape(x.shape)


def e4m3_to_float(codes):
    """Values (float32, same shape) of FP8 E4M3 codes."""
    c = np.asarray(codes, np.uint8)
    cc = _c(c.reshape(-1), np.uint8)
    out = np.zeros(cc.shape, np.float32)
    _load().oracle_e4m3_to_float(cc.size, _p(cc), _p(out))
    return out.reshape(c.shape)


def kmeans_fit(samples, M, K, iters):
    """Fit codebooks on samples [U][N][D].

    Returns (codebook_f16 [U][M][K][Dsub], centroids_f64, assign [U][N][M],
    min_gap [U][M]).
    """
    x = _c(samples, np.float32)
    U, N, D = x.shape
    Dsub = D // M
    cent = np.zeros((U, M, K, Dsub), np.float64)
    assign = np.zeros((U, N, M), np.int32)
    mg = np.zeros((U, M), np.float32)
    _load().oracle_kmeans_fit(U, D, M, K, N, iters, _p(x), _p(cent), _p(assign), _p(mg))
    return cent.astype(np.float16), cent, assign, mg


def kmeans_refine(samples, codebook16, iters):
    """Refresh codebooks [U][M][K][Dsub] (fp16 values) with `iters` Lloyd steps on
    samples [U][N][D], starting from the codebook.

    Returns (codebook_f16, centroids_f64, assign [U][N][M], min_gap [U][M]).
    """
    x = _c(samples, np.float32)
    U, N, D = x.shape
    cent = _c(np.asarray(codebook16, np.float16), np.float64)
    _, M, K, Dsub = cent.shape
    assert cent.shape[0] == U and M * Dsub == D
    assign = np.zeros((U, N, M), np.int32)
    mg = np.zeros((U, M), np.float32)
    _load().oracle_kmeans_refine(U, D, M, K, N, iters, _p(x), _p(cent), _p(assign), _p(mg))
    return cent.astype(np.float16), cent, assign, mg


def kmeans_step(samples, centroids):
    """One Lloyd step from float centroids [U][M][K][Dsub].

    Returns (assign [U][N][M], centroids_out float64, gap [U][N][M]).
    """
    x = _c(samples, np.float32)
    c = _c(centroids, np.float32)
    U, N, D = x.shape
    _, M, K, Dsub = c.shape
    assign = np.zeros((U, N, M), np.int32)
    out = np.zeros(c.shape, np.float64)
    gap = np.zeros((U, N, M), np.float32)
    _load().oracle_kmeans_step(U, D, M, K, N, _p(x), _p(c), _p(assign), _p(out), _p(gap))
    return assign, out, gap


def kmeans_distortion(samples_u, centroids_m, M, m):
    """Mean squared error of samples [N][D] against subspace m's centroids."""
    x = _c(samples_u, np.float32)
    c = _c(centroids_m, np.float64)
    N, D = x.shape
    return float(_load().oracle_kmeans_distortion(N, D, M, c.shape[0], m, _p(x), _p(c)))
