"""Algorithmic byte and FLOP counts for PQ and fp16 decode attention.

Pure host arithmetic (no CUDA): the numbers the benchmark divides by kernel
time to report GB/s and the roofline fraction.  "Algorithmic" means the bytes
the method must move at least once per call, not what a kernel happens to move.

Sources: AQPIM blog §2.1 (fp16 KV-cache size per step and per layer), §3.2
(codebook size), §3.3 (256 B -> M B per vector); Near-memory computing ch.1
§1.1.2 (attention FLOPs per decode token), §1.4.1 (KV growth model).
"""
from __future__ import annotations

import numpy as np

FP16 = 2
FP32 = 4
INT32 = 4


def fp16_cache_bytes(batch: int, heads: int, head_dim: int, tokens: int) -> int:
    """K and V of `tokens` tokens in fp16: B * H * D * 2 (K,V) * 2 bytes * L."""
    return batch * heads * head_dim * 2 * FP16 * tokens


def codebook_bytes(num_subspaces: int, num_codewords: int, dsub: int) -> int:
    """One fp16 codebook [M][K][Dsub]."""
    return num_subspaces * num_codewords * dsub * FP16


def code_bytes_per_vector(num_subspaces: int, num_codewords: int = 256) -> int:
    """8-bit index per subspace (K <= 256)."""
    assert num_codewords <= 256
    return num_subspaces


def compression_ratio(head_dim: int, num_subspaces: int) -> float:
    """fp16 vector bytes over code bytes, codebooks not counted."""
    return head_dim * FP16 / code_bytes_per_vector(num_subspaces)


def attention_flops(heads: int, head_dim: int, tokens: int) -> int:
    """Q·K^T (equally Score·V) for one decode token: H * (1 x D)(D x L) * 2."""
    return heads * head_dim * tokens * 2


def _lens(seq_lens) -> np.ndarray:
    return np.asarray(seq_lens, dtype=np.int64)


def pq_decode_bytes(seq_lens, num_q_heads: int, num_kv_heads: int, num_subspaces: int,
                    head_dim: int = 128, num_codewords: int = 256, page_size: int = 16) -> dict:
    """Bytes one PQ decode-attention call must move, by part.

    codes      every cached token's K and V codes: sum_b L_b * Hkv * 2 * M
    codebooks  each request's K and V codebooks for every kv head
    q, out     fp32 query in, fp32 output out
    tables     block-table entries in use, seq_lens and req_set
    """
    L = _lens(seq_lens)
    B = len(L)
    codes = int(L.sum()) * num_kv_heads * 2 * num_subspaces
    books = B * num_kv_heads * 2 * codebook_bytes(num_subspaces, num_codewords,
                                                  head_dim // num_subspaces)
    q = B * num_q_heads * head_dim * FP32
    out = q
    pages = int(((L + page_size - 1) // page_size).sum())
    tables = pages * INT32 + 2 * B * INT32
    total = codes + books + q + out + tables
    return {"codes": codes, "codebooks": books, "q": q, "out": out, "tables": tables,
            "code_stream": codes + books + pages * INT32, "total": total}


def pq_step_bytes_e4m3(seq_lens, num_q_heads: int, num_kv_heads: int, num_subspaces: int,
                       head_dim: int = 128, num_codewords: int = 256, page_size: int = 16) -> dict:
    """Bytes of one fused decode step whose codebooks are stored as FP8 E4M3
    (one byte per element instead of two)."""
    d = pq_step_bytes(seq_lens, num_q_heads, num_kv_heads, num_subspaces, head_dim, num_codewords,
                      page_size)
    half = d["codebooks"] // 2
    return dict(d, codebooks=d["codebooks"] - half, code_stream=d["code_stream"] - half,
                total=d["total"] - half)


def fp16_decode_bytes(seq_lens, num_q_heads: int, num_kv_heads: int,
                      head_dim: int = 128, page_size: int = 16) -> dict:
    """Bytes one fp16 decode-attention call must move (the uncompressed cache)."""
    L = _lens(seq_lens)
    B = len(L)
    cache = int(L.sum()) * num_kv_heads * 2 * head_dim * FP16
    q = B * num_q_heads * head_dim * FP32
    pages = int(((L + page_size - 1) // page_size).sum())
    tables = pages * INT32 + B * INT32
    return {"cache": cache, "q": q, "out": q, "tables": tables,
            "total": cache + 2 * q + tables}


def kv_tokens_heads(seq_lens, num_kv_heads: int) -> int:
    """The throughput unit: cached tokens times kv heads attended per call."""
    return int(_lens(seq_lens).sum()) * num_kv_heads


def pq_step_bytes(seq_lens, num_q_heads: int, num_kv_heads: int, num_subspaces: int,
                  head_dim: int = 128, num_codewords: int = 256, page_size: int = 16) -> dict:
    """Bytes of one fused decode step: the decode call's bytes plus the new
    tokens' fp16 K/V read and their codes written."""
    d = pq_decode_bytes(seq_lens, num_q_heads, num_kv_heads, num_subspaces, head_dim,
                        num_codewords, page_size)
    B = len(_lens(seq_lens))
    kv_new = B * num_kv_heads * 2 * head_dim * FP16
    new_codes = B * num_kv_heads * 2 * num_subspaces
    d = dict(d, kv_new=kv_new, new_codes=new_codes)
    d["total"] += kv_new + new_codes
    return d
