"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle itself.

Each test names the passage or the closed form it rests on.  They are chosen so
that a dropped term, a wrong sign or index, or a transposed operand anywhere in
the oracle fails at least one of them.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

import workloads as W

D = 128


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# fp16 narrowing used by kmeans_fit (round to nearest, ties to even)
# --------------------------------------------------------------------------
def _fp16_rne_exact(x: float) -> float:
    """Round a double to binary16 by exact rational arithmetic (IEEE 754 RNE)."""
    if x == 0.0:
        return x
    fx = Fraction(x)
    sign = -1 if fx < 0 else 1
    a = abs(fx)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -14)                       # subnormal spacing below 2^-14
    ulp = Fraction(2) ** (e - 10)
    n = a / ulp
    fl = math.floor(n)
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * ulp
    if r >= 65520:                        # beyond max finite after rounding
        return sign * math.inf
    return sign * float(r)


def test_fp16_narrowing_is_round_to_nearest_even():
    rng = _rng(1)
    vals = list(rng.standard_normal(2000) * 3.0)
    vals += list(rng.standard_normal(500) * 1e-5)          # subnormal range
    # exact ties between neighbouring halves: 1 + (2k+1) * 2^-11
    vals += [1.0 + (2 * k + 1) * 2.0 ** -11 for k in range(20)]
    vals += [-(2.0 + (2 * k + 1) * 2.0 ** -10) for k in range(20)]
    vals += [65504.0, 65519.0, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8]
    got = np.array(vals, np.float64).astype(np.float16).astype(np.float64)
    want = np.array([_fp16_rne_exact(v) for v in vals])
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------
# Byte arithmetic printed on the pages
# --------------------------------------------------------------------------
def _golden():
    out = {}
    import os
    p = os.path.join(os.path.dirname(__file__), "golden", "page_numbers.txt")
    for line in open(p, encoding="utf-8"):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, val = line.split("|")[0].split()
        out[key] = float(val)
    return out


def test_byte_arithmetic_matches_pages():
    from decode_attention_product_gb300 import traffic as T
    g = _golden()
    assert T.fp16_cache_bytes(4, 32, 128, 1) == g["kv_step_bytes_B4_H32_D128"]
    assert T.fp16_cache_bytes(4, 32, 128, 2048) == g["kv_layer_bytes_B4_H32_D128_L2048"]
    assert round(32 * T.fp16_cache_bytes(4, 32, 128, 2048) / 1e9, 1) == g["kv_32layers_GB_rounded"]
    assert T.codebook_bytes(4, 256, 32) == g["codebook_bytes_M4_K256_Dsub32"]
    assert 128 * T.FP16 == g["vector_bytes_fp16_D128"]
    assert T.code_bytes_per_vector(4) == g["code_bytes_M4_K256"]
    assert T.compression_ratio(128, 4) == g["compression_ratio_M4"]
    assert T.attention_flops(64, 128, 1000) == g["qk_flops_H64_D128_L1000"]
    assert T.attention_flops(64, 128, 1000) == g["sv_flops_H64_D128_L1000"]
    assert round(T.attention_flops(64, 128, 1000) / 1e6, 1) == g["qk_flops_rounded_M"]


def test_pq_call_bytes_page1_shape():
    """B4 H32 L2048 M4: codes 2*4*32*2048*4 B, codebooks 4*32*2*64 KiB."""
    from decode_attention_product_gb300 import traffic as T
    e = T.pq_step_bytes_e4m3([2048] * 4, 32, 32, 4)
    f = T.pq_step_bytes([2048] * 4, 32, 32, 4)
    assert e["codebooks"] == 4 * 32 * 2 * 4 * 256 * 32          # one byte per E4M3 entry
    assert f["total"] - e["total"] == e["codebooks"]
    b = T.pq_decode_bytes([2048] * 4, 32, 32, 4)
    assert b["codes"] == 2 * 4 * 32 * 2048 * 4 == 2_097_152
    assert b["codebooks"] == 4 * 32 * 2 * 65536 == 16_777_216
    assert b["q"] == b["out"] == 4 * 32 * 128 * 4
    # the fp16 comparison cache is the page's per-layer figure
    assert T.fp16_decode_bytes([2048] * 4, 32, 32)["cache"] == 134_217_728


# --------------------------------------------------------------------------
# Encode: brute force on tiny inputs in exact arithmetic
# --------------------------------------------------------------------------
def _brute_nearest(x, cb):
    """argmin_k sum_j (x_j - c_kj)^2 in exact rationals, lowest index on ties."""
    best, bd = None, None
    for k, c in enumerate(cb):
        d = sum((Fraction(float(a)) - Fraction(float(b))) ** 2 for a, b in zip(x, c))
        if bd is None or d < bd:
            best, bd = k, d
    return best


@pytest.mark.parametrize("K,Dsub,M", [(2, 1, 1), (3, 2, 2), (5, 3, 2), (8, 4, 2), (8, 2, 3)])
def test_encode_matches_exact_brute_force(orc, K, Dsub, M):
    rng = _rng(K * 100 + Dsub)
    Dm = Dsub * M
    # small-integer grids make exact ties frequent
    cb = rng.integers(-3, 4, size=(M, K, Dsub)).astype(np.float16)
    cb[:, -1] = cb[:, 0]                      # a duplicate codeword: ties
    x = rng.integers(-4, 5, size=(60, Dm)).astype(np.float16) / np.float16(2)
    codes = orc.pq_encode(x, cb)
    for i in range(x.shape[0]):
        for m in range(M):
            want = _brute_nearest(x[i, m * Dsub:(m + 1) * Dsub], cb[m])
            assert codes[i, m] == want, (i, m)


def test_encode_exhaustive_ties_two_codewords(orc):
    """Points on the bisector of two codewords are ties: lowest index wins; off
    it, the nearer one."""
    cb = np.array([[[0.0, 0.0], [2.0, 0.0]]], np.float16)        # M=1, K=2
    xs = np.array([[1.0, y] for y in (-2, -1, 0, 1, 2)] +
                  [[0.75, 0.0], [1.25, 0.0]], np.float16)
    codes = orc.pq_encode(xs, cb)[:, 0]
    assert list(codes) == [0, 0, 0, 0, 0, 0, 1]


def test_encode_codewords_are_their_own_codes(orc):
    """AQPIM blog §3.1: a vector equal to a codeword concatenation encodes to
    exactly those indices (distance 0, codewords distinct)."""
    rng = _rng(7)
    M, K, Dsub = 4, 256, 32
    cb = rng.standard_normal((M, K, Dsub)).astype(np.float16)
    want = rng.integers(0, K, size=(300, M))
    x = np.concatenate([cb[m, want[:, m]] for m in range(M)], axis=1)
    codes, gap = orc.pq_encode(x, cb, with_gap=True)
    assert np.array_equal(codes, want)
    assert np.all(gap == 1.0)                 # d1 = 0 -> gap (d2-0)/d2 = 1


def test_tiny_workload_noise_below_half_gap_keeps_generating_index(orc):
    """Tiny recipe: x = codeword + noise.  If the noise norm is below half the
    distance from that codeword to every other one, the triangle inequality
    makes it the unique nearest, so encode must return it."""
    w = W.make("tiny")
    kv = w.kv(0)                                   # [L][H][2][D] fp16
    gen = w.generating_codes(0)                    # [L][H][2][M]
    cbs = w.given_codebooks().astype(np.float64)   # [H][2][M][K][Dsub]
    M, Dsub = w.num_subspaces, w.dsub
    checked = 0
    for h in range(w.num_kv_heads):
        for kvw in range(2):
            x = kv[:, h, kvw].astype(np.float64)
            codes = orc.pq_encode(x, cbs[h, kvw])
            for m in range(M):
                C = cbs[h, kvw, m]
                pick = gen[:, h, kvw, m]
                e = np.linalg.norm(x[:, m * Dsub:(m + 1) * Dsub] - C[pick], axis=1)
                dist = np.linalg.norm(C[:, None] - C[None], axis=2)
                np.fill_diagonal(dist, np.inf)
                safe = e < dist[pick].min(axis=1) / 2
                assert np.array_equal(codes[safe, m], pick[safe])
                checked += int(safe.sum())
    assert checked > 0.9 * w.seq_lens[0] * w.num_kv_heads * 2 * M


def test_encode_append_writes_page_slots(orc):
    """Code of token t lands in page slot_mapping[t] // P, slot % P, K codes
    before V codes (PAM article §2.2.2 paged cache)."""
    rng = _rng(3)
    T, H, M, K, P = 5, 2, 4, 256, 16
    S = 2
    cbs = rng.standard_normal((S, H, 2, M, K, D // M)).astype(np.float16)
    want = rng.integers(0, K, size=(T, H, 2, M))
    tset = np.array([0, 1, 1, 0, 1], np.int32)
    kv = np.zeros((T, H, 2, D), np.float16)
    for t in range(T):
        for h in range(H):
            for w_ in range(2):
                kv[t, h, w_] = np.concatenate(
                    [cbs[tset[t], h, w_, m, want[t, h, w_, m]] for m in range(M)])
    slots = np.array([3 * P + 0, 0 * P + 15, 2 * P + 7, 3 * P + 1, 1 * P + 9], np.int64)
    pages = np.full((4, H, P, 2, M), 0xEE, np.uint8)
    orc.encode_append(kv, tset, slots, cbs, pages, P)
    for t in range(T):
        pg, sl = slots[t] // P, slots[t] % P
        for h in range(H):
            assert list(pages[pg, h, sl, 0]) == list(want[t, h, 0])
            assert list(pages[pg, h, sl, 1]) == list(want[t, h, 1])
    untouched = np.ones(pages.shape[:3], bool)
    for t in range(T):
        untouched[slots[t] // P, :, slots[t] % P] = False
    assert np.all(pages[untouched] == 0xEE)


def test_encode_append_skips_padding_tokens(orc):
    """A negative slot marks a padding token: nothing of it is stored (the
    boundary's convention), and the other tokens land as usual."""
    rng = _rng(4)
    T, H, M, K, P = 4, 1, 4, 256, 16
    cbs = rng.standard_normal((1, H, 2, M, K, D // M)).astype(np.float16)
    kv = rng.standard_normal((T, H, 2, D)).astype(np.float16)
    slots = np.array([-1, 5, -7, 17], np.int64)
    pages = np.full((2, H, P, 2, M), 0xEE, np.uint8)
    orc.encode_append(kv, np.zeros(T, np.int32), slots, cbs, pages, P)
    written = np.zeros(pages.shape[:3], bool)
    written[0, :, 5] = written[1, :, 1] = True
    assert np.all(pages[~written] == 0xEE)
    for t, (pg, sl) in ((1, (0, 5)), (3, (1, 1))):
        for w_ in range(2):
            want = orc.pq_encode(kv[t, 0, w_][None], cbs[0, 0, w_])[0]
            assert list(pages[pg, 0, sl, w_]) == list(want)


# --------------------------------------------------------------------------
# Attention: closed forms and invariants
# --------------------------------------------------------------------------
def test_two_token_closed_form(orc):
    """out = sigma(s1 - s2) v1 + sigma(s2 - s1) v2 for two keys."""
    rng = _rng(11)
    q = rng.standard_normal(D)
    k = rng.standard_normal((2, D))
    v = rng.standard_normal((2, D))
    scale = 0.3
    s1, s2 = scale * q @ k[0], scale * q @ k[1]
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))
    want = w1 * v[0] + (1.0 - w1) * v[1]
    assert np.allclose(orc.attention_dense(q, k, v, scale), want, rtol=1e-13, atol=1e-14)


def test_attention_invariants(orc):
    rng = _rng(12)
    L = 37
    k = rng.standard_normal((L, D))
    v = rng.standard_normal((L, D))
    # q = 0: uniform weights -> mean of V
    assert np.allclose(orc.attention_dense(np.zeros(D), k, v, 0.5), v.mean(0), atol=1e-14)
    # one token -> its value
    assert np.allclose(orc.attention_dense(rng.standard_normal(D), k[:1], v[:1], 0.5), v[0],
                       atol=1e-15)
    # empty -> zero vector (convention)
    assert np.all(orc.attention_dense(np.ones(D), k[:0], v[:0], 0.5) == 0.0)
    # shift invariance of softmax: adding a constant to every score
    q = rng.standard_normal(D)
    kk = k + np.outer(np.ones(L), q) * 0.0
    a = orc.attention_dense(q, kk, v, 0.2)
    e = np.zeros(D); e[0] = 1.0
    b = orc.attention_dense(np.concatenate([q, [1.0]]),
                            np.concatenate([k, np.full((L, 1), 3.0)], 1),
                            np.concatenate([v, np.zeros((L, 1))], 1), 0.2)[:D]
    assert np.allclose(a, b, rtol=1e-12, atol=1e-13)
    # permutation invariance over tokens
    p = rng.permutation(L)
    assert np.allclose(orc.attention_dense(q, k[p], v[p], 0.2), a, rtol=1e-12, atol=1e-13)
    # a dominant score selects its value (saturation)
    q2 = np.zeros(D); q2[5] = 1.0
    k2 = np.zeros((L, D)); k2[17, 5] = 400.0
    assert np.allclose(orc.attention_dense(q2, k2, v, 1.0), v[17], atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_split_merge_equals_single_pass(orc, seed):
    """PAM article §2.2.3: merging blockwise (max, sum) partials equals the
    single-pass softmax, for any partition including empty and 1-token blocks."""
    rng = _rng(100 + seed)
    L = int(rng.integers(1, 300))
    q = rng.standard_normal(D) * 2.0
    k = rng.standard_normal((L, D))
    v = rng.standard_normal((L, D))
    n = int(rng.integers(1, 9))
    cuts = np.sort(rng.integers(0, L + 1, size=n - 1))
    bounds = np.concatenate([[0], cuts, [L]])
    if seed % 2 == 0:                      # force an empty and a 1-token block
        bounds = np.concatenate([[0, 0, 1], np.maximum(bounds[1:], 1)])
    a = orc.attention_dense(q, k, v, 0.125)
    b = orc.attention_split_merge(q, k, v, 0.125, bounds)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def _paged_problem(seed, B=3, Hq=4, Hkv=2, M=4, K=256, lens=(40, 1, 77), S=None, P=16):
    rng = _rng(seed)
    S = S or B
    cbs = rng.standard_normal((S, Hkv, 2, M, K, D // M)).astype(np.float16)
    lens = np.array(lens, np.int32)
    maxp = int(-(-lens.max() // P))
    npages = int(sum(-(-l // P) for l in lens)) + 3
    perm = rng.permutation(npages)
    bt = np.zeros((B, maxp), np.int32)
    nxt = 0
    for b in range(B):
        n = -(-int(lens[b]) // P)
        bt[b, :n] = perm[nxt:nxt + n]
        nxt += n
    pages = rng.integers(0, K, size=(npages, Hkv, P, 2, M)).astype(np.uint8)
    req_set = rng.permutation(S)[:B].astype(np.int32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    return q, pages, cbs, req_set, bt, lens


def _decode_np(cbs, pages, req_set, bt, lens, b, kvh, P=16):
    """Reconstructed K and V of request b, kv head kvh (numpy indexing)."""
    L = int(lens[b])
    t = np.arange(L)
    c = pages[bt[b, t // P], kvh, t % P].astype(np.int64)    # [L][2][M]
    cb = cbs[req_set[b], kvh].astype(np.float64)            # [2][M][K][Dsub]
    M = cb.shape[1]
    Kx = np.concatenate([cb[0, m][c[:, 0, m]] for m in range(M)], axis=1)
    Vx = np.concatenate([cb[1, m][c[:, 1, m]] for m in range(M)], axis=1)
    return Kx, Vx


def test_pq_attention_equals_fp16_attention_on_codeword_cache(orc):
    """When every cached vector is a codeword concatenation, PQ attention over
    the codes equals fp16 attention over the vectors (AQPIM blog §3.1: the
    reconstruction is exact)."""
    q, pages, cbs, req_set, bt, lens = _paged_problem(21)
    B, Hq = q.shape[:2]
    Hkv = cbs.shape[1]
    P = 16
    npages = pages.shape[0]
    kvp = np.zeros((npages, Hkv, 2, P, D), np.float16)
    for b in range(B):
        for h in range(Hkv):
            Kx, Vx = _decode_np(cbs, pages, req_set, bt, lens, b, h)
            for t in range(int(lens[b])):
                kvp[bt[b, t // P], h, 0, t % P] = Kx[t]
                kvp[bt[b, t // P], h, 1, t % P] = Vx[t]
    a = orc.decode_attention(q, pages, cbs, req_set, bt, lens, 0.088, P)
    f = orc.decode_attention_fp16(q, kvp, bt, lens, 0.088)
    assert np.allclose(a, f, rtol=1e-14, atol=1e-15)


def test_pq_attention_factorised_form(orc):
    """The pages' fused flow, written independently: per-subspace lookup table
    LUT_m[k] = <q_m, C^K_m[k]> summed over m gives the score (AQPIM blog §4.1
    steps 2-3, §5.1 item 3); softmax weights binned by V code and multiplied by
    the V codebook give the output.  Must equal the decompress-then-compute
    oracle."""
    q, pages, cbs, req_set, bt, lens = _paged_problem(22, Hq=8, Hkv=2, M=8)
    B, Hq = q.shape[:2]
    Hkv, M = cbs.shape[1], cbs.shape[3]
    G, Dsub, P, scale = Hq // Hkv, D // M, 16, 0.07
    got = orc.decode_attention(q, pages, cbs, req_set, bt, lens, scale, P)
    for b in range(B):
        L = int(lens[b])
        t = np.arange(L)
        for h in range(Hq):
            kvh = h // G
            cb = cbs[req_set[b], kvh].astype(np.float64)
            c = pages[bt[b, t // P], kvh, t % P].astype(np.int64)
            qm = q[b, h].astype(np.float64).reshape(M, Dsub)
            lut = np.einsum("md,mkd->mk", qm, cb[0])                   # [M][K]
            s = scale * sum(lut[m][c[:, 0, m]] for m in range(M))
            p = np.exp(s - s.max())
            p /= p.sum()
            o = np.zeros((M, Dsub))
            for m in range(M):
                wbin = np.bincount(c[:, 1, m], weights=p, minlength=cb.shape[2])
                o[m] = wbin @ cb[1, m]
            assert np.allclose(got[b, h], o.reshape(D), rtol=1e-11, atol=1e-12), (b, h)


def test_gqa_head_mapping(orc):
    """Query head h reads kv head h // (Hq/Hkv) (Near-memory computing ch.1
    §1.4.3: 8 kv heads each serving 8 consecutive query heads)."""
    B, Hq, Hkv, M, K, P = 1, 4, 2, 4, 256, 16
    cbs = np.zeros((1, Hkv, 2, M, K, D // M), np.float16)
    cbs[0, 0, 1, 0, 0, 0] = 1.0       # kv head 0: V = e_0
    cbs[0, 1, 1, 0, 0, 1] = 1.0       # kv head 1: V = e_1
    pages = np.zeros((1, Hkv, P, 2, M), np.uint8)
    q = _rng(5).standard_normal((B, Hq, D)).astype(np.float32)
    out = orc.decode_attention(q, pages, cbs, np.zeros(1, np.int32), np.zeros((1, 1), np.int32),
                               np.array([9], np.int32), 0.1, P)
    e0 = np.eye(D)[0]; e1 = np.eye(D)[1]
    assert np.allclose(out[0, 0], e0) and np.allclose(out[0, 1], e0)
    assert np.allclose(out[0, 2], e1) and np.allclose(out[0, 3], e1)


def _codeword_fp16_pages(cbs, pages, req_set, bt, lens):
    """fp16 pages [NP][Hkv][2][P][D] holding, at every cached token's slot, the
    vectors its codes reconstruct to (written by numpy from the codebooks)."""
    B, Hkv, P = len(lens), cbs.shape[1], 16
    kvp = np.zeros((pages.shape[0], Hkv, 2, P, D), np.float16)
    for b in range(B):
        for h in range(Hkv):
            Kx, Vx = _decode_np(cbs, pages, req_set, bt, lens, b, h)
            for t in range(int(lens[b])):
                kvp[bt[b, t // P], h, 0, t % P] = Kx[t]
                kvp[bt[b, t // P], h, 1, t % P] = Vx[t]
    return kvp


def test_mixed_precision_limits(orc):
    """No fp16 head: the mixed step is PQ attention on every head; every head
    fp16: fp16 attention on every head (AQPIM blog §6.1 item 4 at its two
    ends), with a GQA group of 4 so that the query-head slicing is exercised."""
    q, pages, cbs, req_set, bt, lens = _paged_problem(41, Hq=8, Hkv=2, M=4)
    kvp = _rng(41).standard_normal((pages.shape[0], 2, 2, 16, D)).astype(np.float16)
    pq = orc.decode_attention(q, pages, cbs, req_set, bt, lens, 0.09, 16)
    f16 = orc.decode_attention_fp16(q, kvp, bt, lens, 0.09)
    got0 = orc.decode_attention_mixed(q, None, pages, cbs, req_set, bt, lens, 0.09, 16, 0)
    got2 = orc.decode_attention_mixed(q, kvp, None, None, req_set, bt, lens, 0.09, 16, 2)
    assert np.array_equal(got0, pq) and np.array_equal(got2, f16)


def test_mixed_precision_on_codeword_cache_is_fp16_attention(orc):
    """When every cached vector is a codeword concatenation, fp16 and PQ
    attention agree head by head, so any split of the kv heads into an fp16
    prefix and a PQ rest gives fp16 attention on all heads -- which fails if
    the query heads were sliced by kv head instead of group, the pools taken
    from the wrong end, or the two parts swapped."""
    q, pages, cbs, req_set, bt, lens = _paged_problem(42, Hq=12, Hkv=3, M=4)
    kvp = _codeword_fp16_pages(cbs, pages, req_set, bt, lens)
    want = orc.decode_attention_fp16(q, kvp, bt, lens, 0.08)
    for n16 in range(4):
        got = orc.decode_attention_mixed(q, np.ascontiguousarray(kvp[:, :n16]),
                                         np.ascontiguousarray(pages[:, n16:]),
                                         np.ascontiguousarray(cbs[:, n16:]), req_set, bt, lens, 0.08, 16, n16)
        assert np.allclose(got, want, rtol=1e-13, atol=1e-14), n16


def test_mixed_precision_head_mapping(orc):
    """kv head 0 fp16 with every value e_0, kv head 1 PQ with every value
    codeword e_1: query heads 0..G-1 return e_0, heads G..2G-1 return e_1."""
    G, P, M, K = 3, 16, 4, 256
    kvp = np.zeros((1, 1, 2, P, D), np.float16)
    kvp[0, 0, 1, :, 0] = 1.0
    cbs = np.zeros((1, 1, 2, M, K, D // M), np.float16)
    cbs[0, 0, 1, 0, 0, 1] = 1.0
    pages = np.zeros((1, 1, P, 2, M), np.uint8)
    q = _rng(6).standard_normal((1, 2 * G, D)).astype(np.float32)
    out = orc.decode_attention_mixed(q, kvp, pages, cbs, np.zeros(1, np.int32), np.zeros((1, 1), np.int32),
                                     np.array([11], np.int32), 0.1, P, 1)
    e0, e1 = np.eye(D)[0], np.eye(D)[1]
    for h in range(G):
        assert np.allclose(out[0, h], e0) and np.allclose(out[0, G + h], e1)


def test_block_table_page_and_slot(orc):
    """A saturating score on token t* returns the value stored at page
    block_table[b][t*/P], slot t* % P (PAM article §2.2.2 block table)."""
    P, M, K = 16, 4, 256
    L = 70
    Hkv = 1
    rng = _rng(9)
    npages = 8
    bt = np.array([[6, 2, 7, 0, 5]], np.int32)
    cbs = np.zeros((1, Hkv, 2, M, K, D // M), np.float16)
    cbs[0, 0, 0, 0, 1, 0] = 50.0                 # K code 1 in subspace 0 -> big score
    vals = rng.standard_normal((K, D // M)).astype(np.float16)
    cbs[0, 0, 1, :, :, :] = vals[None]           # V codebooks: same table each subspace
    pages = np.zeros((npages, Hkv, P, 2, M), np.uint8)
    pages[..., 1, :] = rng.integers(0, K, size=(npages, Hkv, P, M))
    for tstar in (0, 15, 16, 37, 69):
        pg = pages.copy()
        pg[bt[0, tstar // P], 0, tstar % P, 0, 0] = 1
        q = np.zeros((1, 1, D), np.float32); q[0, 0, 0] = 10.0
        out = orc.decode_attention(q, pg, cbs, np.zeros(1, np.int32), bt,
                                   np.array([L], np.int32), 1.0, P)[0, 0]
        vc = pg[bt[0, tstar // P], 0, tstar % P, 1]
        want = np.concatenate([vals[vc[m]].astype(np.float64) for m in range(M)])
        assert np.allclose(out, want, atol=1e-12), tstar


def test_decode_attention_special_lengths(orc):
    q, pages, cbs, req_set, bt, lens = _paged_problem(31, lens=(1, 0, 16))
    out = orc.decode_attention(q, pages, cbs, req_set, bt, lens, 0.1, 16)
    Kx, Vx = _decode_np(cbs, pages, req_set, bt, lens, 0, 0)
    assert np.allclose(out[0, 0], Vx[0], atol=1e-15)        # L=1 -> its value
    assert np.all(out[1] == 0.0)                            # L=0 -> zeros
    qz = np.zeros_like(q)
    out = orc.decode_attention(qz, pages, cbs, req_set, bt, lens, 0.1, 16)
    Kx, Vx = _decode_np(cbs, pages, req_set, bt, lens, 2, 1)
    assert np.allclose(out[2, 3], Vx.mean(0), atol=1e-14)   # q=0 -> mean of V


# --------------------------------------------------------------------------
# FP8 E4M3 codebook storage (AQPIM blog §4.2)
# --------------------------------------------------------------------------
def _e4m3_table():
    """Every finite E4M3 magnitude with its code (0..0x7E), from the format's
    definition: exponent field e (bias 7), fraction m/8, e = 0 subnormal."""
    vals, codes = [], []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue                                  # the NaN pattern
            vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
            codes.append((e << 3) | m)
    return np.array(vals), np.array(codes)


def test_e4m3_code_values(orc):
    got = orc.e4m3_to_float(np.array([0x38, 0x7E, 0x01, 0x08, 0x07, 0x3F, 0x40, 0x80, 0xFE, 0x7F, 0xFF],
                                     np.uint8))
    assert list(got[:7]) == [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, 7 * 2.0 ** -9, 1.875, 2.0]
    assert got[7] == 0.0 and np.signbit(got[7]) and got[8] == -448.0
    assert np.isnan(got[9]) and np.isnan(got[10])


def test_e4m3_rounding_by_hand(orc):
    x = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 447.9, 460.0, 470.0, 1e4, -1e4, np.inf,
                  -0.0, 0.09375], np.float32)
    want = [0x38,   # halfway 1 / 1.125: even fraction
            0x3A,   # halfway 1.125 / 1.25: even fraction (1.25)
            0x00,   # halfway 0 / 2^-9
            0x02,   # halfway 2^-9 / 2^-8
            0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E,   # 448 and saturation
            0x80,   # -0 keeps its sign
            0x1C]   # 0.09375 = 1.5 * 2^-4 exactly
    assert [int(v) for v in orc.e4m3_from_float(x)] == want
    assert orc.e4m3_from_float(np.array([np.nan], np.float32))[0] == 0x7F


def test_e4m3_every_code_round_trips(orc):
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    assert np.array_equal(orc.e4m3_from_float(orc.e4m3_to_float(codes)), codes)


def test_e4m3_rounding_exhaustive_over_fp16(orc):
    """Every finite fp16 value goes to the nearest E4M3 value (brute force over
    the format's table), ties to the even code, magnitudes beyond 448
    saturated; the sign is kept."""
    h = np.arange(65536, dtype=np.uint16).view(np.float16)
    h = h[np.isfinite(h)]
    x = h.astype(np.float64)
    vals, codes = _e4m3_table()
    a = np.abs(x)
    dist = np.abs(a[:, None] - vals[None, :])
    best = dist.min(1, keepdims=True)
    tied = dist == best
    # among the nearest, the even code (at most two candidates)
    pick = np.where(tied & (codes[None, :] % 2 == 0), 1, 0) + tied
    want = codes[pick.argmax(1)]
    want = np.where(a >= 448.0, 0x7E, want)
    want = want | np.where(np.signbit(x), 0x80, 0)
    got = orc.e4m3_from_float(h.astype(np.float32))
    assert np.array_equal(got.astype(np.int64), want.astype(np.int64))


# --------------------------------------------------------------------------
# k-means
# --------------------------------------------------------------------------
def test_kmeans_two_clumps_closed_form(orc):
    """1-D, K=2, two separated clumps with sample 0 in the left clump and
    sample 1 in the right: one Lloyd step lands on each clump's mean and stays."""
    left = [0.5, -0.25, 0.0, 0.125, 1.0]
    right = [10.0, 9.5, 11.25, 10.5]
    xs = [left[0], right[0]] + left[1:] + right[1:]
    samples = np.array(xs, np.float16).reshape(1, -1, 1).repeat(2, axis=2)  # D=2, M=2
    for iters in (1, 2, 5):
        cb16, cent, assign, _ = orc.kmeans_fit(samples, M=2, K=2, iters=iters)
        for m in range(2):
            assert cent[0, m, 0, 0] == float(sum(Fraction(v) for v in left) / len(left))
            assert cent[0, m, 1, 0] == float(sum(Fraction(v) for v in right) / len(right))
        lab = [0] * 1 + [1] + [0] * 4 + [1] * 3
        assert list(assign[0, :, 0]) == lab


def test_kmeans_square_vertices(orc):
    """Four symmetric clumps around the vertices of a square (2-D subspace):
    Lloyd from one seed per clump converges to the vertices exactly."""
    V = np.array([[0, 0], [4, 0], [0, 4], [4, 4]], np.float64)
    offs = np.array([[0.5, 0], [-0.5, 0], [0, 0.25], [0, -0.25]])
    pts = [V[i] for i in range(4)] + [V[i] + o for i in range(4) for o in offs]
    samples = np.array(pts, np.float16).reshape(1, -1, 2)
    samples = np.concatenate([samples, samples], axis=2)                 # D=4, M=2
    _, cent, _, _ = orc.kmeans_fit(samples, M=2, K=4, iters=4)
    for m in range(2):
        assert np.array_equal(cent[0, m], V)


def test_kmeans_fewer_samples_than_codewords_is_sample_codebook(orc):
    """N < K with centroid k initialised to sample k mod N: every sample owns
    its own centroid from the first step on, so the codebook is the samples
    repeated and every assignment is the sample's own index."""
    rng = _rng(41)
    U, N, M, K = 3, 64, 4, 256
    samples = rng.standard_normal((U, N, D)).astype(np.float16)
    cb16, cent, assign, mg = orc.kmeans_fit(samples, M=M, K=K, iters=10)
    for u in range(U):
        for m in range(M):
            sub = samples[u, :, m * 32:(m + 1) * 32]
            assert np.array_equal(cb16[u, m], sub[np.arange(K) % N])
            assert np.array_equal(assign[u, :, m], np.arange(N))
    assert np.all(mg > 0.0)


def test_kmeans_distortion_never_increases(orc):
    """Lloyd's objective sum_n min_k ||x_n - c_k||^2 is non-increasing."""
    rng = _rng(43)
    N, M, K = 400, 4, 16
    centres = rng.standard_normal((8, D)) * 2
    samples = (centres[rng.integers(0, 8, N)] + 0.5 * rng.standard_normal((N, D)))
    samples = samples.astype(np.float16)[None]
    prev = [math.inf] * M
    for it in range(1, 9):
        _, cent, _, _ = orc.kmeans_fit(samples, M=M, K=K, iters=it)
        for m in range(M):
            d = orc.kmeans_distortion(samples[0], cent[0, m], M, m)
            assert d <= prev[m] * (1 + 1e-6)
            prev[m] = d


def test_kmeans_step_continues_fit(orc):
    """One step from the fit's centroids after t iterations equals the fit after
    t+1 iterations (assignments exact, centroids to fp64 rounding)."""
    rng = _rng(44)
    U, N, M, K = 2, 300, 4, 32
    samples = rng.standard_normal((U, N, D)).astype(np.float16)
    _, c3, _, _ = orc.kmeans_fit(samples, M=M, K=K, iters=3)
    _, c4, a4, _ = orc.kmeans_fit(samples, M=M, K=K, iters=4)
    a, c, gap = orc.kmeans_step(samples, c3.astype(np.float32))
    assert np.array_equal(a, a4)
    assert np.allclose(c, c4, rtol=1e-15, atol=0)


def test_kmeans_refine_closed_forms(orc):
    """Refresh from a given codebook (AQPIM blog §6.1 item 3).  1-D, K = 4:
    rows at -1 and 12 pull the two clumps and land on their exact means; rows
    at 100 (twice) get no members and keep their value; from four identical
    rows every sample ties onto row 0, which becomes the mean of all."""
    left = [0.5, -0.25, 0.0, 0.125, 1.0]
    right = [10.0, 9.5, 11.25, 10.5]
    samples = np.array(left + right, np.float16).reshape(1, -1, 1).repeat(2, axis=2)   # D=2, M=2
    start = np.array([-1.0, 12.0, 100.0, 100.0], np.float16).reshape(1, 1, 4, 1).repeat(2, axis=1)
    for iters in (1, 3):
        cb16, cent, assign, _ = orc.kmeans_refine(samples, start, iters)
        for m in range(2):
            assert cent[0, m, 0, 0] == float(sum(Fraction(v) for v in left) / len(left))
            assert cent[0, m, 1, 0] == float(sum(Fraction(v) for v in right) / len(right))
            assert cent[0, m, 2, 0] == 100.0 and cent[0, m, 3, 0] == 100.0
            assert list(assign[0, :, m]) == [0] * 5 + [1] * 4
    same = np.full((1, 2, 4, 1), 5.0, np.float16)
    _, cent, assign, _ = orc.kmeans_refine(samples, same, 1)
    assert np.all(assign == 0)
    assert cent[0, 0, 0, 0] == float(sum(Fraction(v) for v in left + right) / 9)
    assert np.all(cent[0, :, 1:, 0] == 5.0)


def test_kmeans_refine_from_the_seeding_is_the_fit(orc):
    """Starting from the fit's own seeding (row k = sample k mod N, exact fp16),
    the refresh runs exactly the fit's steps."""
    rng = _rng(46)
    U, N, M, K = 2, 300, 4, 32
    samples = rng.standard_normal((U, N, D)).astype(np.float16)
    seed = np.stack([samples[:, np.arange(K) % N, m * (D // M):(m + 1) * (D // M)] for m in range(M)], axis=1)
    for iters in (1, 4):
        cf, cent_f, a_f, g_f = orc.kmeans_fit(samples, M=M, K=K, iters=iters)
        cr, cent_r, a_r, g_r = orc.kmeans_refine(samples, seed, iters)
        assert np.array_equal(cent_f, cent_r) and np.array_equal(a_f, a_r)
        assert np.array_equal(cf.view(np.uint16), cr.view(np.uint16))


def test_kmeans_refine_distortion_never_increases(orc):
    """Lloyd's objective on the recent samples never rises from the starting
    codebook on."""
    rng = _rng(47)
    N, M, K = 400, 4, 16
    centres = rng.standard_normal((8, D)) * 2
    samples = (centres[rng.integers(0, 8, N)] + 0.5 * rng.standard_normal((N, D))).astype(np.float16)[None]
    start = rng.standard_normal((1, M, K, D // M)).astype(np.float16)
    prev = [orc.kmeans_distortion(samples[0], start[0, m].astype(np.float64), M, m) for m in range(M)]
    for it in range(1, 7):
        _, cent, _, _ = orc.kmeans_refine(samples, start, it)
        for m in range(M):
            d = orc.kmeans_distortion(samples[0], cent[0, m], M, m)
            assert d <= prev[m] * (1 + 1e-6)
            prev[m] = d


def test_kmeans_update_is_member_mean(orc):
    """After a step, each non-empty centroid is the exact mean of the samples
    assigned to it and empty ones keep their input value."""
    rng = _rng(45)
    U, N, M, K = 1, 50, 2, 64
    samples = rng.standard_normal((U, N, 8)).astype(np.float16)
    cin = rng.standard_normal((U, M, K, 4)).astype(np.float32)
    a, c, _ = orc.kmeans_step(samples, cin)
    for m in range(M):
        sub = samples[0, :, m * 4:(m + 1) * 4].astype(np.float64)
        for k in range(K):
            mem = sub[a[0, :, m] == k]
            want = mem.mean(0) if len(mem) else cin[0, m, k].astype(np.float64)
            assert np.allclose(c[0, m, k], want, rtol=1e-15, atol=0)
        # and each assignment is the nearest centroid (brute force in float64)
        d = ((sub[:, None, :] - cin[0, m][None].astype(np.float64)) ** 2).sum(-1)
        assert np.array_equal(a[0, :, m], d.argmin(1))
