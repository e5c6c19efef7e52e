"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: codes and k-means assignments bit-exact wherever the oracle's relative
runner-up gap exceeds 1e-4 (and, since both sides decide with the same fp32
arithmetic, everywhere in practice -- asserted separately); codebooks bit-exact;
attention outputs within |o - o*| <= 2e-3 + 2e-3 |o*|.
"""
import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-3
GAP = 1e-4


@pytest.fixture(params=["auto", "1", "2"])
def kernel(request, monkeypatch):
    """Which PQ decode kernel the planner may use: its own choice, the
    token-share kernel, or the whole-split kernel (where a split fits)."""
    if request.param == "auto":
        monkeypatch.delenv("AQPQ_DECODE_KERNEL", raising=False)
    else:
        monkeypatch.setenv("AQPQ_DECODE_KERNEL", request.param)
    return request.param


@pytest.fixture
def kernel1(monkeypatch):
    monkeypatch.setenv("AQPQ_DECODE_KERNEL", "1")


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_product_gb300 import build
    build.build()
    from decode_attention_product_gb300 import api
    return api


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def close(got, want):
    got = np.asarray(got, np.float64)
    err = np.abs(got - want)
    bound = ATOL + RTOL * np.abs(want)
    assert np.all(np.isfinite(got)), "non-finite output"
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tol; max err {err.max():.3e}"
    return float(err.max())


def run_pq(A, p, num_splits=0, max_seq_len=None):
    st = A.new_status()
    L = int(max(p["seq_lens"].max(), 0)) if max_seq_len is None else max_seq_len
    out = A.decode_attention(dev(p["q"]), dev(p["code_pages"]), dev(p["codebooks"]),
                             dev(p["req_set"]), dev(p["block_table"]), dev(p["seq_lens"]),
                             L, 1.0 / np.sqrt(128), num_splits=num_splits, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(st.item())


def oracle_pq(orc, p):
    return orc.decode_attention(p["q"], p["code_pages"], p["codebooks"], p["req_set"],
                                p["block_table"], p["seq_lens"], 1.0 / np.sqrt(128), 16)


# --------------------------------------------------------------------------
# decode attention (random codes and codebooks; stage parity)
# --------------------------------------------------------------------------
CASES = [
    # (B, Hq, Hkv, M, lens)
    (1, 2, 2, 4, [512]),                       # the tiny shape
    (3, 4, 4, 4, [1, 17, 333]),                # ragged tails, 1-token request
    (2, 8, 2, 4, [700, 45]),                   # GQA group 4
    (2, 16, 2, 4, [1000, 257]),                # GQA group 8: several chunks per CTA
    (2, 4, 2, 4, [64, 31]),                    # group 2
    (2, 4, 4, 8, [400, 1500]),                 # M = 8 (Dsub 16)
    (1, 16, 2, 8, [3001]),                     # M = 8 with group 8
    (2, 8, 2, 8, [700, 45]),                   # M = 8 with group 4 (clusters of 8 cover the group twice)
    (1, 2, 2, 4, [9001]),                      # group 1, several chunks per CTA
    (4, 4, 4, 4, [0, 16, 15, 48]),             # empty request, page-exact lengths
    (8, 64, 8, 4, [300, 1, 77, 160, 999, 64, 5, 410]),   # Qwen-shaped GQA: 2 head sub-groups
    (1, 2, 2, 4, [30000]),                     # one split: a CTA streams several chunks
    (1, 4, 2, 8, [20000, ]),                   # the same with M = 8, group 2
    (1, 8, 2, 4, [12000]),                     # streamed with group 4: a fixed-point frame per head
    (1, 16, 2, 4, [8000]),                     # streamed with group 8
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}Hq{c[1]}Hkv{c[2]}M{c[3]}" for c in CASES])
@pytest.mark.parametrize("splits", [0, 1, 2, 7])
def test_decode_matches_oracle(A, orc, case, splits, kernel):
    B, Hq, Hkv, M, lens = case
    p = W.paged_codes_problem(hash((B, Hq, Hkv, M, tuple(lens))) % 10000, B, Hq, Hkv, M, lens,
                              num_sets=B + 1)
    got, st = run_pq(A, p, num_splits=splits)
    assert st == 0
    close(got, oracle_pq(orc, p))
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(got[b] == 0.0)


# many (request, kv head) units: the planner switches to clusters of 2 CTAs
MANY = [(48, 32, 32, 4), (48, 32, 32, 8)]


def _many_lens(n, seed):
    return [int(x) for x in np.random.default_rng(seed).integers(1, 300, size=n)]


@pytest.mark.parametrize("case", MANY, ids=[f"B{c[0]}H{c[1]}M{c[3]}" for c in MANY])
def test_decode_many_units_cluster2(A, orc, case, kernel1):
    B, Hq, Hkv, M = case
    lens = _many_lens(B, M)
    assert A.decode_plan(B, Hq, Hkv, max(lens), M)[1] == 2
    p = W.paged_codes_problem(31 + M, B, Hq, Hkv, M, lens, num_sets=B)
    got, st = run_pq(A, p)
    assert st == 0
    close(got, oracle_pq(orc, p))


def test_decode_plan_variants_agree(A, orc, kernel):
    """Cluster sizes 4 and the split counts the planner picks for the long shape
    give the same answer as the oracle."""
    p = W.paged_codes_problem(5, 1, 4, 4, 8, [20000], num_sets=1)
    want = oracle_pq(orc, p)
    for s in (0, 3, 16):
        got, st = run_pq(A, p, num_splits=s)
        assert st == 0
        close(got, want)


def test_decode_repeated_calls_agree(A, kernel):
    """The value bins accumulate as unsigned fixed-point integers, so the order
    of the shared-memory atomics cannot change them, and every other reduction
    has a fixed order: repeated calls agree bit for bit."""
    p = W.paged_codes_problem(6, 2, 8, 8, 4, [900, 1200])
    a, _ = run_pq(A, p)
    b, _ = run_pq(A, p)
    assert np.array_equal(a, b)


def test_decode_data_errors_flag_and_nan(A, kernel):
    p = W.paged_codes_problem(7, 3, 4, 4, 4, [40, 40, 40], num_sets=3)
    # request 0: block-table entry outside the pool; request 1: set outside the array
    p["block_table"][0, 1] = p["num_pages"] + 5
    p["req_set"][1] = 99
    got, st = run_pq(A, p)
    assert st & 1 and st & 4
    assert np.all(np.isnan(got[0])) and np.all(np.isnan(got[1]))
    assert np.all(np.isfinite(got[2]))
    # a device length beyond the planned maximum
    p = W.paged_codes_problem(8, 2, 4, 4, 4, [40, 64], num_sets=2)
    got, st = run_pq(A, p, max_seq_len=48)
    assert st & 2
    assert np.all(np.isnan(got[1])) and np.all(np.isfinite(got[0]))


# --------------------------------------------------------------------------
# fp16 comparison kernel
# --------------------------------------------------------------------------
FP16_CASES = [(1, 2, 2, [512]), (3, 4, 4, [1, 17, 333]), (2, 16, 2, [1000, 37]),
              (2, 8, 2, [64, 0]), (1, 4, 4, [5000])]


@pytest.mark.parametrize("case", FP16_CASES)
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_fp16_decode_matches_oracle(A, orc, case, splits):
    B, Hq, Hkv, lens = case
    p = W.paged_fp16_problem(sum(lens) + B, B, Hq, Hkv, lens)
    st = A.new_status()
    out = A.decode_attention_fp16(dev(p["q"]), dev(p["kv_pages"]), dev(p["block_table"]),
                                  dev(p["seq_lens"]), int(max(lens)), 1.0 / np.sqrt(128),
                                  num_splits=splits, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = orc.decode_attention_fp16(p["q"], p["kv_pages"], p["block_table"], p["seq_lens"],
                                     1.0 / np.sqrt(128))
    close(out.cpu().numpy(), want)


# --------------------------------------------------------------------------
# encode
# --------------------------------------------------------------------------
def _encode_case(A, orc, w, t0, t1):
    """Encode tokens [t0, t1) of every request of workload w on both sides, with
    codebooks fitted (by the oracle) on each request's first 64 tokens."""
    B, Hkv, M = w.batch, w.num_kv_heads, w.num_subspaces
    if w.mixture:
        samples = np.stack([w.fit_samples(w.kv(b, t1=w.n_fit)) for b in range(B)])
        cb16, _, _, _ = orc.kmeans_fit(samples.reshape(-1, *samples.shape[3:]), M, 256, 3)
        cbs = cb16.reshape(B, Hkv, 2, M, 256, w.dsub)
    else:
        cbs = np.stack([w.given_codebooks()] * B)
    kvs = [w.kv(b, t0=t0, t1=t1) for b in range(B)]
    assert sum(len(k) for k in kvs) > 0
    bt, npages = w.block_table()
    kv = np.concatenate(kvs)
    tset = np.concatenate([np.full(len(k), b, np.int32) for b, k in enumerate(kvs)])
    slots = np.concatenate([w.slot_mapping(bt, b, t0, t0 + len(k)) for b, k in enumerate(kvs)])
    want = np.zeros((npages, Hkv, 16, 2, M), np.uint8)
    gap = orc.encode_append(kv, tset, slots, cbs, want, 16)
    pages = torch.zeros((npages, Hkv, 16, 2, M), dtype=torch.uint8, device="cuda")
    st = A.new_status()
    A.encode_append(dev(kv), dev(tset), dev(slots), dev(cbs), pages, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = pages.cpu().numpy()
    # compare every written slot: bit-exact where the gap clears the band ...
    pg, sl = slots // 16, slots % 16
    g_codes = got[pg, :, sl]                     # [T][Hkv][2][M]
    w_codes = want[pg, :, sl]
    clear = gap > GAP
    assert np.array_equal(g_codes[clear], w_codes[clear])
    # ... and, the decision arithmetic being the same, everywhere
    assert np.array_equal(g_codes, w_codes)
    return clear.mean()


def test_encode_tiny_workload(A, orc):
    assert _encode_case(A, orc, W.make("tiny"), 0, 512) > 0.99


def test_encode_small_batch_append(A, orc):
    # a decode step: one token per request (codeword-parallel kernel)
    _encode_case(A, orc, W.make("page1"), 2047, 2048)
    _encode_case(A, orc, W.make("long", seq_lens=[200]), 100, 101)


def test_encode_prefill_tiles(A, orc):
    # 767 and 829 tokens x 8 / 4 heads: still the codeword-parallel kernel; ragged requests
    w = W.make("ragged", seq_lens=[300, 70, 333, 64], num_q_heads=8, num_kv_heads=8)
    _encode_case(A, orc, w, 0, 10**9)
    w = W.make("long", seq_lens=[700, 129], num_q_heads=4, num_kv_heads=4)
    _encode_case(A, orc, w, 0, 10**9)


def test_encode_prefill_tensor_core_tiles(A, orc):
    # more than 8192 token-heads: 128-token tiles on the tensor cores; ragged
    # requests, tiles shared by two requests, a ragged tail
    w = W.make("ragged", seq_lens=[1000, 333, 65, 700, 129], num_q_heads=8, num_kv_heads=8)
    assert _encode_case(A, orc, w, 0, 10**9) > 0.99
    w = W.make("long", seq_lens=[1500, 700], num_q_heads=8, num_kv_heads=8)       # M = 8
    assert _encode_case(A, orc, w, 0, 10**9) > 0.99


def _encode_direct(A, orc, kv, tset, slots, cbs, npages):
    """Both sides encode the same arrays; every written slot must agree."""
    Hkv, M = kv.shape[1], cbs.shape[3]
    want = np.zeros((npages, Hkv, 16, 2, M), np.uint8)
    orc.encode_append(kv, tset, slots, cbs, want, 16)
    pages = torch.zeros((npages, Hkv, 16, 2, M), dtype=torch.uint8, device="cuda")
    st = A.new_status()
    A.encode_append(dev(kv), dev(tset), dev(slots), dev(cbs), pages, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = pages.cpu().numpy()
    assert np.array_equal(got, want)
    return got


@pytest.mark.parametrize("M", [4, 8])
def test_encode_tensor_core_near_ties(A, orc, M):
    """Codebooks that defeat any approximate filter: set 0 holds every row four
    times (as the k-means seeding leaves them), set 1 one row repeated with a
    one-ulp change in one element per row (all 256 codewords tie to within
    rounding: the full-scan fallback), set 2 random rows.  Tokens sit on or
    near codewords, the sets interleave token by token (several passes per
    tile), some tokens are padding and one has an infinite component."""
    g = np.random.default_rng(11 + M)
    T, Hkv, S, Dsub = 1100, 8, 3, 128 // M
    cbs = g.standard_normal((S, Hkv, 2, M, 256, Dsub)).astype(np.float16)
    cbs[0] = np.concatenate([cbs[0][..., :64, :]] * 4, axis=-2)
    one = np.repeat(cbs[1][..., :1, :], 256, axis=-2)
    bits = one.view(np.uint16)
    j = g.integers(0, Dsub, size=bits.shape[:-1])
    np.put_along_axis(bits, j[..., None],
                      np.take_along_axis(bits, j[..., None], -1) + g.integers(0, 2, j.shape)[..., None]
                      .astype(np.uint16), -1)
    cbs[1] = one
    tset = (np.arange(T) % S).astype(np.int32)
    pick = g.integers(0, 256, size=(T, Hkv, 2, M))
    hh = np.arange(Hkv)[None, :, None, None]
    ww = np.arange(2)[None, None, :, None]
    mm = np.arange(M)[None, None, None, :]
    words = cbs[tset[:, None, None, None], hh, ww, mm, pick].astype(np.float32)   # [T][Hkv][2][M][Dsub]
    noise = g.standard_normal(words.shape).astype(np.float32) * 0.02
    noise[::7] = 0.0                                       # exactly on a codeword
    kv = (words + noise).reshape(T, Hkv, 2, 128).astype(np.float16)
    kv[5, 3, 1, 7] = np.inf
    npages = (T + 15) // 16 + 3
    slots = g.permutation(npages * 16)[:T].astype(np.int64)
    slots[::97] = -1                                       # padding tokens
    _encode_direct(A, orc, kv, tset, slots, cbs, npages)


def test_encode_bad_slots_flagged(A):
    kv = torch.zeros((2, 1, 2, 128), dtype=torch.float16, device="cuda")
    cbs = torch.zeros((1, 1, 2, 4, 256, 32), dtype=torch.float16, device="cuda")
    pages = torch.full((2, 1, 16, 2, 4), 7, dtype=torch.uint8, device="cuda")
    st = A.new_status()
    A.encode_append(kv, dev(np.array([0, 5], np.int32)), dev(np.array([40, -1], np.int64)), cbs,
                    pages, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 1                   # page 2 outside a 2-page pool; -1 skipped
    assert torch.all(pages == 7)


# --------------------------------------------------------------------------
# codebook fit
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name,N,iters", [("page1", 64, 10), ("long", 64, 10), ("page1", 1024, 10), ("tiny", 300, 10),
                                          ("page1", 1024, 60), ("long", 512, 40)])
def test_fit_matches_oracle(A, orc, name, N, iters):
    """The GPU fit stops once an assignment repeats (a fixed point); the oracle
    runs every step: the codebooks and last assignments must still agree bit
    for bit."""
    w = W.make(name)
    units = []
    for b in range(min(w.batch, 2)):
        kv = w.kv(b, t1=N)
        units.append(np.ascontiguousarray(kv[:N].transpose(1, 2, 0, 3)).reshape(-1, N, 128))
    samples = np.concatenate(units)[:24]                            # [U][N][D]
    M = w.num_subspaces
    cb16, _, assign, mg = orc.kmeans_fit(samples, M, 256, iters)
    cb_gpu, asg_gpu = A.fit_codebooks(dev(samples), M, iters, with_assign=True)
    torch.cuda.synchronize()
    assert np.array_equal(asg_gpu.cpu().numpy(), assign)
    assert np.array_equal(cb_gpu.cpu().numpy().view(np.uint16), cb16.view(np.uint16))


def test_kmeans_step_matches_oracle(A, orc):
    w = W.make("page1")
    kv = w.kv(0, t1=1024)
    samples = np.ascontiguousarray(kv.transpose(1, 2, 0, 3)).reshape(-1, 1024, 128)[:8]
    _, cent, _, _ = orc.kmeans_fit(samples, 4, 256, 2)
    c32 = cent.astype(np.float32)
    a_o, c_o, gap = orc.kmeans_step(samples, c32)
    c_g, a_g = A.kmeans_step(dev(samples), dev(c32))
    torch.cuda.synchronize()
    assert np.array_equal(a_g.cpu().numpy(), a_o)
    assert np.array_equal(c_g.cpu().numpy(), c_o.astype(np.float32))


@pytest.mark.parametrize("name", ["page1", "long"])
def test_refine_matches_oracle(A, orc, name):
    """Periodic codebook refresh: codebooks fitted on tokens [0, 64) of each
    request, refined in place on tokens [64, 128) for 3 steps; codebooks and
    assignments bit-exact, then the 64 recent tokens re-encode identically."""
    w = W.make(name, seq_lens=[256, 256]) if name == "long" else W.make(name)
    M, Hkv = w.num_subspaces, w.num_kv_heads
    B = 2
    first = np.concatenate([np.ascontiguousarray(w.kv(b, t1=64).transpose(1, 2, 0, 3)).reshape(-1, 64, 128)
                            for b in range(B)])
    recent_kv = [w.kv(b, t0=64, t1=128) for b in range(B)]
    recent = np.concatenate([np.ascontiguousarray(k.transpose(1, 2, 0, 3)).reshape(-1, 64, 128)
                             for k in recent_kv])
    cb16, _, _, _ = orc.kmeans_fit(first, M, 256, 10)
    cb_ref, _, asg_ref, _ = orc.kmeans_refine(recent, cb16, 3)
    cb_gpu = dev(cb16)
    asg_gpu = A.refine_codebooks(dev(recent), cb_gpu, 3, with_assign=True)
    torch.cuda.synchronize()
    assert np.array_equal(asg_gpu.cpu().numpy(), asg_ref)
    assert np.array_equal(cb_gpu.cpu().numpy().view(np.uint16), cb_ref.view(np.uint16))
    assert not np.array_equal(cb_ref.view(np.uint16), cb16.view(np.uint16))   # it did move
    # re-encode the recent tokens with the refreshed codebooks
    cbs = cb_ref.reshape(B, Hkv, 2, M, 256, 128 // M)
    kv = np.concatenate(recent_kv)
    tset = np.repeat(np.arange(B, dtype=np.int32), 64)
    slots = np.arange(B * 64, dtype=np.int64)
    _encode_direct(A, orc, kv, tset, slots, cbs, (B * 64) // 16)


@pytest.mark.parametrize("n", [65536, 65536 - 3, 13])
def test_e4m3_conversion_matches_oracle(A, orc, n):
    """Every fp16 bit pattern to E4M3 and every code back to fp16, against the
    oracle's definition (NaN compared by class: its sign is unspecified)."""
    h = np.arange(65536, dtype=np.uint16)[:n].view(np.float16)
    got = A.to_e4m3(dev(h)).cpu().numpy()
    with np.errstate(invalid="ignore"):                  # NaN patterns cast to NaN
        want = orc.e4m3_from_float(h.astype(np.float32))
    nan = np.isnan(h)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7F) == 0x7F)
    codes = np.arange(256, dtype=np.uint8)
    back = A.from_e4m3(dev(codes)).cpu().numpy()
    ref = orc.e4m3_to_float(codes).astype(np.float16)
    fin = ~np.isnan(ref)
    assert np.array_equal(back[fin].view(np.uint16), ref[fin].view(np.uint16))
    assert np.all(np.isnan(back[~fin]))


# --------------------------------------------------------------------------
# fused decode step (append the token at position seq_len-1, then attend)
# --------------------------------------------------------------------------
STEP_CASES = [
    # (B, Hq, Hkv, M, lens)
    (3, 4, 4, 4, [1, 17, 333]),                # new token alone; page boundary at 16
    (2, 16, 2, 4, [1000, 257]),                # GQA group 8
    (2, 4, 4, 8, [400, 1500]),                 # M = 8
    (2, 8, 2, 8, [700, 45]),                   # M = 8, group 4
    (1, 2, 2, 4, [9001]),                      # long: splits
    (4, 4, 4, 4, [16, 32, 48, 2048]),          # new token first in its page
    (8, 64, 8, 4, [300, 1, 77, 160, 999, 64, 5, 410]),   # GQA with 2 head sub-groups per kv head
    (1, 4, 4, 8, [20000]),                     # M = 8, long: clusters of 8 over several splits
    (1, 2, 2, 4, [30001]),                     # with one split: several chunks per CTA, one pass
    (1, 8, 2, 4, [12001]),                     # the same with group 4 (per-head frames)
]


@pytest.mark.parametrize("case", STEP_CASES, ids=[f"B{c[0]}Hq{c[1]}Hkv{c[2]}M{c[3]}" for c in STEP_CASES])
@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("overlap", [False, True])
def test_decode_step_matches_oracle(A, orc, case, splits, overlap, kernel):
    B, Hq, Hkv, M, lens = case
    p = W.paged_codes_problem(hash((B, Hq, M, tuple(lens), 7)) % 10000, B, Hq, Hkv, M, lens,
                              num_sets=B + 1)
    rng = np.random.default_rng(len(lens) * 31 + M)
    kv_new = rng.standard_normal((B, Hkv, 2, 128)).astype(np.float16)
    # oracle: encode each new token into its slot, then attend
    want_pages = p["code_pages"].copy()
    slots = np.array([p["block_table"][b, (L - 1) // 16] * 16 + (L - 1) % 16
                      for b, L in enumerate(lens)], np.int64)
    orc.encode_append(kv_new, p["req_set"], slots, p["codebooks"], want_pages, 16)
    pw = dict(p, code_pages=want_pages)
    want = oracle_pq(orc, pw)
    # GPU
    pages = dev(p["code_pages"])
    st = A.new_status()
    out = A.decode_step(dev(p["q"]), dev(kv_new), pages, dev(p["codebooks"]), dev(p["req_set"]),
                        dev(p["block_table"]), dev(p["seq_lens"]), int(max(lens)),
                        1.0 / np.sqrt(128), num_splits=splits, overlap=overlap, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(pages.cpu().numpy(), want_pages)    # the new codes, nothing else
    close(out.cpu().numpy(), want)


@pytest.mark.parametrize("case", STEP_CASES + [(MANY[0][0], MANY[0][1], MANY[0][2], MANY[0][3], None)],
                         ids=[f"B{c[0]}Hq{c[1]}Hkv{c[2]}M{c[3]}" for c in STEP_CASES] + ["many_cluster2"])
@pytest.mark.parametrize("splits", [0, 3])
def test_decode_step_e4m3_codebooks(A, orc, case, splits):
    """FP8 E4M3 codebooks (AQPIM blog §4.2): the step on the codes equals the
    oracle's step on their exact values (new codes bit-exact, outputs within
    tolerance)."""
    B, Hq, Hkv, M, lens = case
    if lens is None:
        lens = _many_lens(B, M + 1)
    p = W.paged_codes_problem(hash((B, Hq, M, tuple(lens), 8)) % 10000, B, Hq, Hkv, M, lens, num_sets=B + 1)
    cb8 = orc.e4m3_from_float(p["codebooks"].astype(np.float32))
    cbw = orc.e4m3_to_float(cb8).astype(np.float16)
    assert not np.array_equal(cbw, p["codebooks"])                 # the rounding is visible
    kv_new = np.random.default_rng(len(lens) * 37 + M).standard_normal((B, Hkv, 2, 128)).astype(np.float16)
    want_pages = p["code_pages"].copy()
    slots = np.array([p["block_table"][b, (L - 1) // 16] * 16 + (L - 1) % 16 for b, L in enumerate(lens)],
                     np.int64)
    orc.encode_append(kv_new, p["req_set"], slots, cbw, want_pages, 16)
    want = oracle_pq(orc, dict(p, code_pages=want_pages, codebooks=cbw))
    pages = dev(p["code_pages"])
    st = A.new_status()
    out = A.decode_step(dev(p["q"]), dev(kv_new), pages, dev(cb8), dev(p["req_set"]), dev(p["block_table"]),
                        dev(p["seq_lens"]), int(max(lens)), 1.0 / np.sqrt(128), num_splits=splits, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(pages.cpu().numpy(), want_pages)
    close(out.cpu().numpy(), want)


@pytest.mark.parametrize("case", MANY, ids=[f"B{c[0]}H{c[1]}M{c[3]}" for c in MANY])
@pytest.mark.parametrize("overlap", [False, True])
def test_decode_step_many_units_cluster2(A, orc, case, overlap, kernel1):
    B, Hq, Hkv, M = case
    lens = _many_lens(B, M + 1)
    assert A.decode_plan(B, Hq, Hkv, max(lens), M)[1] == 2
    p = W.paged_codes_problem(41 + M, B, Hq, Hkv, M, lens, num_sets=B)
    kv_new = np.random.default_rng(M).standard_normal((B, Hkv, 2, 128)).astype(np.float16)
    want_pages = p["code_pages"].copy()
    slots = np.array([p["block_table"][b, (L - 1) // 16] * 16 + (L - 1) % 16 for b, L in enumerate(lens)],
                     np.int64)
    orc.encode_append(kv_new, p["req_set"], slots, p["codebooks"], want_pages, 16)
    want = oracle_pq(orc, dict(p, code_pages=want_pages))
    pages = dev(p["code_pages"])
    st = A.new_status()
    out = A.decode_step(dev(p["q"]), dev(kv_new), pages, dev(p["codebooks"]), dev(p["req_set"]),
                        dev(p["block_table"]), dev(p["seq_lens"]), int(max(lens)), 1.0 / np.sqrt(128),
                        overlap=overlap, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(pages.cpu().numpy(), want_pages)
    close(out.cpu().numpy(), want)


def test_decode_step_equals_append_then_decode(A, kernel):
    """The fused step gives the two-call sequence's codes and (to fp32
    rounding) its output."""
    p = W.paged_codes_problem(77, 4, 32, 32, 4, [2048] * 4)
    kv_new = np.random.default_rng(5).standard_normal((4, 32, 2, 128)).astype(np.float16)
    bt, lens = p["block_table"], p["seq_lens"]
    slots = np.array([bt[b, (L - 1) // 16] * 16 + (L - 1) % 16 for b, L in enumerate(lens)], np.int64)
    pa, pb = dev(p["code_pages"]), dev(p["code_pages"])
    A.encode_append(dev(kv_new), dev(p["req_set"]), dev(slots), dev(p["codebooks"]), pa)
    o1 = A.decode_attention(dev(p["q"]), pa, dev(p["codebooks"]), dev(p["req_set"]), dev(bt),
                            dev(lens), 2048)
    o2 = A.decode_step(dev(p["q"]), dev(kv_new), pb, dev(p["codebooks"]), dev(p["req_set"]), dev(bt),
                       dev(lens), 2048)
    torch.cuda.synchronize()
    assert torch.equal(pa, pb)
    assert torch.allclose(o1, o2, rtol=1e-5, atol=1e-6)


def test_decode_step_bad_new_page_flagged(A, kernel):
    """The new token's page id outside the pool: bad-page status, NaN output for
    that request, no code written anywhere for it, the other request intact."""
    p = W.paged_codes_problem(9, 2, 4, 4, 4, [40, 40], num_sets=2)
    p["block_table"][0, 39 // 16] = p["num_pages"] + 3
    kv_new = np.random.default_rng(9).standard_normal((2, 4, 2, 128)).astype(np.float16)
    before = p["code_pages"].copy()
    pages = dev(p["code_pages"])
    st = A.new_status()
    out = A.decode_step(dev(p["q"]), dev(kv_new), pages, dev(p["codebooks"]), dev(p["req_set"]),
                        dev(p["block_table"]), dev(p["seq_lens"]), 40, 1.0 / np.sqrt(128), status=st)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert int(st.item()) & 1
    assert np.all(np.isnan(got[0])) and np.all(np.isfinite(got[1]))
    after = pages.cpu().numpy()
    for j in range(3):
        pg = p["block_table"][0, j]
        if 0 <= pg < p["num_pages"]:
            assert np.array_equal(after[pg], before[pg])


def test_decode_step_graphs_with_pinned_buffers(A, orc):
    """api.DecodeStep: two captured graphs (copy in, fused step, copy out) with
    their own pinned buffers and inputs, the second launched before the first
    is waited for; each host output matches the oracle's step on its inputs."""
    B, Hq, Hkv, M, lens = 2, 8, 8, 4, [700, 1300]
    p = W.paged_codes_problem(55, B, Hq, Hkv, M, lens, num_sets=B)
    rng = np.random.default_rng(55)
    slots = np.array([p["block_table"][b, (L - 1) // 16] * 16 + (L - 1) % 16 for b, L in enumerate(lens)], np.int64)
    pages = dev(p["code_pages"])
    args = (pages, dev(p["codebooks"]), dev(p["req_set"]), dev(p["block_table"]), dev(p["seq_lens"]), max(lens),
            dev(slots), dev(p["req_set"]), Hq, 1.0 / np.sqrt(128))
    sets, steps = [], []
    for i in range(2):
        q = rng.standard_normal((B, Hq, 128)).astype(np.float32)
        kv = rng.standard_normal((B, Hkv, 2, 128)).astype(np.float16)
        ds = A.DecodeStep(*args)
        if i == 0:                                   # the caller's three pinned tensors
            host = (torch.from_numpy(q).pin_memory(), torch.from_numpy(kv).pin_memory(),
                    torch.empty((B, Hq, 128), dtype=torch.float32).pin_memory())
            ds.capture_host(*host)
        else:                                        # the step's own packed pinned buffers
            host = ds.pinned_io()
            host[0].copy_(torch.from_numpy(q))
            host[1].copy_(torch.from_numpy(kv))
            ds.capture_host()
        sets.append((q, kv, host))
        steps.append(ds)
    steps[0].launch()
    steps[1].launch()
    steps[0].wait()
    got0 = sets[0][2][2].numpy().copy()
    steps[1].wait()
    got1 = sets[1][2][2].numpy().copy()
    for ds in steps:
        ds.check_status()
    for (q, kv, _), got in zip(sets, (got0, got1)):
        want_pages = p["code_pages"].copy()
        orc.encode_append(kv, p["req_set"], slots, p["codebooks"], want_pages, 16)
        want = orc.decode_attention(q, want_pages, p["codebooks"], p["req_set"], p["block_table"], p["seq_lens"],
                                    1.0 / np.sqrt(128), 16)
        close(got, want)


def test_decode_step_host_buffers(A, orc):
    """aq_decode_step_host (api.HostDecodeStep): inputs and output in pinned
    host memory, copies and the step enqueued by one call; the output equals
    aq_decode_step's on device copies of the same inputs bit for bit, and the
    oracle's within tolerance; the new codes land in the cache."""
    B, Hq, Hkv, M, lens = 3, 8, 4, 4, [333, 1024, 17]
    p = W.paged_codes_problem(66, B, Hq, Hkv, M, lens, num_sets=B)
    rng = np.random.default_rng(66)
    q = rng.standard_normal((B, Hq, 128)).astype(np.float32)
    kv = rng.standard_normal((B, Hkv, 2, 128)).astype(np.float16)
    pages_h, pages_d = dev(p["code_pages"]), dev(p["code_pages"])
    args = (dev(p["codebooks"]), dev(p["req_set"]), dev(p["block_table"]), dev(p["seq_lens"]), max(lens))
    hs = A.HostDecodeStep(pages_h, *args, Hq, 1.0 / np.sqrt(128))
    hs.q_host.copy_(torch.from_numpy(q))
    hs.kv_host.copy_(torch.from_numpy(kv))
    hs.launch()
    hs.sync()
    hs.check_status()
    got = hs.out_host.numpy().copy()
    ref = A.decode_step(dev(q), dev(kv), pages_d, args[0], args[1], args[2], args[3], max(lens), 1.0 / np.sqrt(128))
    torch.cuda.synchronize()
    assert np.array_equal(got, ref.cpu().numpy())
    assert torch.equal(pages_h, pages_d)
    slots = np.array([p["block_table"][b, (L - 1) // 16] * 16 + (L - 1) % 16 for b, L in enumerate(lens)], np.int64)
    want_pages = p["code_pages"].copy()
    orc.encode_append(kv, p["req_set"], slots, p["codebooks"], want_pages, 16)
    assert np.array_equal(pages_h.cpu().numpy(), want_pages)
    want = orc.decode_attention(q, want_pages, p["codebooks"], p["req_set"], p["block_table"], p["seq_lens"],
                                1.0 / np.sqrt(128), 16)
    close(got, want)


def test_decode_step_host_pageable_matches_pinned(A):
    """aq_decode_step_host on pageable host buffers (plain numpy arrays: the
    DMA-copy path) and on page-locked ones (api.HostDecodeStep: the gather
    kernel and the direct output write): the same outputs and codes bit for
    bit, over two steps with new inputs."""
    import ctypes
    B, Hq, Hkv, M, lens = 3, 8, 4, 4, [333, 1024, 17]
    p = W.paged_codes_problem(68, B, Hq, Hkv, M, lens, num_sets=B)
    rng = np.random.default_rng(68)
    args = (dev(p["codebooks"]), dev(p["req_set"]), dev(p["block_table"]), dev(p["seq_lens"]), max(lens))
    pages_a, pages_b = dev(p["code_pages"]), dev(p["code_pages"])
    pinned = A.HostDecodeStep(pages_a, *args, Hq, 1.0 / np.sqrt(128))
    paged = A.HostDecodeStep(pages_b, *args, Hq, 1.0 / np.sqrt(128))
    q_np = np.zeros((B, Hq, 128), np.float32)
    kv_np = np.zeros((B, Hkv, 2, 128), np.float16)
    out_np = np.zeros((B, Hq, 128), np.float32)
    call = list(paged._args)
    call[4], call[5], call[18] = (ctypes.c_void_p(a.ctypes.data) for a in (q_np, kv_np, out_np))
    for _ in range(2):
        q = rng.standard_normal((B, Hq, 128)).astype(np.float32)
        kv = rng.standard_normal((B, Hkv, 2, 128)).astype(np.float16)
        pinned.q_host.copy_(torch.from_numpy(q))
        pinned.kv_host.copy_(torch.from_numpy(kv))
        pinned.launch()
        q_np[...] = q
        kv_np[...] = kv
        assert paged._fn(*call) == 0
        pinned.sync()
        paged.sync()
        pinned.check_status()
        paged.check_status()
        assert np.array_equal(pinned.out_host.numpy(), out_np)
        assert torch.equal(pages_a, pages_b)

