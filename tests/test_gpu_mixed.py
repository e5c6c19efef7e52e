"""GPU parity of the mixed-precision decode step (AQPIM blog §6.1 item 4):
kv heads [0, n16) keep an fp16 cache, the others a PQ cache, in one step.

Both sides start from the same raw K/V vectors.  The GPU fits the PQ heads'
codebooks, encodes their first L-1 tokens, writes the fp16 heads' first L-1
tokens into fp16 pages, then runs aq_decode_step_mixed with token L-1 as the
new token.  The oracle fits, encodes all L tokens and writes all L fp16 rows,
then runs its mixed attention.  Codebooks, code pages and fp16 pages must be
bit-exact; outputs within |o - o*| <= 2e-3 + 2e-3 |o*|.
"""
import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-3


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_product_gb300 import build
    build.build()
    from decode_attention_product_gb300 import api
    return api


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def fp16_pages(kvs, bt, npages, heads, upto):
    """fp16 pages [NP][len(heads)][2][P][D] with tokens [0, upto(b)) of every
    request (numpy placement of the raw vectors, no arithmetic)."""
    H = len(heads)
    pages = np.zeros((npages, H, 2, 16, 128), np.float16)
    for b, k in enumerate(kvs):
        n = upto(len(k))
        t = np.arange(n)
        pages[bt[b, t // 16], :, :, t % 16] = k[:n][:, heads]
    return pages


CASES = [
    # (workload overrides, n16 values)
    ("page1", dict(seq_lens=[300, 1000, 65, 2048], num_q_heads=8, num_kv_heads=8), [0, 1, 5, 8]),
    ("qwen_gqa", dict(seq_lens=[1000, 64, 640, 999]), [0, 2, 8]),
]


@pytest.mark.parametrize("e4m3", [False, True], ids=["fp16_codebooks", "e4m3_codebooks"])
@pytest.mark.parametrize("name,over,n16s", CASES, ids=[c[0] for c in CASES])
def test_mixed_step_matches_oracle(A, orc, name, over, n16s, e4m3):
    w = W.make(name, **over)
    w.layers = 1
    B, Hkv, M = w.batch, w.num_kv_heads, w.num_subspaces
    kvs = w.kv_all(threads=8)
    bt, npages = w.block_table()
    q = w.queries()
    last = np.stack([k[-1] for k in kvs])
    L = int(w.seq_lens.max())
    for n16 in n16s:
        pq_heads = list(range(n16, Hkv))
        npq = len(pq_heads)
        # ---- GPU: caches for the first L-1 tokens, then the mixed step ----
        kvp = dev(fp16_pages(kvs, bt, npages, list(range(n16)), lambda n: n - 1)) if n16 else None
        pages = cbs_step = None
        cb_gpu = None
        st = A.new_status()
        if npq:
            samples = np.stack([w.fit_samples(k[:, pq_heads]) for k in kvs])
            cb = A.fit_codebooks(dev(samples.reshape(-1, *samples.shape[3:])), M, w.fit_iters)
            cb = cb.view(B, npq, 2, M, 256, w.dsub)
            cbs_step = cb
            if e4m3:
                cbs_step = A.to_e4m3(cb)
                cb = A.from_e4m3(cbs_step)
            cb_gpu = cb
            kv = np.concatenate([k[:-1, pq_heads] for k in kvs])
            tset = np.concatenate([np.full(len(k) - 1, b, np.int32) for b, k in enumerate(kvs)])
            slots = np.concatenate([w.slot_mapping(bt, b, 0, len(k) - 1) for b, k in enumerate(kvs)])
            pages = torch.zeros((npages, npq, 16, 2, M), dtype=torch.uint8, device="cuda")
            if len(kv):
                A.encode_append(dev(kv), dev(tset), dev(slots), cb, pages, st)
        out = A.decode_step_mixed(dev(q), dev(last), n16, kvp, pages, cbs_step,
                                  torch.arange(B, dtype=torch.int32, device="cuda"), dev(bt), dev(w.seq_lens),
                                  L, num_subspaces=M, scale=w.scale, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        # ---- oracle: the same from the raw vectors, all L tokens ----
        want_kvp = fp16_pages(kvs, bt, npages, list(range(n16)), lambda n: n) if n16 else None
        want_pages = cbw = None
        if npq:
            samples = np.stack([w.fit_samples(k[:, pq_heads]) for k in kvs])
            cb16, _, _, _ = orc.kmeans_fit(samples.reshape(-1, *samples.shape[3:]), M, 256, w.fit_iters)
            cb16 = cb16.reshape(B, npq, 2, M, 256, w.dsub)
            cbw = orc.e4m3_to_float(orc.e4m3_from_float(cb16.astype(np.float32))).astype(np.float16) if e4m3 else cb16
            assert np.array_equal(cb_gpu.cpu().numpy().view(np.uint16), cbw.view(np.uint16))
            kv = np.concatenate([k[:, pq_heads] for k in kvs])
            tset = np.concatenate([np.full(len(k), b, np.int32) for b, k in enumerate(kvs)])
            slots = np.concatenate([w.slot_mapping(bt, b, 0, len(k)) for b, k in enumerate(kvs)])
            want_pages = np.zeros((npages, npq, 16, 2, M), np.uint8)
            orc.encode_append(kv, tset, slots, cbw, want_pages, 16)
            assert np.array_equal(pages.cpu().numpy(), want_pages)
        if n16:
            assert np.array_equal(kvp.cpu().numpy().view(np.uint16), want_kvp.view(np.uint16))
        want = orc.decode_attention_mixed(q, want_kvp, want_pages, cbw, np.arange(B, dtype=np.int32), bt,
                                          w.seq_lens, w.scale, 16, n16)
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        err = np.abs(got - want)
        bad = err > ATOL + RTOL * np.abs(want)
        assert not bad.any(), f"n16={n16}: {bad.sum()} outside tol, max err {err.max():.3e}"


def test_mixed_step_rejects_bad_head_count(A):
    q = torch.zeros((1, 4, 128), device="cuda")
    kv = torch.zeros((1, 4, 2, 128), dtype=torch.float16, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    kvp = torch.zeros((1, 5, 2, 16, 128), dtype=torch.float16, device="cuda")
    from decode_attention_product_gb300._lib import AQError
    with pytest.raises(AQError):
        A.decode_step_mixed(q, kv, 5, kvp, None, None, None, bt, lens, 1)
