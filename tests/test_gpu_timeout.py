"""The decode kernels' bounded waits, made to run out.

With the wait limit lowered to zero (aq_set_wait_limit_ns), the waits of a
page1-sized decode on cold data give up before their copies land: the call
must still return, report AQ_DEV_TIMEOUT in the status word, and leave every
output either NaN (touched by a wait that ran out) or correct; the context
stays usable, and the next call with the default limit is correct everywhere.
The kernels always wait (up to 200 ms) for their copies to land before they
exit, whatever the limit, so nothing is left in flight.
"""
import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-3
AQ_DEV_TIMEOUT = 8


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


@pytest.mark.parametrize("kernel", ["1", "2"])
def test_zero_wait_limit_reports_timeout_and_nan(A, orc, kernel, monkeypatch):
    from decode_attention_product_gb300 import _lib
    monkeypatch.setenv("AQPQ_DECODE_KERNEL", kernel)
    p = W.paged_codes_problem(321, 4, 32, 32, 4, [2048] * 4)
    want = orc.decode_attention(p["q"], p["code_pages"], p["codebooks"], p["req_set"], p["block_table"],
                                p["seq_lens"], 1.0 / np.sqrt(128), 16)
    t = {k: dev(v) for k, v in p.items() if k != "num_pages"}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

    def run():
        st = A.new_status()
        flush.zero_()                                  # cold L2: the copies take microseconds
        out = A.decode_attention(t["q"], t["code_pages"], t["codebooks"], t["req_set"], t["block_table"],
                                 t["seq_lens"], 2048, 1.0 / np.sqrt(128), status=st)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64), int(st.item())

    lib = _lib.load()
    prev = lib.aq_set_wait_limit_ns(0)
    try:
        got, st = run()
    finally:
        lib.aq_set_wait_limit_ns(prev)
    assert st & AQ_DEV_TIMEOUT
    nan = np.isnan(got)
    assert nan.any()
    ok = ~nan
    assert np.all(np.abs(got[ok] - want[ok]) <= ATOL + RTOL * np.abs(want[ok]))
    # the context is intact: the default limit gives the full answer
    got2, st2 = run()
    assert st2 == 0
    assert np.all(np.abs(got2 - want) <= ATOL + RTOL * np.abs(want))


@pytest.mark.parametrize("e4m3", [False, True], ids=["fp16_codebooks", "e4m3_codebooks"])
@pytest.mark.parametrize("heads", [(32, 32), (64, 8)], ids=["token_share", "head_split"])
def test_fused_step_zero_wait_limit(A, orc, heads, e4m3):
    """The fused step (append + attention) with every wait limit at zero, on
    cold data: the token-share kernel (one query head per kv head) and the
    head-split kernel (groups of 8), fp16 and E4M3 codebooks (raw slices
    widened after they land).  The call returns and reports the timeout;
    every output is NaN or correct; every byte of a new token's page slot is
    either its old value or the oracle's code (a CTA that gave up writes no
    codes), and nothing else in the cache changes.  The same step with the
    default limit on a fresh cache is then correct everywhere."""
    from decode_attention_product_gb300 import _lib
    Hq, Hkv = heads
    B, M, L = (4, 4, 2048) if Hq == Hkv else (8, 4, 1000)
    p = W.paged_codes_problem(322 + Hkv, B, Hq, Hkv, M, [L] * B)
    rng = np.random.default_rng(322 + Hkv)
    kv = rng.standard_normal((B, Hkv, 2, 128)).astype(np.float16)
    cb = dev(p["codebooks"])
    cb_step = A.to_e4m3(cb) if e4m3 else cb
    cb_w = A.from_e4m3(cb_step).cpu().numpy() if e4m3 else p["codebooks"]
    slots = np.array([p["block_table"][b, (L - 1) // 16] * 16 + (L - 1) % 16 for b in range(B)], np.int64)
    want_pages = p["code_pages"].copy()
    orc.encode_append(kv, p["req_set"], slots, cb_w, want_pages, 16)
    want = orc.decode_attention(p["q"], want_pages, cb_w, p["req_set"], p["block_table"], p["seq_lens"],
                                1.0 / np.sqrt(128), 16)
    t = {k: dev(v) for k, v in p.items() if k not in ("num_pages", "code_pages", "codebooks")}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

    def run():
        pages = dev(p["code_pages"])
        st = A.new_status()
        flush.zero_()                                  # cold L2: the copies take microseconds
        out = A.decode_step(t["q"], dev(kv), pages, cb_step, t["req_set"], t["block_table"], t["seq_lens"], L,
                            1.0 / np.sqrt(128), status=st)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64), pages.cpu().numpy(), int(st.item())

    lib = _lib.load()
    prev = lib.aq_set_wait_limit_ns(0)
    try:
        got, pages, st = run()
    finally:
        lib.aq_set_wait_limit_ns(prev)
    assert st & AQ_DEV_TIMEOUT
    nan = np.isnan(got)
    assert nan.any()
    ok = ~nan
    assert np.all(np.abs(got[ok] - want[ok]) <= ATOL + RTOL * np.abs(want[ok]))
    old = p["code_pages"]
    assert np.all((pages == old) | (pages == want_pages))
    changed = want_pages != old                        # only the new tokens' slots may change
    assert np.array_equal(pages[~changed], old[~changed])
    # the context is intact: the default limit gives the full answer
    got2, pages2, st2 = run()
    assert st2 == 0
    assert np.array_equal(pages2, want_pages)
    assert np.all(np.abs(got2 - want) <= ATOL + RTOL * np.abs(want))
