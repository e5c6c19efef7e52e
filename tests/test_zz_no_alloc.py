"""aq_decode_attention_noalloc, the decode entry point for callers that cannot
allocate device memory (its split scratch is a fixed array inside the
library), checked through the C ABI against aq_decode_attention with a
caller-supplied workspace, on two calls in a row.

Kept in its own file, collected last, so that a run stopping at the first
failure has run every other test before it."""
import ctypes

import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_product_gb300 import build
    build.build()
    from decode_attention_product_gb300 import _lib, api
    return _lib, api


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _noalloc(lib, _lib, t, M, max_seq_len, splits, out, status):
    B, Hq, _ = t["q"].shape
    Hkv = t["codebooks"].shape[1]
    cfg = _lib.config(M)
    return lib.aq_decode_attention_noalloc(
        ctypes.byref(cfg), B, Hq, Hkv, t["q"].data_ptr(), t["code_pages"].data_ptr(),
        t["code_pages"].shape[0], t["codebooks"].data_ptr(), t["codebooks"].shape[0],
        t["req_set"].data_ptr(), t["block_table"].data_ptr(), t["block_table"].shape[1],
        t["seq_lens"].data_ptr(), max_seq_len, 128 ** -0.5, splits, out.data_ptr(),
        status.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("splits", [0, 7])
def test_noalloc_matches_workspace_entry_point(splits):
    _lib, api = _setup()
    lib = _lib.load()
    M, lens = 8, [20000, 7000]
    p = W.paged_codes_problem(11, 2, 8, 8, M, lens, num_sets=2)
    t = {k: _dev(v) for k, v in p.items() if k != "num_pages"}
    L = max(lens)
    assert api.decode_plan(2, 8, 8, L, M, splits)[0] > 1      # the scratch is exercised
    ref = api.decode_attention(t["q"], t["code_pages"], t["codebooks"], t["req_set"],
                               t["block_table"], t["seq_lens"], L, num_splits=splits)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy().astype(np.float64)
    for _ in range(2):
        out = torch.full((2, 8, 128), float("nan"), device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, _lib, t, M, L, splits, out, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= TOL + TOL * np.abs(ref))
        # same plan, same kernels, only the scratch differs: bit-identical
        assert np.array_equal(got, ref)


def test_noalloc_rejects_scratch_beyond_its_array():
    _lib, _ = _setup()
    lib = _lib.load()
    cfg = _lib.config(4)
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: rejected before any launch
    # 4096 requests x 32 heads x 64 splits of (128 + 2) floats is far beyond 4 MiB
    r = lib.aq_decode_attention_noalloc(ctypes.byref(cfg), 4096, 32, 32, fake, fake, 1 << 20, fake,
                                        4096, fake, fake, 4096, fake, 65536, 0.1, 64, fake, None,
                                        None)
    assert r == 3                             # AQ_ERR_WORKSPACE_TOO_SMALL
