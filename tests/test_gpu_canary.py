"""Out-of-bounds write checks: every output, workspace and cache buffer sits
inside a larger canary-filled allocation, and after the call the canary bytes
around the region the call may write are unchanged.  Covers the token-share
kernel (one split, several splits with the combine, a streamed share), the
head-split kernel of a GQA group of 8 and the fp16 comparison kernel with its
combine; the outputs are also checked against the oracle.
"""
import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-3
PAD = 4096                                             # canary bytes on each side
CANARY = 0xA5


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


def fenced(nbytes, dtype, shape=None, fill=None):
    """A view of `nbytes` in the middle of a canary-filled byte buffer: (buffer, view).
    `fill` (a numpy array) is copied into the view."""
    buf = torch.full((PAD + nbytes + PAD,), CANARY, dtype=torch.uint8, device="cuda")
    view = buf[PAD:PAD + nbytes].view(dtype)
    if shape is not None:
        view = view.view(shape)
    if fill is not None:
        view.copy_(torch.from_numpy(np.ascontiguousarray(fill)).cuda())
    return buf, view


def assert_fence(buf, what):
    b = buf.cpu().numpy()
    assert np.all(b[:PAD] == CANARY) and np.all(b[-PAD:] == CANARY), f"write outside {what}"


def close(got, want):
    err = np.abs(np.asarray(got, np.float64) - want)
    assert np.all(np.isfinite(got)) and np.all(err <= ATOL + RTOL * np.abs(want)), f"max err {err.max():.3e}"


PQ_CASES = [
    # (B, Hq, Hkv, M, lens, splits)
    (2, 4, 4, 4, [700, 45], 0),                # token-share, one split
    (2, 4, 4, 4, [700, 45], 3),                # token-share, three splits + combine
    (1, 2, 2, 4, [30001], 1),                  # token-share, a streamed share
    (2, 16, 2, 4, [1000, 257], 0),             # head-split kernel, group of 8
    (1, 4, 4, 8, [20000], 0),                  # M = 8, clusters of 8 over several splits
]


@pytest.mark.parametrize("case", PQ_CASES, ids=[f"B{c[0]}Hq{c[1]}Hkv{c[2]}M{c[3]}S{c[5]}" for c in PQ_CASES])
def test_fused_step_writes_inside_its_buffers(A, orc, case):
    B, Hq, Hkv, M, lens, splits = case
    p = W.paged_codes_problem(900 + B * Hq + M, B, Hq, Hkv, M, lens, num_sets=B)
    kv = np.random.default_rng(901).standard_normal((B, Hkv, 2, 128)).astype(np.float16)
    slots = np.array([p["block_table"][b, (L - 1) // 16] * 16 + (L - 1) % 16 for b, L in enumerate(lens)],
                     np.int64)
    want_pages = p["code_pages"].copy()
    orc.encode_append(kv, p["req_set"], slots, p["codebooks"], want_pages, 16)
    want = orc.decode_attention(p["q"], want_pages, p["codebooks"], p["req_set"], p["block_table"],
                                p["seq_lens"], 1.0 / np.sqrt(128), 16)
    L = int(max(lens))
    _, _, wsb = A.decode_plan(B, Hq, Hkv, L, M, splits)
    out_buf, out = fenced(B * Hq * 128 * 4, torch.float32, (B, Hq, 128))
    ws_buf, ws = fenced(max(wsb, 16), torch.uint8)
    pg_buf, pages = fenced(p["code_pages"].nbytes, torch.uint8, p["code_pages"].shape, p["code_pages"])
    st = A.new_status()
    A.decode_step(dev(p["q"]), dev(kv), pages, dev(p["codebooks"]), dev(p["req_set"]), dev(p["block_table"]),
                  dev(p["seq_lens"]), L, 1.0 / np.sqrt(128), num_splits=splits, out=out,
                  workspace=ws if wsb else None, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_fence(out_buf, "the output")
    assert_fence(ws_buf, "the workspace")
    assert_fence(pg_buf, "the code pages")
    assert np.array_equal(pages.cpu().numpy(), want_pages)
    close(out.cpu().numpy(), want)


@pytest.mark.parametrize("splits", [1, 3])
def test_fp16_decode_writes_inside_its_buffers(A, orc, splits):
    B, Hq, Hkv, lens = 2, 8, 2, [700, 45]
    p = W.paged_fp16_problem(903, B, Hq, Hkv, lens)
    want = orc.decode_attention_fp16(p["q"], p["kv_pages"], p["block_table"], p["seq_lens"], 1.0 / np.sqrt(128))
    L = int(max(lens))
    _, _, wsb = A.decode_plan(B, Hq, Hkv, L, 4, splits, fp16=True)
    out_buf, out = fenced(B * Hq * 128 * 4, torch.float32, (B, Hq, 128))
    ws_buf, ws = fenced(max(wsb, 16), torch.uint8)
    st = A.new_status()
    A.decode_attention_fp16(dev(p["q"]), dev(p["kv_pages"]), dev(p["block_table"]), dev(p["seq_lens"]), L,
                            1.0 / np.sqrt(128), num_splits=splits, out=out, workspace=ws if wsb else None,
                            status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_fence(out_buf, "the output")
    assert_fence(ws_buf, "the workspace")
    close(out.cpu().numpy(), want)
