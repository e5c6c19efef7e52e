"""The C ABI without a GPU: the library loads, exports every function that
include/aqpq.h declares, and rejects invalid arguments on the host before any
CUDA call (so these run on a CPU-only machine)."""
import ctypes
import os
import re
import subprocess

import pytest

from decode_attention_product_gb300 import _lib, build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "aqpq.h")
FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: checks fail first


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(aq_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert _declared() == sorted(_lib.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (aq_[a-z0-9_]+)$", out, flags=re.M))
    for name in _declared():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_debug_checks_build_compiles_and_exports_every_symbol():
    """The AQ_DEBUG_CHECKS variant (kernels that also check internal invariants
    and report AQ_DEV_INVARIANT) cross-compiles for sm_103a without a GPU, into
    its own directory, and exports the same entry points."""
    path = B.build(debug=True)
    assert path == B.DEBUG_LIB and path != _lib.LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (aq_[a-z0-9_]+)$", out, flags=re.M))
    assert set(_declared()) <= exported


def test_status_strings(lib):
    assert lib.aq_status_string(0) == b"AQ_OK"
    assert lib.aq_status_string(3) == b"AQ_ERR_WORKSPACE_TOO_SMALL"
    assert lib.aq_status_string(99) == b"AQ_ERR_UNKNOWN"
    assert lib.aq_version().startswith(b"aqpq")


def test_wait_limit_setter(lib):
    """Host state only: set, read back as the previous value, clamp at 1 s,
    restore the default (no kernel runs)."""
    prev = lib.aq_set_wait_limit_ns(12345)
    assert prev == 200_000_000
    assert lib.aq_set_wait_limit_ns(5 * 10**9) == 12345
    assert lib.aq_set_wait_limit_ns(prev) == 10**9


def _cfg(M=4, D=128, K=256, P=16):
    return _lib.PQConfig(D, M, K, P)


def _decode(lib, cfg, B=2, Hq=4, Hkv=4, max_pages=8, max_seq_len=100, scale=0.1, splits=0,
            ws=None, wsb=0, q=FAKE):
    return lib.aq_decode_attention(
        ctypes.byref(cfg) if cfg is not None else None, B, Hq, Hkv, q, FAKE, 64, FAKE, 4, FAKE,
        FAKE, max_pages, FAKE, max_seq_len, scale, splits, FAKE, ws, wsb, None, None)


def test_decode_argument_checks(lib):
    INV, UNS, WS = 1, 2, 3
    assert _decode(lib, None) == INV
    assert _decode(lib, _cfg(D=64)) == UNS              # head_dim other than 128
    assert _decode(lib, _cfg(M=3)) == INV               # D % M != 0
    assert _decode(lib, _cfg(M=16)) == UNS              # Dsub 8 not built
    assert _decode(lib, _cfg(K=512)) == INV             # codes are 8-bit
    assert _decode(lib, _cfg(K=128)) == UNS
    assert _decode(lib, _cfg(P=32)) == UNS
    assert _decode(lib, _cfg(), Hq=6, Hkv=4) == INV     # Hq % Hkv != 0
    assert _decode(lib, _cfg(), Hq=48, Hkv=2) == UNS    # group of 24
    assert _decode(lib, _cfg(), max_pages=4, max_seq_len=65) == INV   # beyond the table
    assert _decode(lib, _cfg(), scale=float("nan")) == INV
    assert _decode(lib, _cfg(), B=-1) == INV
    assert _decode(lib, _cfg(), q=None) == INV
    assert _decode(lib, _cfg(), B=0) == 0               # empty batch: nothing to do
    # forced splits need a workspace
    assert _decode(lib, _cfg(), max_seq_len=100, splits=3) == WS


def test_misaligned_tensors_rejected(lib):
    odd = ctypes.c_void_p(0x10008)                      # 8-byte but not 16-byte aligned
    assert _decode(lib, _cfg(), q=odd) == 1
    cfg = _cfg()
    assert lib.aq_encode_append(ctypes.byref(cfg), 4, 2, odd, FAKE, FAKE, FAKE, 1, FAKE, 1, None,
                                None) == 1
    assert lib.aq_fit_codebooks(ctypes.byref(cfg), 4, 64, 10, FAKE, odd, None, None) == 1


def test_fp16_decode_argument_checks(lib):
    cfg = _cfg()
    r = lib.aq_decode_attention_fp16(ctypes.byref(cfg), 2, 4, 4, FAKE, None, 8, FAKE, 8, FAKE, 100,
                                     0.1, 0, FAKE, None, 0, None, None)
    assert r == 1                                       # kv_pages NULL
    r = lib.aq_decode_attention_fp16(ctypes.byref(cfg), 2, 4, 4, FAKE, FAKE, 8, FAKE, 8, FAKE, 100,
                                     0.1, 4, FAKE, None, 0, None, None)
    assert r == 3


def test_encode_and_fit_argument_checks(lib):
    cfg = _cfg()
    assert lib.aq_encode_append(ctypes.byref(cfg), 4, 0, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 1, None,
                                None) == 1          # no kv heads
    assert lib.aq_encode_append(ctypes.byref(cfg), 4, 2, None, FAKE, FAKE, FAKE, 1, FAKE, 1, None,
                                None) == 1
    assert lib.aq_encode_append(ctypes.byref(cfg), 0, 2, None, None, None, None, 1, None, 1, None,
                                None) == 0          # nothing to encode
    assert lib.aq_fit_codebooks(ctypes.byref(cfg), 4, 0, 10, FAKE, FAKE, None, None) == 1
    assert lib.aq_fit_codebooks(ctypes.byref(cfg), 4, 2048, 10, FAKE, FAKE, None, None) == 2
    assert lib.aq_fit_codebooks(ctypes.byref(cfg), 4, 64, 0, FAKE, FAKE, None, None) == 1
    assert lib.aq_fit_codebooks(ctypes.byref(cfg), 0, 64, 10, None, None, None, None) == 0
    assert lib.aq_kmeans_step(ctypes.byref(cfg), 4, 64, FAKE, FAKE, FAKE, None, None) == 1
    assert lib.aq_refine_codebooks(ctypes.byref(cfg), 4, 64, 0, FAKE, FAKE, None, None) == 1   # iters
    assert lib.aq_refine_codebooks(ctypes.byref(cfg), 4, 2048, 3, FAKE, FAKE, None, None) == 2
    assert lib.aq_refine_codebooks(ctypes.byref(cfg), 4, 64, 3, None, FAKE, None, None) == 1
    assert lib.aq_refine_codebooks(ctypes.byref(cfg), 4, 64, 3, FAKE, ctypes.c_void_p(0x10008), None,
                                   None) == 1                          # misaligned codebooks
    assert lib.aq_refine_codebooks(ctypes.byref(cfg), 0, 64, 3, None, None, None, None) == 0


def test_decode_step_flags_checked(lib):
    cfg = _cfg()
    def step(flags, kv_new=FAKE):
        return lib.aq_decode_step(ctypes.byref(cfg), 2, 4, 4, FAKE, kv_new, FAKE, 64, FAKE, 4, FAKE, FAKE,
                                  8, FAKE, 100, 0.1, 0, flags, FAKE, None, 0, None, None)
    assert step(4) == 1                                 # unknown flag
    assert step(2, kv_new=None) == 1                    # a step needs its new token


def test_decode_step_host_argument_checks(lib):
    """The host-buffer step checks every argument (its own and the step's)
    before it enqueues a transfer or a kernel: without a GPU each rejected call
    returns its argument error, never a CUDA one."""
    cfg = _cfg()
    B, Hq, Hkv = 2, 4, 4
    need = lib.aq_decode_step_host_staging(B, Hq, Hkv)
    assert need >= B * Hq * 128 * 4 * 2 + B * Hkv * 2 * 128 * 2

    def step(c=cfg, batch=B, Hq=Hq, q=FAKE, staging=FAKE, sbytes=None, flags=0, scale=0.1, splits=0,
             max_seq_len=100):
        if sbytes is None:
            sbytes = lib.aq_decode_step_host_staging(batch, Hq, Hkv)
        return lib.aq_decode_step_host(ctypes.byref(c) if c is not None else None, batch, Hq, Hkv, q, FAKE, FAKE,
                                       64, FAKE, 4, FAKE, FAKE, 8, FAKE, max_seq_len, scale, splits, flags, FAKE,
                                       staging, sbytes, None, 0, None, None)
    assert step(q=None) == 1                            # host query missing
    assert step(staging=None) == 1
    assert step(staging=ctypes.c_void_p(0x10008)) == 1  # staging not 16-byte aligned
    assert step(sbytes=need - 1) == 3                   # staging too small
    assert step(flags=4) == 1                           # unknown flag
    assert step(c=None) == 1                            # the step's own checks, before any transfer
    assert step(c=_cfg(M=16)) == 2
    assert step(Hq=6) == 1
    assert step(scale=float("nan")) == 1
    assert step(splits=3) == 3                          # forced splits need a workspace
    assert step(c=None, batch=0) == 1                   # an empty batch still needs a valid config
    assert step(batch=0, q=None, staging=None, sbytes=0) == 0   # nothing to do


def test_e4m3_conversion_argument_checks(lib):
    assert lib.aq_codebooks_to_e4m3(-1, FAKE, FAKE, None) == 1
    assert lib.aq_codebooks_to_e4m3(0, None, None, None) == 0
    assert lib.aq_codebooks_to_e4m3(8, None, FAKE, None) == 1
    assert lib.aq_codebooks_to_e4m3(8, FAKE, ctypes.c_void_p(0x10004), None) == 1
    assert lib.aq_codebooks_from_e4m3(8, FAKE, None, None) == 1
    assert lib.aq_codebooks_from_e4m3(8, ctypes.c_void_p(0x10001), FAKE, None) == 1


def _plan(lib, B, Hq, Hkv, L, M=4, splits=0, fp16=0):
    cfg = _cfg(M=M)
    s, c, w = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    r = lib.aq_decode_plan(ctypes.byref(cfg), B, Hq, Hkv, L, splits, fp16, ctypes.byref(s),
                           ctypes.byref(c), ctypes.byref(w))
    assert r == 0
    return s.value, c.value, w.value


def test_plans_for_the_workloads(lib):
    # B4 H32 L2048 M4: 128 clusters of 4 CTAs fill the GPU, no split, no workspace
    assert _plan(lib, 4, 32, 32, 2048) == (1, 4, 0)
    # 80-layer GQA shape (8 kv heads serve 64 query heads)
    s, c, w = _plan(lib, 8, 64, 8, 1000)
    assert c == 4 and s == 1 and w == 0
    # B1 H32 L131072 M8: 2 splits of clusters of 8 (each CTA streams 8192
    # tokens); the workspace (B*Hq*S*(D+2) floats) also covers the E4M3 plan,
    # whose CTAs hold one chunk and so split into 16
    s, c, w = _plan(lib, 1, 32, 32, 131072, M=8)
    assert (s, c) == (2, 8) and w == 1 * 32 * 16 * 130 * 4
    # ragged 256 requests: enough clusters already
    assert _plan(lib, 256, 32, 32, 4096)[0] == 1
    # forced split counts are honoured (rounded so no split is empty)
    assert _plan(lib, 2, 4, 4, 100, splits=3)[0] == 3
    assert _plan(lib, 2, 4, 4, 100, splits=50)[0] == 7     # 7 pages
    assert _plan(lib, 2, 4, 4, 0, splits=5)[0] == 1


def test_every_supported_shape_has_a_plan(lib):
    """Each supported (M, group) pair plans within the shared-memory budget,
    for short and very long sequences; a very long one is split at least for
    E4M3 codebooks (one chunk per CTA), so the reported workspace is never 0,
    and covers the plan's own splits."""
    for M in (4, 8):
        for G in (1, 2, 4, 8):
            for L in (1, 100, 4096, 131072):
                s, c, w = _plan(lib, 2, 4 * G, 4, L, M=M)
                assert c in ((1, 2, 4, 8) if M == 8 else (1, 2, 4)) and s >= 1
                assert w >= (2 * 4 * G * s * 130 * 4 if s > 1 else 0)
                if L == 131072:
                    assert w > 0


def test_mixed_workspace_covers_every_pq_plan(lib):
    """The mixed step's workspace holds the fp16 part's split partials and the
    PQ part's for any plan that part can take: either codebook format, and the
    token-share plan that replaces the head-split one when the codebooks get no
    TMA view.  aq_decode_plan's workspace for the PQ heads alone covers those
    plans (B * Hq_pq * S * (D + 2) floats); the mixed step indexes partials by
    the full query-head numbering, so it needs the same S over all Hq heads."""
    for (B, Hq, Hkv, n16, L, M) in [(1, 64, 8, 2, 131072, 4), (1, 64, 8, 2, 131072, 8), (2, 32, 8, 4, 20000, 4),
                                    (1, 32, 32, 4, 131072, 8), (4, 32, 32, 4, 2048, 4), (8, 64, 8, 1, 1000, 4)]:
        cfg = _cfg(M=M)
        ws = ctypes.c_size_t()
        assert lib.aq_decode_step_mixed_workspace(ctypes.byref(cfg), B, Hq, Hkv, n16, L, ctypes.byref(ws)) == 0
        G = Hq // Hkv
        s16, _, _ = _plan(lib, B, n16 * G, n16, L, M=M, fp16=1)
        _, _, wpq = _plan(lib, B, (Hkv - n16) * G, Hkv - n16, L, M=M)
        spq = wpq // (B * (Hkv - n16) * G * 130 * 4)
        need = (B * Hq * s16 * 130 * 4 if s16 > 1 else 0) + (B * Hq * spq * 130 * 4 if spq > 1 else 0)
        assert ws.value >= need, (B, Hq, Hkv, n16, L, M, ws.value, need)


def test_wrappers_reject_tensors_on_another_device():
    """The torch wrappers run the C call with the tensors' device current and
    refuse a call whose tensors sit on different devices (checked without a
    GPU: CPU tensors report device index -1, the stand-in reports device 1)."""
    torch = pytest.importorskip("torch")
    from decode_attention_product_gb300 import api

    class OnDevice1:
        device = "cuda:1"

        def get_device(self):
            return 1
    a = torch.zeros(4)
    assert api._same_device(a, x=torch.zeros(2), y=None) == -1
    with pytest.raises(ValueError, match="cuda:1"):
        api._same_device(a, codebooks=OnDevice1())


def test_lengths_beyond_the_split_limit_are_unsupported(lib):
    """A CTA holds a bounded share of tokens and a call runs at most 4096
    splits, so the longest request a plan can take is bounded: the planner
    reports AQ_ERR_UNSUPPORTED beyond it (never a plan the launch would refuse),
    and the decode calls return the same before any CUDA call.  M = 4 with one
    query head per kv head holds 2048 tokens per CTA, 16 chunks of them when
    streamed (fp16 codebooks, clusters of 4): 2^29 tokens at most; E4M3
    codebooks stream nothing: 2^25 tokens at most."""
    UNS = 2
    s, c, w = _plan(lib, 1, 1, 1, 1 << 28)
    assert s <= 4096 and c == 4 and w >= s * 130 * 4
    assert _plan(lib, 1, 1, 1, 1 << 29)[:2] == (4096, 4)
    cfg = _cfg()
    out = (ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t())
    r = lib.aq_decode_plan(ctypes.byref(cfg), 1, 1, 1, 1 << 30, 0, 0, *(ctypes.byref(x) for x in out))
    assert r == UNS
    r = lib.aq_decode_plan(ctypes.byref(_cfg(M=8)), 1, 1, 1, 1 << 29, 0, 0, *(ctypes.byref(x) for x in out))
    assert r == UNS
    assert _plan(lib, 1, 1, 1, 1 << 30, fp16=1)[0] >= 1        # the fp16 comparison plan has no such bound
    # the calls themselves: rejected on the host.  Their pointers are fake, so
    # they run only where no GPU could be reached if a regression let them pass
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        return
    L = (1 << 30)
    assert _decode(lib, _cfg(), B=1, Hq=1, Hkv=1, max_pages=L // 16, max_seq_len=L) == UNS
    L = (1 << 25) + 16
    r = lib.aq_decode_step(ctypes.byref(cfg), 1, 1, 1, FAKE, FAKE, FAKE, 64, FAKE, 1, FAKE, FAKE, L // 16 + 1,
                           FAKE, L, 0.1, 0, 2, FAKE, FAKE, 1 << 30, None, None)   # AQ_STEP_E4M3
    assert r == UNS
