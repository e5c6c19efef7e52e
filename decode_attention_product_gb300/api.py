"""Torch-facing wrappers of the C ABI (device memory and streams from PyTorch).

Each function checks dtypes, devices and contiguity, passes raw pointers and
the current CUDA stream to libaqpq, and raises AQError on a non-OK status.  No
arithmetic of the method happens here.  Names follow include/aqpq.h.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

HEAD_DIM = 128
CODEWORDS = 256
PAGE = 16


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _same_device(ref, **tensors) -> int:
    """ref's device index, once every given tensor is on that device (the
    library launches on the current device, which each wrapper sets to this
    one for the call)."""
    d = ref.get_device()
    for name, t in tensors.items():
        if t is not None and t.get_device() != d:
            raise ValueError(f"{name} is on {t.device}, the call's other tensors on {ref.device}")
    return d


def _need(t, dtype, name, ndim=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t


def new_status(device=None) -> torch.Tensor:
    """A zeroed int32 device_status word."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def fit_codebooks(samples: torch.Tensor, num_subspaces: int, iters: int = 10,
                  with_assign: bool = False):
    """Lloyd k-means codebooks from samples [U][N][D] fp16 -> fp16 [U][M][K][Dsub]."""
    _need(samples, torch.float16, "samples", 3)
    U, N, D = samples.shape
    M = num_subspaces
    cb = torch.empty((U, M, CODEWORDS, D // M), dtype=torch.float16, device=samples.device)
    asg = torch.empty((U, N, M), dtype=torch.int32, device=samples.device) if with_assign else None
    cfg = _lib.config(M, head_dim=D)
    dev = samples.get_device()
    with torch.cuda.device(dev):
        st = _lib.load().aq_fit_codebooks(ctypes.byref(cfg), U, N, iters, _ptr(samples), _ptr(cb),
                                          _ptr(asg), _stream(dev))
    _lib.check(st, "aq_fit_codebooks")
    return (cb, asg) if with_assign else cb


def refine_codebooks(samples: torch.Tensor, codebooks: torch.Tensor, iters: int = 3,
                     with_assign: bool = False):
    """Periodic codebook update in place: `iters` Lloyd steps on samples [U][N][D]
    fp16 starting from codebooks [U][M][K][Dsub] fp16 (returns the assignment
    [U][N][M] of the last step when asked)."""
    _need(samples, torch.float16, "samples", 3)
    _need(codebooks, torch.float16, "codebooks", 4)
    U, N, D = samples.shape
    M = codebooks.shape[1]
    if codebooks.shape[0] != U:
        raise ValueError("one codebook per sample unit")
    dev = _same_device(samples, codebooks=codebooks)
    asg = torch.empty((U, N, M), dtype=torch.int32, device=samples.device) if with_assign else None
    cfg = _lib.config(M, head_dim=D)
    with torch.cuda.device(dev):
        st = _lib.load().aq_refine_codebooks(ctypes.byref(cfg), U, N, iters, _ptr(samples), _ptr(codebooks),
                                             _ptr(asg), _stream(dev))
    _lib.check(st, "aq_refine_codebooks")
    return asg


def to_e4m3(x: torch.Tensor) -> torch.Tensor:
    """FP8 E4M3 codes (uint8, same shape) of an fp16 tensor (nearest, ties to
    even, saturating)."""
    _need(x, torch.float16, "x")
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    dev = x.get_device()
    with torch.cuda.device(dev):
        st = _lib.load().aq_codebooks_to_e4m3(x.numel(), _ptr(x), _ptr(out), _stream(dev))
    _lib.check(st, "aq_codebooks_to_e4m3")
    return out


def from_e4m3(codes: torch.Tensor) -> torch.Tensor:
    """The exact fp16 values (same shape) of FP8 E4M3 codes."""
    _need(codes, torch.uint8, "codes")
    out = torch.empty(codes.shape, dtype=torch.float16, device=codes.device)
    dev = codes.get_device()
    with torch.cuda.device(dev):
        st = _lib.load().aq_codebooks_from_e4m3(codes.numel(), _ptr(codes), _ptr(out), _stream(dev))
    _lib.check(st, "aq_codebooks_from_e4m3")
    return out


def kmeans_step(samples: torch.Tensor, centroids: torch.Tensor):
    """One Lloyd step from fp32 centroids [U][M][K][Dsub]: (centroids_out, assign)."""
    _need(samples, torch.float16, "samples", 3)
    _need(centroids, torch.float32, "centroids", 4)
    U, N, D = samples.shape
    M = centroids.shape[1]
    dev = _same_device(samples, centroids=centroids)
    out = torch.empty_like(centroids)
    asg = torch.empty((U, N, M), dtype=torch.int32, device=samples.device)
    cfg = _lib.config(M, head_dim=D)
    with torch.cuda.device(dev):
        st = _lib.load().aq_kmeans_step(ctypes.byref(cfg), U, N, _ptr(samples), _ptr(centroids),
                                        _ptr(out), _ptr(asg), _stream(dev))
    _lib.check(st, "aq_kmeans_step")
    return out, asg


def encode_append(kv: torch.Tensor, token_set: torch.Tensor, slot_mapping: torch.Tensor,
                  codebooks: torch.Tensor, code_pages: torch.Tensor,
                  status: torch.Tensor | None = None) -> None:
    """Encode kv [T][Hkv][2][D] fp16 into code_pages [NP][Hkv][P][2][M] uint8 (in place)."""
    _need(kv, torch.float16, "kv", 4)
    _need(token_set, torch.int32, "token_set", 1)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(codebooks, torch.float16, "codebooks", 6)
    _need(code_pages, torch.uint8, "code_pages", 5)
    T, Hkv, _, D = kv.shape
    M = codebooks.shape[3]
    dev = _same_device(kv, token_set=token_set, slot_mapping=slot_mapping, codebooks=codebooks,
                 code_pages=code_pages, status=status)
    cfg = _lib.config(M, head_dim=D, page_size=code_pages.shape[2])
    with torch.cuda.device(dev):
        st = _lib.load().aq_encode_append(
            ctypes.byref(cfg), T, Hkv, _ptr(kv), _ptr(token_set), _ptr(slot_mapping), _ptr(codebooks),
            codebooks.shape[0], _ptr(code_pages), code_pages.shape[0], _ptr(status), _stream(dev))
    _lib.check(st, "aq_encode_append")


def decode_plan(batch: int, num_q_heads: int, num_kv_heads: int, max_seq_len: int,
                num_subspaces: int = 4, num_splits: int = 0, fp16: bool = False):
    """(num_splits, cluster_size, workspace_bytes) a decode call will use."""
    cfg = _lib.config(num_subspaces)
    s, c, w = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    st = _lib.load().aq_decode_plan(ctypes.byref(cfg), batch, num_q_heads, num_kv_heads,
                                    max_seq_len, num_splits, int(fp16), ctypes.byref(s),
                                    ctypes.byref(c), ctypes.byref(w))
    _lib.check(st, "aq_decode_plan")
    return s.value, c.value, w.value


def workspace_for(batch, num_q_heads, num_kv_heads, max_seq_len, num_subspaces=4, num_splits=0,
                  fp16=False, device="cuda"):
    """A device workspace of the size the planned call needs (None when 0)."""
    _, _, w = decode_plan(batch, num_q_heads, num_kv_heads, max_seq_len, num_subspaces,
                          num_splits, fp16)
    return torch.empty(w, dtype=torch.uint8, device=device) if w else None


def decode_attention(q: torch.Tensor, code_pages: torch.Tensor, codebooks: torch.Tensor,
                     req_set: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                     max_seq_len: int, scale: float | None = None, num_splits: int = 0,
                     out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     status: torch.Tensor | None = None) -> torch.Tensor:
    """PQ decode attention; returns out [B][Hq][D] fp32."""
    _need(q, torch.float32, "q", 3)
    _need(code_pages, torch.uint8, "code_pages", 5)
    _need(codebooks, torch.float16, "codebooks", 6)
    _need(req_set, torch.int32, "req_set", 1)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    Hkv, M = codebooks.shape[1], codebooks.shape[3]
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = workspace_for(B, Hq, Hkv, max_seq_len, M, num_splits, device=q.device)
    dev = _same_device(q, code_pages=code_pages, codebooks=codebooks, req_set=req_set, block_table=block_table,
                 seq_lens=seq_lens, out=out, workspace=workspace, status=status)
    cfg = _lib.config(M, head_dim=D, page_size=code_pages.shape[2])
    with torch.cuda.device(dev):
        st = _lib.load().aq_decode_attention(
            ctypes.byref(cfg), B, Hq, Hkv, _ptr(q), _ptr(code_pages), code_pages.shape[0],
            _ptr(codebooks), codebooks.shape[0], _ptr(req_set), _ptr(block_table), block_table.shape[1],
            _ptr(seq_lens), max_seq_len, float(scale), num_splits, _ptr(out), _ptr(workspace),
            workspace.numel() if workspace is not None else 0, _ptr(status), _stream(dev))
    _lib.check(st, "aq_decode_attention")
    return out


def decode_step(q: torch.Tensor, kv_new: torch.Tensor, code_pages: torch.Tensor,
                codebooks: torch.Tensor, req_set: torch.Tensor, block_table: torch.Tensor,
                seq_lens: torch.Tensor, max_seq_len: int, scale: float | None = None,
                num_splits: int = 0, overlap: bool = False, out: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None,
                status: torch.Tensor | None = None) -> torch.Tensor:
    """Fused decode step: append kv_new [B][Hkv][2][D] fp16 (the token at
    position seq_lens[b]-1) to code_pages, then PQ decode attention over all
    seq_lens[b] tokens; returns out [B][Hq][D] fp32.  Codebooks are fp16, or
    uint8 FP8 E4M3 codes (to_e4m3) for half the codebook bytes."""
    _need(q, torch.float32, "q", 3)
    _need(kv_new, torch.float16, "kv_new", 4)
    _need(code_pages, torch.uint8, "code_pages", 5)
    e4m3 = codebooks.dtype == torch.uint8
    _need(codebooks, torch.uint8 if e4m3 else torch.float16, "codebooks", 6)
    _need(req_set, torch.int32, "req_set", 1)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    Hkv, M = codebooks.shape[1], codebooks.shape[3]
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = workspace_for(B, Hq, Hkv, max_seq_len, M, num_splits, device=q.device)
    dev = _same_device(q, kv_new=kv_new, code_pages=code_pages, codebooks=codebooks, req_set=req_set,
                 block_table=block_table, seq_lens=seq_lens, out=out, workspace=workspace, status=status)
    cfg = _lib.config(M, head_dim=D, page_size=code_pages.shape[2])
    with torch.cuda.device(dev):
        st = _lib.load().aq_decode_step(
            ctypes.byref(cfg), B, Hq, Hkv, _ptr(q), _ptr(kv_new), _ptr(code_pages), code_pages.shape[0],
            _ptr(codebooks), codebooks.shape[0], _ptr(req_set), _ptr(block_table), block_table.shape[1],
            _ptr(seq_lens), max_seq_len, float(scale), num_splits,
            (_lib.STEP_OVERLAP if overlap else 0) | (_lib.STEP_E4M3 if e4m3 else 0),
            _ptr(out), _ptr(workspace), workspace.numel() if workspace is not None else 0, _ptr(status),
            _stream(dev))
    _lib.check(st, "aq_decode_step")
    return out


def decode_step_mixed(q: torch.Tensor, kv_new: torch.Tensor, num_fp16_heads: int,
                      kv_pages_f16: torch.Tensor | None, code_pages: torch.Tensor | None,
                      codebooks: torch.Tensor | None, req_set: torch.Tensor | None,
                      block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                      num_subspaces: int = 4, scale: float | None = None, overlap: bool = False,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                      status: torch.Tensor | None = None) -> torch.Tensor:
    """Mixed-precision decode step: kv heads [0, num_fp16_heads) append their
    new K/V to the fp16 cache kv_pages_f16 [NP16][n16][2][P][D] and attend over
    it, the other kv heads take the fused PQ step over code_pages / codebooks
    (pools of Hkv - n16 heads); returns out [B][Hq][D] fp32."""
    _need(q, torch.float32, "q", 3)
    _need(kv_new, torch.float16, "kv_new", 4)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    Hkv = kv_new.shape[1]
    n16 = int(num_fp16_heads)
    e4m3 = False
    if n16 > 0:
        _need(kv_pages_f16, torch.float16, "kv_pages_f16", 5)
    if n16 < Hkv:
        _need(code_pages, torch.uint8, "code_pages", 5)
        e4m3 = codebooks is not None and codebooks.dtype == torch.uint8
        _need(codebooks, torch.uint8 if e4m3 else torch.float16, "codebooks", 6)
        _need(req_set, torch.int32, "req_set", 1)
        num_subspaces = codebooks.shape[3]
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    cfg = _lib.config(num_subspaces, head_dim=D)
    if workspace is None:
        w = ctypes.c_size_t()
        st = _lib.load().aq_decode_step_mixed_workspace(ctypes.byref(cfg), B, Hq, Hkv, n16, max_seq_len,
                                                        ctypes.byref(w))
        _lib.check(st, "aq_decode_step_mixed_workspace")
        workspace = torch.empty(w.value, dtype=torch.uint8, device=q.device) if w.value else None
    dev = _same_device(q, kv_new=kv_new, kv_pages_f16=kv_pages_f16, code_pages=code_pages, codebooks=codebooks,
                 req_set=req_set, block_table=block_table, seq_lens=seq_lens, out=out, workspace=workspace,
                 status=status)
    with torch.cuda.device(dev):
        st = _lib.load().aq_decode_step_mixed(
            ctypes.byref(cfg), B, Hq, Hkv, n16, _ptr(q), _ptr(kv_new), _ptr(kv_pages_f16),
            kv_pages_f16.shape[0] if kv_pages_f16 is not None else 0, _ptr(code_pages),
            code_pages.shape[0] if code_pages is not None else 0, _ptr(codebooks),
            codebooks.shape[0] if codebooks is not None else 0, _ptr(req_set), _ptr(block_table),
            block_table.shape[1], _ptr(seq_lens), max_seq_len, float(scale),
            (_lib.STEP_OVERLAP if overlap else 0) | (_lib.STEP_E4M3 if e4m3 else 0), _ptr(out),
            _ptr(workspace), workspace.numel() if workspace is not None else 0, _ptr(status), _stream(dev))
    _lib.check(st, "aq_decode_step_mixed")
    return out


def decode_attention_fp16(q: torch.Tensor, kv_pages: torch.Tensor, block_table: torch.Tensor,
                          seq_lens: torch.Tensor, max_seq_len: int, scale: float | None = None,
                          num_splits: int = 0, out: torch.Tensor | None = None,
                          workspace: torch.Tensor | None = None,
                          status: torch.Tensor | None = None) -> torch.Tensor:
    """fp16-cache decode attention (the comparison point); kv_pages [NP][Hkv][2][P][D]."""
    _need(q, torch.float32, "q", 3)
    _need(kv_pages, torch.float16, "kv_pages", 5)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    Hkv = kv_pages.shape[1]
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = workspace_for(B, Hq, Hkv, max_seq_len, 4, num_splits, fp16=True, device=q.device)
    dev = _same_device(q, kv_pages=kv_pages, block_table=block_table, seq_lens=seq_lens, out=out,
                 workspace=workspace, status=status)
    cfg = _lib.config(4, head_dim=D, page_size=kv_pages.shape[3])
    with torch.cuda.device(dev):
        st = _lib.load().aq_decode_attention_fp16(
            ctypes.byref(cfg), B, Hq, Hkv, _ptr(q), _ptr(kv_pages), kv_pages.shape[0],
            _ptr(block_table), block_table.shape[1], _ptr(seq_lens), max_seq_len, float(scale),
            num_splits, _ptr(out), _ptr(workspace), workspace.numel() if workspace is not None else 0,
            _ptr(status), _stream(dev))
    _lib.check(st, "aq_decode_attention_fp16")
    return out


class DecodeStep:
    """One decode step of a fixed batch: append each request's current K/V
    token (the one at position seq_len-1) into the PQ code cache, then PQ
    decode attention over the cache, as one aq_decode_step launch.

    Holds the cache tensors, the workspace, the output and a device status
    word.  `run(q, new_kv)` launches the step on the current stream.
    `capture_host(q_host, kv_host, out_host)` records the whole step -- copies
    of the pinned host inputs to the device, the step, the copy of the output
    back to pinned host memory -- into a CUDA graph; `replay()` launches it and,
    with wait=True, blocks until the output is on the host.  `launch()` /
    `wait()` split that in two, so that a caller keeping two sets of pinned
    buffers can launch step i before it waits for step i-1's output (the copies
    and the kernel of one step overlap the host's work on the other).
    `overlap=True` launches the step as a programmatic dependent of the
    preceding kernel (aq_decode_step's AQ_STEP_OVERLAP contract).
    """

    def __init__(self, code_pages, codebooks, req_set, block_table, seq_lens, max_seq_len,
                 new_slot, new_set, num_q_heads, scale=None, num_splits=0, overlap=False):
        self.code_pages, self.codebooks = code_pages, codebooks
        self.req_set, self.block_table, self.seq_lens = req_set, block_table, seq_lens
        self.max_seq_len = int(max_seq_len)
        self.new_slot, self.new_set = new_slot, new_set
        self.B, self.Hq = int(seq_lens.shape[0]), int(num_q_heads)
        self.Hkv, self.M = int(codebooks.shape[1]), int(codebooks.shape[3])
        self.scale = scale
        self.num_splits = num_splits
        dev = code_pages.device
        self.workspace = workspace_for(self.B, self.Hq, self.Hkv, self.max_seq_len, self.M,
                                       num_splits, device=dev)
        self.status = new_status(dev)
        self.out = torch.empty((self.B, self.Hq, HEAD_DIM), dtype=torch.float32, device=dev)
        self.graph = None
        self._host = None
        self._done = None
        self._io = None
        self.overlap = overlap

    def run(self, q, new_kv, out=None):
        return decode_step(q, new_kv, self.code_pages, self.codebooks, self.req_set,
                           self.block_table, self.seq_lens, self.max_seq_len, self.scale,
                           self.num_splits, overlap=self.overlap, out=self.out if out is None else out,
                           workspace=self.workspace, status=self.status)

    def pinned_io(self):
        """(q_host, kv_host, out_host): pinned host views of one input buffer
        (q [B][Hq][D] fp32 then the new K/V [B][Hkv][2][D] fp16) and an output
        buffer [B][Hq][D] fp32, for capture_host() without arguments: the inputs
        then reach the device in one copy."""
        if self._io is None:
            nq = self.B * self.Hq * HEAD_DIM * 4
            nkv = self.B * self.Hkv * 2 * HEAD_DIM * 2
            buf = torch.empty(nq + nkv, dtype=torch.uint8).pin_memory()
            q = buf[:nq].view(torch.float32).view(self.B, self.Hq, HEAD_DIM)
            kv = buf[nq:].view(torch.float16).view(self.B, self.Hkv, 2, HEAD_DIM)
            out = torch.empty((self.B, self.Hq, HEAD_DIM), dtype=torch.float32).pin_memory()
            self._io = (buf, q, kv, out)
        return self._io[1:]

    def capture_host(self, q_host=None, kv_host=None, out_host=None):
        """Capture copy-in, step, copy-out into a CUDA graph (pinned host
        tensors; none given: this object's pinned_io(), copied in one piece)."""
        dev = self.out.device
        if q_host is None:
            self.pinned_io()
            buf, q_host, kv_host, out_host = self._io
            buf_d = torch.empty(buf.shape, dtype=buf.dtype, device=dev)
            nq = q_host.numel() * 4
            q_d = buf_d[:nq].view(torch.float32).view(q_host.shape)
            kv_d = buf_d[nq:].view(torch.float16).view(kv_host.shape)
            copies = [(buf_d, buf)]
        else:
            for t, n in ((q_host, "q_host"), (kv_host, "kv_host"), (out_host, "out_host")):
                if t.is_cuda or not t.is_pinned():
                    raise ValueError(f"{n} must be a pinned host tensor")
            q_d = torch.empty(q_host.shape, dtype=q_host.dtype, device=dev)
            kv_d = torch.empty(kv_host.shape, dtype=kv_host.dtype, device=dev)
            copies = [(q_d, q_host), (kv_d, kv_host)]
        self._host = (q_host, kv_host, out_host, q_d, kv_d, copies)
        # one eager run sets kernel attributes outside the capture
        for d, h in copies:
            d.copy_(h)
        self.run(q_d, kv_d)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for d, h in copies:
                d.copy_(h, non_blocking=True)
            self.run(q_d, kv_d)
            out_host.copy_(self.out, non_blocking=True)
        self.graph = g
        return g

    def replay(self, wait=True):
        self.graph.replay()
        if wait:
            torch.cuda.current_stream().synchronize()

    def launch(self):
        """Replay the captured step on the current stream without waiting
        (replays on different streams may overlap: use distinct caches)."""
        self.graph.replay()
        if self._done is None:
            self._done = torch.cuda.Event()
        self._done.record()

    def wait(self):
        """Block until the last launch()'s output is in pinned host memory."""
        self._done.synchronize()

    def check_status(self):
        """Raise if a kernel flagged a data error (reads the status word)."""
        st = int(self.status.item())
        if st:
            raise RuntimeError(f"device status {st:#x}")


class HostDecodeStep:
    """aq_decode_step_host for a fixed batch and cache: one C call per step
    enqueues the copy of the query and the new K/V from pinned host memory, the
    fused step and the copy of the output back to pinned host memory, on
    `stream` (a torch.cuda.Stream; the current one if None).

    `q_host`, `kv_host`, `out_host` are the pinned tensors (write the next
    step's inputs into the first two, read the output from the last one after
    `sync()`); `launch()` enqueues one step.  The call's arguments are
    marshalled once, here; `launch()` itself does no device switch, so the
    cache's device must be the current one when it is called.
    """

    def __init__(self, code_pages, codebooks, req_set, block_table, seq_lens, max_seq_len,
                 num_q_heads, scale=None, num_splits=0, stream=None):
        _need(code_pages, torch.uint8, "code_pages", 5)
        e4m3 = codebooks.dtype == torch.uint8
        _need(codebooks, torch.uint8 if e4m3 else torch.float16, "codebooks", 6)
        for t, n in ((req_set, "req_set"), (seq_lens, "seq_lens")):
            _need(t, torch.int32, n, 1)
        _need(block_table, torch.int32, "block_table", 2)
        self.B, self.Hq = int(seq_lens.shape[0]), int(num_q_heads)
        self.Hkv, self.M = int(codebooks.shape[1]), int(codebooks.shape[3])
        dev = code_pages.device
        _same_device(code_pages, codebooks=codebooks, req_set=req_set, block_table=block_table,
                     seq_lens=seq_lens)
        self.stream = stream or torch.cuda.current_stream(dev)
        self.q_host = torch.empty((self.B, self.Hq, HEAD_DIM), dtype=torch.float32).pin_memory()
        self.kv_host = torch.empty((self.B, self.Hkv, 2, HEAD_DIM), dtype=torch.float16).pin_memory()
        self.out_host = torch.empty((self.B, self.Hq, HEAD_DIM), dtype=torch.float32).pin_memory()
        lib = _lib.load()
        n = lib.aq_decode_step_host_staging(self.B, self.Hq, self.Hkv)
        self.staging = torch.empty(n, dtype=torch.uint8, device=dev)
        self.workspace = workspace_for(self.B, self.Hq, self.Hkv, int(max_seq_len), self.M, num_splits,
                                       device=dev)
        self.status = new_status(dev)
        self._keep = (code_pages, codebooks, req_set, block_table, seq_lens)
        self._cfg = _lib.config(self.M, page_size=code_pages.shape[2])
        scale = HEAD_DIM ** -0.5 if scale is None else scale
        self._fn = lib.aq_decode_step_host
        self._args = (ctypes.byref(self._cfg), self.B, self.Hq, self.Hkv, _ptr(self.q_host), _ptr(self.kv_host),
                      _ptr(code_pages), code_pages.shape[0], _ptr(codebooks), codebooks.shape[0], _ptr(req_set),
                      _ptr(block_table), block_table.shape[1], _ptr(seq_lens), int(max_seq_len), float(scale),
                      num_splits, _lib.STEP_E4M3 if e4m3 else 0, _ptr(self.out_host), _ptr(self.staging),
                      self.staging.numel(), _ptr(self.workspace),
                      self.workspace.numel() if self.workspace is not None else 0, _ptr(self.status),
                      ctypes.c_void_p(self.stream.cuda_stream))

    def launch(self):
        """Enqueue one step (copies in, step, copy out) on the stream."""
        st = self._fn(*self._args)
        if st != _lib.AQ_OK:
            _lib.check(st, "aq_decode_step_host")

    def sync(self):
        """Wait until the last launched step's output is in out_host."""
        self.stream.synchronize()

    def check_status(self):
        """Raise if a kernel flagged a data error (reads the status word)."""
        st = int(self.status.item())
        if st:
            raise RuntimeError(f"device status {st:#x}")
