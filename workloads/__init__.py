"""Seeded synthetic inputs for PQ decode attention (shared by tests and bench).

This module draws random numbers and lays them out; it holds none of the
method's arithmetic (no fitting, encoding, reconstruction or attention).  Both
the CPU oracle and the CUDA path receive exactly what it returns.

Recipes (one per workload; sizes as named):

* ``tiny``      B=1, 2 heads, D=128, M=4, K=256, L=512.  Codebooks fp16 N(0,1)
                are given; each cached K/V vector is, per subspace, a uniformly
                drawn codeword plus N(0, 0.05^2) noise, stored as fp16.
* ``page1``     B=4, 32 heads, D=128, L=2048, M=4, K=256.  K/V from a 16-cluster
                Gaussian mixture per head (centres N(0,I), sigma 0.2, per-channel
                scale U[0.5,2]); codebooks fitted on the first 64 tokens.
* ``qwen_gqa``  80 layers, B=8, 64 query heads over 8 kv heads, L=1000, M=4.
* ``long``      B=1, 32 heads, L=131072, M=8 (Dsub=16); the mixture has two
                outlier channels per head with 10x scale.
* ``ragged``    256 requests, 32 heads, M=4; 77 requests of 4096 tokens and 179
                of U[64,512] tokens in shuffled order; pages of 16 tokens under a
                shuffled block table; codebooks per request.

Queries are fp32 N(0,1); scale = 1/sqrt(128).  Mixture draw for one vector of
head h:  z ~ U{0..15},  x = s_h * (c_h[z] + 0.2 * eps),  eps ~ N(0, I).
Mixture parameters are per (layer, kv head, K-or-V); samples are per request,
drawn from a generator keyed by (seed, layer, request), so any request can be
regenerated alone.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HEAD_DIM = 128
CODEWORDS = 256
PAGE = 16
N_FIT = 64
FIT_ITERS = 10
SEED_BASE = 1234
CHUNK = 4096       # tokens per independently keyed draw


def _rng(*key):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    num_subspaces: int
    seq_lens: np.ndarray          # int32 [B]
    seed: int
    layers: int = 1
    head_dim: int = HEAD_DIM
    num_codewords: int = CODEWORDS
    page_size: int = PAGE
    n_fit: int = N_FIT
    fit_iters: int = FIT_ITERS
    outlier_channels: int = 0
    shuffle_pages: bool = False
    mixture: bool = True          # False: the tiny codeword+noise recipe

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def dsub(self) -> int:
        return self.head_dim // self.num_subspaces

    @property
    def max_pages(self) -> int:
        return int(-(-int(self.seq_lens.max()) // self.page_size))

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.sum())

    # -- queries ---------------------------------------------------------
    def queries(self, layer: int = 0) -> np.ndarray:
        """fp32 [B][Hq][D], N(0,1)."""
        g = _rng(self.seed, layer, 0x51)
        return g.standard_normal((self.batch, self.num_q_heads, self.head_dim),
                                 dtype=np.float32)

    # -- paging ----------------------------------------------------------
    def block_table(self):
        """(block_table int32 [B][max_pages], num_pages).

        Pages are numbered densely over all requests; with shuffle_pages the
        physical page ids are a random permutation.  Unused table entries are 0.
        """
        pages_per = [-(-int(L) // self.page_size) for L in self.seq_lens]
        num_pages = int(sum(pages_per))
        perm = np.arange(num_pages, dtype=np.int32)
        if self.shuffle_pages:
            perm = _rng(self.seed, 0x7ab1e).permutation(num_pages).astype(np.int32)
        bt = np.zeros((self.batch, self.max_pages), np.int32)
        nxt = 0
        for b, n in enumerate(pages_per):
            bt[b, :n] = perm[nxt:nxt + n]
            nxt += n
        return bt, num_pages

    def slot_mapping(self, block_table: np.ndarray, b: int, t0: int, t1: int) -> np.ndarray:
        """int64 page*P + slot for tokens [t0, t1) of request b."""
        t = np.arange(t0, t1)
        return (block_table[b, t // self.page_size].astype(np.int64) * self.page_size
                + t % self.page_size)

    # -- raw cache vectors ----------------------------------------------
    def _mixture_params(self, layer: int):
        g = _rng(self.seed, layer, 0x313)
        H, D = self.num_kv_heads, self.head_dim
        centres = g.standard_normal((H, 2, 16, D), dtype=np.float32)
        scales = g.uniform(0.5, 2.0, size=(H, 2, D)).astype(np.float32)
        if self.outlier_channels:
            for h in range(H):
                for w in range(2):
                    ch = g.choice(D, size=self.outlier_channels, replace=False)
                    scales[h, w, ch] *= 10.0
        return centres, scales

    def given_codebooks(self) -> np.ndarray:
        """Tiny recipe only: fp16 N(0,1) codebooks [Hkv][2][M][K][Dsub]."""
        g = _rng(self.seed, 0, 0xcb)
        return g.standard_normal(
            (self.num_kv_heads, 2, self.num_subspaces, self.num_codewords, self.dsub),
            dtype=np.float32).astype(np.float16)

    def _kv_chunk(self, b: int, layer: int, c: int) -> np.ndarray:
        """Tokens [c*CHUNK, min((c+1)*CHUNK, L)) of request b, fp16 [T][Hkv][2][D]."""
        L = int(self.seq_lens[b])
        n = min(CHUNK, L - c * CHUNK)
        g = _rng(self.seed, layer, 0x4b56, b, c)
        H, D = self.num_kv_heads, self.head_dim
        if not self.mixture:
            M, K = self.num_subspaces, self.num_codewords
            cbs = self.given_codebooks().astype(np.float32)       # [H][2][M][K][Dsub]
            pick = g.integers(0, K, size=(n, H, 2, M))
            noise = g.standard_normal((n, H, 2, D), dtype=np.float32) * np.float32(0.05)
            hh = np.arange(H)[None, :, None, None]
            ww = np.arange(2)[None, None, :, None]
            mm = np.arange(M)[None, None, None, :]
            words = cbs[hh, ww, mm, pick]                          # [n][H][2][M][Dsub]
            return (words.reshape(n, H, 2, D) + noise).astype(np.float16)
        centres, scales = self._mixture_params(layer)
        z = g.integers(0, 16, size=(n, H, 2))
        x = g.standard_normal((n, H, 2, D), dtype=np.float32)       # eps
        x *= np.float32(0.2)
        rows = (np.arange(H * 2).reshape(1, H, 2) * 16 + z).reshape(-1)
        x += np.take(centres.reshape(H * 2 * 16, D), rows, axis=0).reshape(n, H, 2, D)
        x *= scales[None]
        return x.astype(np.float16)

    def kv(self, b: int, layer: int = 0, t0: int = 0, t1: int | None = None,
           threads: int = 1) -> np.ndarray:
        """Raw fp16 K/V of request b, tokens [t0, t1): [T][Hkv][2][D].

        Tokens are drawn in fixed chunks of CHUNK, each from its own keyed
        generator, so a slice equals the same tokens of a full draw.
        """
        L = int(self.seq_lens[b])
        t1 = L if t1 is None else min(t1, L)
        if t1 <= t0:
            return np.zeros((0, self.num_kv_heads, 2, self.head_dim), np.float16)
        c0, c1 = t0 // CHUNK, (t1 - 1) // CHUNK + 1
        if threads > 1 and c1 - c0 > 1:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                parts = list(ex.map(lambda c: self._kv_chunk(b, layer, c), range(c0, c1)))
        else:
            parts = [self._kv_chunk(b, layer, c) for c in range(c0, c1)]
        x = np.concatenate(parts) if len(parts) > 1 else parts[0]
        return x[t0 - c0 * CHUNK: t1 - c0 * CHUNK]

    def generating_codes(self, b: int) -> np.ndarray:
        """Tiny recipe only: the codeword indices drawn for request b [L][H][2][M]."""
        assert not self.mixture
        L = int(self.seq_lens[b])
        out = []
        for c in range(-(-L // CHUNK)):
            n = min(CHUNK, L - c * CHUNK)
            g = _rng(self.seed, 0, 0x4b56, b, c)
            out.append(g.integers(0, self.num_codewords,
                                  size=(n, self.num_kv_heads, 2, self.num_subspaces)))
        return np.concatenate(out)

    def kv_all(self, layer: int = 0, threads: int = 8):
        """Every request's K/V, drawn in parallel: list of [L_b][Hkv][2][D]."""
        if self.batch == 1:
            return [self.kv(0, layer, threads=threads)]
        with ThreadPoolExecutor(max_workers=threads) as ex:
            return list(ex.map(lambda b: self.kv(b, layer), range(self.batch)))

    def fit_samples(self, kv_b: np.ndarray) -> np.ndarray:
        """The first n_fit tokens of one request, per kv head and K/V:
        [Hkv][2][N][D] (a view/copy, no arithmetic)."""
        n = min(self.n_fit, kv_b.shape[0])
        return np.ascontiguousarray(kv_b[:n].transpose(1, 2, 0, 3))


def _ragged_lens(seed: int, n: int = 256) -> np.ndarray:
    g = _rng(seed, 0x1e5)
    n_long = int(round(0.3 * n))
    lens = np.concatenate([np.full(n_long, 4096),
                           g.integers(64, 513, size=n - n_long)])
    return g.permutation(lens).astype(np.int32)


def make(name: str, seed: int | None = None, **overrides) -> Workload:
    """The named workload (seed defaults to 1234 + its index)."""
    idx = {"tiny": 0, "page1": 1, "qwen_gqa": 2, "long": 3, "ragged": 4}[name]
    seed = SEED_BASE + idx if seed is None else seed
    if name == "tiny":
        w = Workload(name, 1, 2, 2, 4, np.array([512], np.int32), seed, mixture=False)
    elif name == "page1":
        w = Workload(name, 4, 32, 32, 4, np.full(4, 2048, np.int32), seed)
    elif name == "qwen_gqa":
        w = Workload(name, 8, 64, 8, 4, np.full(8, 1000, np.int32), seed, layers=80)
    elif name == "long":
        w = Workload(name, 1, 32, 32, 8, np.array([131072], np.int32), seed,
                     outlier_channels=2)
    elif name == "ragged":
        w = Workload(name, 256, 32, 32, 4, _ragged_lens(seed), seed, shuffle_pages=True)
    else:  # pragma: no cover
        raise KeyError(name)
    for k, v in overrides.items():
        if k == "seq_lens":
            v = np.asarray(v, np.int32)
        setattr(w, k, v)
    if "seq_lens" in overrides:
        w.batch = len(w.seq_lens)
    return w


NAMES = ("tiny", "page1", "qwen_gqa", "long", "ragged")


def paged_codes_problem(seed: int, batch: int, num_q_heads: int, num_kv_heads: int,
                        num_subspaces: int, seq_lens, num_sets: int | None = None,
                        shuffle: bool = True, extra_pages: int = 3, page_size: int = PAGE,
                        head_dim: int = HEAD_DIM, num_codewords: int = CODEWORDS) -> dict:
    """Random inputs for the decode step alone: fp16 N(0,1) codebooks, uniform
    uint8 codes in every page slot, fp32 N(0,1) queries, a (shuffled) block
    table with `extra_pages` unused pages in the pool, and a random request ->
    codebook-set map.  Returns numpy arrays keyed by argument name."""
    g = _rng(seed, 0x9a9ed)
    lens = np.asarray(seq_lens, np.int32)
    assert len(lens) == batch
    S = num_sets or batch
    M, Dsub = num_subspaces, head_dim // num_subspaces
    codebooks = g.standard_normal((S, num_kv_heads, 2, M, num_codewords, Dsub),
                                  dtype=np.float32).astype(np.float16)
    pages_per = [-(-int(L) // page_size) for L in lens]
    num_pages = int(sum(pages_per)) + extra_pages
    perm = g.permutation(num_pages) if shuffle else np.arange(num_pages)
    max_pages = max(1, max(pages_per) if pages_per else 1)
    bt = np.zeros((batch, max_pages), np.int32)
    nxt = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[nxt:nxt + n]
        nxt += n
    code_pages = g.integers(0, num_codewords, size=(num_pages, num_kv_heads, page_size, 2, M),
                            dtype=np.uint8)
    req_set = g.integers(0, S, size=batch).astype(np.int32)
    q = g.standard_normal((batch, num_q_heads, head_dim), dtype=np.float32)
    return {"q": q, "code_pages": code_pages, "codebooks": codebooks, "req_set": req_set,
            "block_table": bt, "seq_lens": lens, "num_pages": num_pages}


def paged_fp16_problem(seed: int, batch: int, num_q_heads: int, num_kv_heads: int, seq_lens,
                       shuffle: bool = True, extra_pages: int = 3, page_size: int = PAGE,
                       head_dim: int = HEAD_DIM) -> dict:
    """Random fp16 K/V pages [NP][Hkv][2][P][D] (N(0,1)), queries and a block table."""
    g = _rng(seed, 0xf16)
    lens = np.asarray(seq_lens, np.int32)
    pages_per = [-(-int(L) // page_size) for L in lens]
    num_pages = int(sum(pages_per)) + extra_pages
    perm = g.permutation(num_pages) if shuffle else np.arange(num_pages)
    max_pages = max(1, max(pages_per) if pages_per else 1)
    bt = np.zeros((batch, max_pages), np.int32)
    nxt = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[nxt:nxt + n]
        nxt += n
    kv_pages = g.standard_normal((num_pages, num_kv_heads, 2, page_size, head_dim),
                                 dtype=np.float32).astype(np.float16)
    q = g.standard_normal((batch, num_q_heads, head_dim), dtype=np.float32)
    return {"q": q, "kv_pages": kv_pages, "block_table": bt, "seq_lens": lens,
            "num_pages": num_pages}
