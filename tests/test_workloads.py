"""The seeded input generators follow the recipes they state (CPU only).

These pin the synthetic inputs themselves -- the shapes, the ragged length mix,
the paging, the Gaussian-mixture draw, the outlier channels and the
regeneration of any slice from its own keyed generator -- so that the parity
tests and the benchmark run on the workloads the documentation describes.
"""
import numpy as np
import pytest

import workloads as W

SHAPES = {
    # name: (batch, Hq, Hkv, M, lens, layers)
    "tiny": (1, 2, 2, 4, {512}, 1),
    "page1": (4, 32, 32, 4, {2048}, 1),
    "qwen_gqa": (8, 64, 8, 4, {1000}, 80),
    "long": (1, 32, 32, 8, {131072}, 1),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_shapes_and_seeds(name):
    B, Hq, Hkv, M, lens, layers = SHAPES[name]
    w = W.make(name)
    assert (w.batch, w.num_q_heads, w.num_kv_heads, w.num_subspaces, w.layers) == (B, Hq, Hkv, M, layers)
    assert set(w.seq_lens.tolist()) == lens and len(w.seq_lens) == B
    assert w.seed == W.SEED_BASE + W.NAMES.index(name)
    assert w.head_dim == 128 and w.num_codewords == 256 and w.page_size == 16
    assert w.n_fit == 64 and w.fit_iters == 10
    assert w.scale == pytest.approx(128 ** -0.5)
    q = w.queries()
    assert q.dtype == np.float32 and q.shape == (B, Hq, 128)


def test_ragged_length_mix():
    """256 requests: exactly round(0.3 * 256) = 77 of 4096 tokens, the other
    179 uniform in [64, 512], in shuffled order; pages under a shuffled table."""
    w = W.make("ragged")
    L = w.seq_lens
    assert len(L) == 256 and w.num_kv_heads == 32 and w.num_subspaces == 4 and w.shuffle_pages
    assert int((L == 4096).sum()) == 77
    short = L[L != 4096]
    assert len(short) == 179 and short.min() >= 64 and short.max() <= 512
    assert len(np.unique(short)) > 100                      # spread over the range
    longs = np.flatnonzero(L == 4096)
    assert longs.max() - longs.min() > 150 and not np.all(np.diff(longs) == 1)   # interleaved
    assert 300_000 < int(L.sum()) < 420_000


@pytest.mark.parametrize("name", ["page1", "ragged"])
def test_block_table_is_a_page_permutation(name):
    w = W.make(name)
    bt, npages = w.block_table()
    per = -(-w.seq_lens.astype(np.int64) // 16)
    assert npages == int(per.sum()) and bt.shape == (w.batch, int(per.max()))
    used = np.concatenate([bt[b, :per[b]] for b in range(w.batch)])
    assert np.array_equal(np.sort(used), np.arange(npages))     # every page exactly once
    if w.shuffle_pages:
        assert not np.array_equal(used, np.arange(npages))
    b = int(np.argmax(w.seq_lens))
    s = w.slot_mapping(bt, b, 0, int(w.seq_lens[b]))
    t = np.arange(int(w.seq_lens[b]))
    assert s.dtype == np.int64
    assert np.array_equal(s // 16, bt[b, t // 16]) and np.array_equal(s % 16, t % 16)


def test_slices_regenerate_from_their_own_generators():
    """A slice crossing a 4096-token chunk boundary equals the same tokens of
    the full draw; another request or layer gives different vectors."""
    w = W.make("long", seq_lens=[9000], num_kv_heads=2, num_q_heads=2)
    full = w.kv(0)
    assert full.shape == (9000, 2, 2, 128) and full.dtype == np.float16
    assert np.array_equal(w.kv(0, 0, 4000, 8300), full[4000:8300])
    assert np.array_equal(w.kv(0, 0, 8190, 9000, threads=2), full[8190:])
    assert not np.array_equal(w.kv(0, 1, 0, 64), full[:64])
    again = W.make("long", seq_lens=[9000], num_kv_heads=2, num_q_heads=2)
    assert np.array_equal(again.kv(0, 0, 0, 100), full[:100])
    assert np.array_equal(w.fit_samples(full), full[:64].transpose(1, 2, 0, 3))


def test_long_has_two_outlier_channels_per_head():
    """Per (kv head, K or V): channel scales in [0.5, 2] except exactly two,
    which are 10x (so in [5, 20])."""
    w = W.make("long")
    _, scales = w._mixture_params(0)
    assert scales.shape == (32, 2, 128)
    big = scales > 2.0
    assert np.all(big.sum(axis=2) == 2)
    assert np.all((scales[big] >= 5.0) & (scales[big] <= 20.0))
    assert np.all((scales[~big] >= 0.5) & (scales[~big] <= 2.0))
    assert not np.any(W.make("page1")._mixture_params(0)[1] > 2.0)


def test_mixture_draw_follows_its_recipe():
    """x = s * (c_z + 0.2 eps): divided by the channel scales, every vector
    lies within the 0.2-sigma noise of one of its head's 16 centres."""
    w = W.make("page1", seq_lens=[4096], batch=1, num_kv_heads=2, num_q_heads=2)
    centres, scales = w._mixture_params(0)
    x = w.kv(0).astype(np.float32)                          # [T][H][2][D]
    for h in range(2):
        for kv in range(2):
            u = x[:, h, kv] / scales[h, kv]
            d = ((u[:, None, :] - centres[h, kv][None]) ** 2).sum(-1)   # [T][16]
            z = d.argmin(1)
            resid = u - centres[h, kv][z]
            assert 0.19 < resid.std() < 0.21
            assert abs(resid.mean()) < 0.01
            counts = np.bincount(z, minlength=16)
            assert counts.min() > 4096 / 16 * 0.7            # z uniform over the 16


def test_tiny_recipe_is_codeword_plus_small_noise():
    w = W.make("tiny")
    cbs = w.given_codebooks().astype(np.float32)             # [H][2][M][K][Dsub]
    codes = w.generating_codes(0)                             # [L][H][2][M]
    x = w.kv(0).astype(np.float32).reshape(512, 2, 2, 4, 32)
    hh = np.arange(2)[None, :, None, None]
    ww = np.arange(2)[None, None, :, None]
    mm = np.arange(4)[None, None, None, :]
    noise = x - cbs[hh, ww, mm, codes]
    assert 0.045 < noise.std() < 0.055 and abs(noise.mean()) < 0.005
