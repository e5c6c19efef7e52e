"""Multi-rank logic on CPU ranks (gloo, world size 2): bench.py's maximum of
the timed region over ranks and weak-scaling job value, and split-KV across
ranks (page-range shards whose (max, sum, output) partials are all-gathered and
merged) against single-pass attention."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "took" 10 * (r + 1) ms; the job time is the slowest rank's
        t = bench.max_over_ranks(10.0 * (rank + 1))
        v = bench.job_value(units_per_rank=1000, steps=5, seconds=t / 1e3, world=world)
        q.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, t, v in res:
        assert t == 20.0                       # max over ranks, seen by every rank
        assert v == pytest.approx(2 * 1000 * 5 / 0.020)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_value(10, 2, 0.5, 1) == 40.0


# --------------------------------------------------------------------------
# split-KV across ranks (CPU emulation): each rank attends over its page range
# of every request and keeps the (max, sum, unnormalised output) partials; the
# partials are all-gathered and merged by the rule the combine kernel applies
# (PAM article §2.2.3: statistics of blocks merged by a reduction).  With
# world 2 the result must equal single-pass attention over the whole request.
# --------------------------------------------------------------------------
def _shard_partials(orc, p, rank, world, scale):
    import numpy as np
    q = p["q"].astype(np.float64)
    B, Hq, D = q.shape
    cp, cbs, bt = p["code_pages"], p["codebooks"].astype(np.float64), p["block_table"]
    Hkv = cbs.shape[1]
    G = Hq // Hkv
    part = np.zeros((B, Hq, D + 2), np.float64)
    for b, L in enumerate(p["seq_lens"]):
        t0, t1 = int(L) * rank // world, int(L) * (rank + 1) // world
        for h in range(Hq):
            kvh = h // G
            if t1 <= t0:
                part[b, h, D] = -np.inf                # empty shard: no statistics
                continue
            t = np.arange(t0, t1)
            codes = cp[bt[b, t // 16], kvh, t % 16]     # [T][2][M]
            cb = cbs[p["req_set"][b], kvh]               # [2][M][K][Dsub]
            k = orc.pq_reconstruct(cb[0], codes[:, 0])
            v = orc.pq_reconstruct(cb[1], codes[:, 1])
            s = scale * (k @ q[b, h])
            m = s.max()
            w = np.exp(s - m)
            part[b, h, :D] = w @ v
            part[b, h, D], part[b, h, D + 1] = m, w.sum()
    return part


def _merge(parts):
    import numpy as np
    D = parts.shape[-1] - 2
    m, l, o = parts[..., D], parts[..., D + 1], parts[..., :D]
    M = np.where(l > 0, m, -np.inf).max(axis=0)
    f = np.where(l > 0, np.exp(m - M), 0.0)
    return (f[..., None] * o).sum(axis=0) / (f * l).sum(axis=0)[..., None]


def _shard_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import numpy as np
    import oracle
    import workloads as W
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = W.paged_codes_problem(17, 3, 4, 2, 4, [300, 77, 1], num_sets=3)
        scale = 1.0 / np.sqrt(128)
        mine = torch.from_numpy(_shard_partials(oracle, p, rank, world, scale))
        gathered = [torch.zeros_like(mine) for _ in range(world)]
        dist.all_gather(gathered, mine)
        merged = _merge(np.stack([g.numpy() for g in gathered]))
        want = oracle.decode_attention(p["q"], p["code_pages"], p["codebooks"], p["req_set"],
                                       p["block_table"], p["seq_lens"], scale, 16)
        q.put((rank, float(np.abs(merged - want).max())))
    finally:
        dist.destroy_process_group()


def test_split_kv_across_ranks_merges_to_single_pass():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, err in res:
        assert err < 1e-12, (rank, err)


def test_reference_arm_prints_once_under_torchrun():
    """bench.py --impl reference launched as the multi-GPU bench is (torchrun,
    2 ranks on 127.0.0.1): rank 0 alone times the oracle and prints one JSON
    line with the reference arm's keys; the other rank exits 0 without work.
    No GPU is touched."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--workload", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "3", "--cpu-budget", "0.2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["dtype"] == "f64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("tiny")
