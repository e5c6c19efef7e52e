"""Benchmark: PQ-KV decode attention on one GB300 (or N, one process each).

One step = one decode step of the batch: append the current token of every
request into the PQ code cache (encode against the request's codebooks), then
PQ decode attention over the L cached tokens of every request, kv head and
query head.  The cache (codebooks fitted on the first 64 tokens, all L tokens
encoded) is built once before timing, as a serving system does at prefill.

Printed: one JSON line (rank 0).  `value` = KV tokens x kv heads attended per
second over the whole job (device-timed, inputs resident in HBM, L2 defeated
by rotating through input copies larger than twice the L2); `e2e` = the same
through the public API with pinned host buffers, copies in the timed region
and the host waiting for every step's output; `roofline` = the decode kernel's
algorithmic bytes per launch over its event-timed duration against the measured
HBM copy bandwidth; `cpu_baseline` = the CPU oracle on a bounded sample.

  python bench.py [--steps K] [--warmup W] [--workload page1|ragged|long|qwen_gqa|tiny]
  python bench.py --impl reference      # the CPU oracle arm
  torchrun --nproc-per-node N bench.py --gpus N   # weak scaling, one process per GPU
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import signal
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "PQ-KV decode attention: KV tokens·heads/s; code-stream GB/s as % of HBM peak"
UNIT = "KV tokens*heads/s"


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (the job finishes with its slowest
    rank); x itself when torch.distributed is not initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    if device is None:
        device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: int, steps: int, seconds: float, world: int) -> float:
    """Whole-job throughput under weak scaling: every rank processes the same
    per-GPU workload, the job takes the slowest rank's time."""
    return world * units_per_rank * steps / seconds


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense fp16/bf16 tensor-core peak (TFLOP/s, burst) and where it came from."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def measure_prefill(w, api, torch, base, hbm_peak):
    """Warm timings of the cache build: the codebook fit on each request's
    first tokens and the tensor-core encode of every prefill token (the same
    inputs build_cache used), and of one periodic codebook refresh.  The encode reads each K/V vector once and forms
    its dot products with all 256 codewords of every subspace on the tensor
    cores (2 x 128 x 256 FLOP per vector), so both bounds are reported."""
    kvs, bt = base["kvs"], base["bt_np"]
    Hkv, M = w.num_kv_heads, w.num_subspaces
    kv = torch.from_numpy(np.concatenate(kvs)).cuda()
    tset = torch.from_numpy(np.concatenate([np.full(len(k), b, np.int32) for b, k in enumerate(kvs)])).cuda()
    slots = torch.from_numpy(np.concatenate([w.slot_mapping(bt, b, 0, len(k)) for b, k in enumerate(kvs)])).cuda()
    samples = np.stack([w.fit_samples(k) for k in kvs])
    samples_d = torch.from_numpy(samples.reshape(-1, *samples.shape[3:])).cuda()
    pages = torch.zeros_like(base["pages"])
    st = api.new_status()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def timed(fn, reps=5):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    enc_ms = timed(lambda: api.encode_append(kv, tset, slots, base["codebooks"], pages, st))
    fit_ms = timed(lambda: api.fit_codebooks(samples_d, M, w.fit_iters))
    # periodic refresh (every 64 generated tokens): 3 Lloyd steps on the 64 most
    # recent vectors of every unit, in place on a copy of the codebooks
    recent = np.stack([w.fit_samples(k[-64:]) for k in kvs])
    recent_d = torch.from_numpy(recent.reshape(-1, *recent.shape[3:])).cuda()
    cb_copy = base["codebooks"].reshape(-1, M, 256, w.dsub).clone()
    refresh_ms = timed(lambda: api.refine_codebooks(recent_d, cb_copy, 3))
    assert int(st.item()) == 0 and torch.equal(pages, base["pages"])
    T = kv.shape[0]
    vecs = T * Hkv * 2
    s = enc_ms / 1e3
    tf_peak, tf_kind = measured_tensor_peak()
    gbs = vecs * 128 * 2 / s / 1e9
    tflops = vecs * 2 * 128 * 256 / s / 1e12
    return {"fit_ms": fit_ms, "fit_units": int(samples_d.shape[0]), "fit_iters": w.fit_iters,
            "refresh_ms": refresh_ms, "refresh": "3 Lloyd steps on each unit's 64 most recent vectors",
            "encode_ms": enc_ms, "encode_tokens": T,
            "encode_vectors_per_s": vecs / s,
            "encode_kv_read": {"gbs": gbs, "frac": gbs / hbm_peak},
            "encode_mma": {"tflops": tflops, "frac": tflops / tf_peak, "peak_kind": tf_kind},
            "encode_kernel": "encode_mma_kernel (tcgen05)",
            "cold_first_call_ms": {"fit": base["fit_ms"], "encode": base["encode_prefill_ms"]}}


def measured_traffic(workload: str, mode: str):
    """DRAM bytes (read + write) per launch of the decode kernel from one ncu
    capture, recorded in profiles/traffic.json with the SHA-256 of the kernel
    source it was taken on; None when there is no capture for this workload
    and mode or the kernel source has changed since."""
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tp):
        return None
    with open(tp) as f:
        e = json.load(f).get(f"{workload}/{mode}")
    if not e:
        return None
    src = os.path.join(ROOT, "decode_attention_product_gb300", "csrc", "decode_pq.cu")
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    return float(e["dram_bytes"]) if e.get("decode_pq_sha256") == digest else None


def step_kernel_name(group: int, subspaces: int) -> str:
    """The decode kernel the library's planner picks for a fused step: for at
    least 4 query heads per kv head (and no AQPQ_DECODE_KERNEL override asking
    for the other) the whole-split design on clusters of one subspace per CTA --
    the head-split kernel when the group covers the cluster, else the
    whole-split kernel -- otherwise the token-share kernel."""
    forced = os.environ.get("AQPQ_DECODE_KERNEL", "")
    if forced == "2" or (forced != "1" and group >= 4):
        name = "pq_headsplit_kernel" if group >= 4 and group >= subspaces else "pq_attend_kernel"
    else:
        name = "pq_decode_kernel"
    return name + " (fused step)"


def workload_desc(w) -> str:
    return (f"{w.name}: B{w.batch} Hq{w.num_q_heads} Hkv{w.num_kv_heads} D{w.head_dim} "
            f"M{w.num_subspaces} K{w.num_codewords} L{int(w.seq_lens.max())}"
            + (f" ({w.total_tokens} tokens, ragged)" if w.name == "ragged" else "")
            + (f" x{w.layers} layers" if w.layers > 1 else ""))


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return parse_clock_samples(lines)


def parse_clock_samples(lines):
    """The clocks object of the JSON line from `nvidia-smi --query-gpu=<Q>
    --format=csv,noheader,nounits` rows: the median SM clock, the largest
    maximum clock, and every throttle reason that was Active in any sample."""
    rows = []
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) >= 9:
            rows.append(parts)
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
    smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
    return {"sm_mhz": float(np.median(sm)) if sm else None,
            "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
            "samples": len(rows)}


# --------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline leg and --impl reference)
# --------------------------------------------------------------------------
class OracleStep:
    """The oracle's decode step (append one token per request, then decode
    attention over all heads), request by request on the host cores.  The
    per-request cache (oracle codebook fit + prefill encode) is built once,
    untimed, for `n_req` requests; `run(budget_s)` cycles over them until the
    timed work reaches the budget."""

    def __init__(self, w, n_req: int = 4, layer: int = 0):
        import oracle
        oracle.build()
        self.oracle, self.w = oracle, w
        self.q = w.queries(layer)
        M, Hkv = w.num_subspaces, w.num_kv_heads
        self.reqs = []
        for b in range(min(n_req, w.batch)):
            L = int(w.seq_lens[b])
            kv = w.kv(b, layer, 0, L)
            samples = w.fit_samples(kv)
            cb16, _, _, _ = oracle.kmeans_fit(samples.reshape(-1, *samples.shape[2:]), M, 256,
                                              w.fit_iters)
            cbs = cb16.reshape(1, Hkv, 2, M, 256, w.dsub)
            npg = -(-L // 16)
            pages = np.zeros((npg, Hkv, 16, 2, M), np.uint8)
            slots = np.arange(L, dtype=np.int64)
            oracle.encode_append(kv[:L - 1], np.zeros(L - 1, np.int32), slots[:L - 1], cbs, pages, 16)
            self.reqs.append((b, L, kv[L - 1:L].copy(), cbs, pages,
                              np.arange(npg, dtype=np.int32)[None]))

    def run(self, budget_s: float):
        o, w = self.oracle, self.w
        units, elapsed, n = 0, 0.0, 0
        while elapsed < budget_s:
            b, L, kv_new, cbs, pages, bt = self.reqs[n % len(self.reqs)]
            t0 = time.perf_counter()
            o.encode_append(kv_new, np.zeros(1, np.int32), np.array([L - 1], np.int64), cbs, pages, 16)
            o.decode_attention(self.q[b:b + 1], pages, cbs, np.zeros(1, np.int32), bt,
                               np.array([L], np.int32), w.scale, 16)
            elapsed += time.perf_counter() - t0
            units += L * w.num_kv_heads
            n += 1
        return units, elapsed, n

    def describe(self, n):
        return (f"{n} request-steps of {self.w.name} cycling over its first {len(self.reqs)} "
                f"requests (append 1 token + decode attention, all heads)")


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    ost = OracleStep(w)
    # each step a bounded sample, the whole run within about two minutes
    # (--cpu-budget caps a step's sample too: short runs for tests)
    budget = min(4.0, 120.0 / (args.steps + args.warmup), args.cpu_budget)
    units = secs = n_tot = 0
    for i in range(args.warmup + args.steps):
        u, s_, n = ost.run(budget)
        if i >= args.warmup:
            units, secs, n_tot = units + u, secs + s_, n_tot + n
    v = units / secs
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(w)},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": ost.oracle.num_threads(),
                             "kind": "oracle", "sample": ost.describe(n_tot)},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
def build_cache(w, api, torch, layer=0):
    """Fit codebooks (GPU) on each request's first 64 tokens and encode all L
    tokens into pages (GPU).  Returns device tensors and the new-token K/V."""
    Hkv, M = w.num_kv_heads, w.num_subspaces
    kvs = w.kv_all(layer, threads=16)
    samples = np.stack([w.fit_samples(k) for k in kvs])                 # [B][Hkv][2][N][D]
    samples_d = torch.from_numpy(samples.reshape(-1, *samples.shape[3:])).cuda()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    cbs = api.fit_codebooks(samples_d, M, w.fit_iters)
    t1.record()
    torch.cuda.synchronize()
    fit_ms = t0.elapsed_time(t1)
    cbs = cbs.view(w.batch, Hkv, 2, M, 256, w.dsub)
    bt, npages = w.block_table()
    kv = np.concatenate(kvs)
    tset = np.concatenate([np.full(len(k), b, np.int32) for b, k in enumerate(kvs)])
    slots = np.concatenate([w.slot_mapping(bt, b, 0, len(k)) for b, k in enumerate(kvs)])
    pages = torch.zeros((npages, Hkv, 16, 2, M), dtype=torch.uint8, device="cuda")
    st = api.new_status()
    kv_d = torch.from_numpy(kv).cuda()
    t0.record()
    api.encode_append(kv_d, torch.from_numpy(tset).cuda(), torch.from_numpy(slots).cuda(), cbs,
                      pages, st)
    t1.record()
    torch.cuda.synchronize()
    enc_ms = t0.elapsed_time(t1)
    assert int(st.item()) == 0
    # the decode step's "current token": the last cached token of each request
    last = np.stack([k[-1] for k in kvs])                                # [B][Hkv][2][D]
    last_slot = np.array([w.slot_mapping(bt, b, len(k) - 1, len(k))[0] for b, k in enumerate(kvs)],
                         np.int64)
    del kv_d, samples_d
    return {"codebooks": cbs, "pages": pages, "bt": torch.from_numpy(bt).cuda(),
            "seq_lens": torch.from_numpy(w.seq_lens).cuda(),
            "req_set": torch.arange(w.batch, dtype=torch.int32, device="cuda"),
            "q": torch.from_numpy(w.queries(layer)).cuda(),
            "new_kv": torch.from_numpy(last).cuda(), "new_slot": torch.from_numpy(last_slot).cuda(),
            "new_set": torch.arange(w.batch, dtype=torch.int32, device="cuda"),
            "fit_ms": fit_ms, "encode_prefill_ms": enc_ms, "npages": npages, "bt_np": bt,
            "kvs": kvs}


MIN_REGION_MS = 200.0     # every timed region lasts at least this long


def time_steps(torch, step, R, steps, dist=False, min_region_ms=None, clocks=None):
    """Device time per step of a rotation of steps, replayed from CUDA graphs.

    `step(i)` launches step i, which uses input copy i % R.  One graph holds R
    consecutive steps (copies 0..R-1) and one the tail of the timed count, so
    consecutive steps always use different copies.  The timed region runs
    `reps` x `steps` steps, reps chosen so that the region lasts at least
    `min_region_ms`; a lead-in replay is enqueued before the start event, so
    the GPU is already busy when the region starts and the host's graph-launch
    latency stays outside it.  CUDA events on the launching stream; barrier and
    synchronize on both sides.  Returns (ms per step, steps timed, region ms).
    """
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                step(i)
        return g

    if min_region_ms is None:
        min_region_ms = MIN_REGION_MS
    g_cycle = capture(R)
    g_cycle.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    g_cycle.replay()
    e0.record()
    g_cycle.replay()
    g_cycle.replay()
    e1.record()
    torch.cuda.synchronize()
    est = e0.elapsed_time(e1) / (2 * R)
    reps = max(1, math.ceil(min_region_ms / max(steps * est, 1e-6)))
    total = steps * reps
    n_cyc, tail = divmod(total, R)
    g_tail = capture(tail) if tail else None
    torch.cuda.synchronize()
    if dist:
        torch.distributed.barrier()
    if clocks is not None:
        clocks.start()
    torch.cuda.synchronize()
    if dist:
        torch.distributed.barrier()
    g_cycle.replay()                                   # lead-in, not timed
    e0.record()
    for _ in range(n_cyc):
        g_cycle.replay()
    if g_tail is not None:
        g_tail.replay()
    e1.record()
    torch.cuda.synchronize()
    if dist:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks is not None else None
    region = e0.elapsed_time(e1)
    return region / total, total, region, clk


def rotation(base, torch, l2, keys=("codebooks", "pages", "q", "new_kv")):
    """Input copies for rotation: enough that R consecutive steps read more than
    2 x L2, so every timed step reads cold codebooks and codes."""
    per_copy = sum(base[k].numel() * base[k].element_size() for k in keys)
    R = max(2, min(64, math.ceil(2.2 * l2 / per_copy)))
    copies = [base] + [{k: (v.clone() if torch.is_tensor(v) and k in keys else v)
                        for k, v in base.items()} for _ in range(R - 1)]
    return copies, R, per_copy


def measure_fused_step(args, w, api, torch, T, base, local_rank, dist, world, e4m3=True):
    """The fused decode step of workload w (aq_decode_step, launched as a
    programmatic dependent of the previous step, which wrote another copy):
    device time per step, roofline of the step kernel, clocks during the
    timed region; plus the same step with E4M3 codebooks."""
    M, Hq, Hkv = w.num_subspaces, w.num_q_heads, w.num_kv_heads
    Lmax = int(w.seq_lens.max())
    l2 = torch.cuda.get_device_properties(local_rank).L2_cache_size
    copies, R, per_copy = rotation(base, torch, l2)
    splits, cluster, wsb = api.decode_plan(w.batch, Hq, Hkv, Lmax, M)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    outs = [torch.empty((w.batch, Hq, 128), dtype=torch.float32, device="cuda") for _ in range(R)]
    status = api.new_status()

    def step(i):
        c = copies[i % R]
        api.decode_step(c["q"], c["new_kv"], c["pages"], c["codebooks"], c["req_set"], c["bt"],
                        c["seq_lens"], Lmax, w.scale, overlap=True, out=outs[i % R], workspace=ws,
                        status=status)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ms, n_timed, region, clk = time_steps(torch, step, R, args.steps, dist, clocks=ClockSampler(local_rank))
    ms = max_over_ranks(ms)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    units = T.kv_tokens_heads(w.seq_lens, Hkv)
    byt = T.pq_step_bytes(w.seq_lens, Hq, Hkv, M)
    peak, peak_kind = measured_peaks()
    achieved = byt["total"] / (ms / 1e3) / 1e9
    out = {
        "workload": workload_desc(w), "ms_per_step": ms, "steps_timed": n_timed, "region_ms": region,
        "value": job_value(units, 1, ms / 1e3, world), "unit": UNIT,
        "plan": {"splits": splits, "cluster": cluster},
        "l2": f"rotating {R} input copies of {per_copy / 1e6:.1f} MB "
              f"({R * per_copy / 1e6:.0f} MB > 2 x L2 {l2 / 1e6:.0f} MB)",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": measured_traffic(w.name, "step"),
                     "kernel": step_kernel_name(Hq // Hkv, M), "bytes_per_launch": byt["total"],
                     "launch_ms": ms, "peak_kind": peak_kind},
        "code_stream": {"gbs": byt["code_stream"] / (ms / 1e3) / 1e9,
                        "codes_only_gbs": byt["codes"] / (ms / 1e3) / 1e9,
                        "frac_of_peak": byt["code_stream"] / (ms / 1e3) / 1e9 / peak},
        "clocks": clk,
        "launches_per_step": 1 + (1 if splits > 1 else 0),
    }
    del copies, outs
    if e4m3:
        out["e4m3_codebooks"] = measure_e4m3(args, w, api, torch, base, Lmax, units, T, local_rank)
    return out


def run_ours(args, w, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    from decode_attention_product_gb300 import api, build as B, traffic as T
    if rank == 0 or world == 1:
        B.build()
    if world > 1:
        torch.distributed.barrier()
        B.build()
    dist = world > 1
    Lmax = int(w.seq_lens.max())
    base = build_cache(w, api, torch)
    M, Hq, Hkv = w.num_subspaces, w.num_q_heads, w.num_kv_heads
    units = T.kv_tokens_heads(w.seq_lens, Hkv)
    peak, peak_kind = measured_peaks()
    splits, cluster, wsb = api.decode_plan(w.batch, Hq, Hkv, Lmax, M)
    if not args.two_call:
        main = measure_fused_step(args, w, api, torch, T, base, local_rank, dist, world)
        ms, n_timed = main["ms_per_step"], main["steps_timed"]
        roof = dict(main["roofline"], timing=(
            f"one fused kernel per step: CUDA events around graph replays of {n_timed} steps "
            f"({args.steps} x {n_timed // args.steps}, region {main['region_ms']:.0f} ms, lead-in "
            f"replay enqueued first), divided by the steps run"))
        launches = n_timed * main["launches_per_step"]
        clk = main["clocks"]
    else:
        # two launches per step (append, then decode attention): the step is
        # timed as a whole, the decode launch alone from a decode-only rotation
        l2 = torch.cuda.get_device_properties(local_rank).L2_cache_size
        copies, R, per_copy = rotation(base, torch, l2)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
        outs = [torch.empty((w.batch, Hq, 128), dtype=torch.float32, device="cuda") for _ in range(R)]
        status = api.new_status()

        def step(i):
            c = copies[i % R]
            api.encode_append(c["new_kv"], c["new_set"], c["new_slot"], c["codebooks"], c["pages"], status)
            api.decode_attention(c["q"], c["pages"], c["codebooks"], c["req_set"], c["bt"],
                                 c["seq_lens"], Lmax, w.scale, out=outs[i % R], workspace=ws, status=status)

        def dec(i):
            c = copies[i % R]
            api.decode_attention(c["q"], c["pages"], c["codebooks"], c["req_set"], c["bt"],
                                 c["seq_lens"], Lmax, w.scale, out=outs[i % R], workspace=ws, status=status)

        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        ms, n_timed, region, clk = time_steps(torch, step, R, args.steps, dist,
                                              clocks=ClockSampler(local_rank))
        ms = max_over_ranks(ms)
        dec_ms, _, _, _ = time_steps(torch, dec, R, args.steps, dist)
        assert int(status.item()) == 0, f"device status {int(status.item())}"
        byt = T.pq_decode_bytes(w.seq_lens, Hq, Hkv, M)
        achieved = byt["total"] / (dec_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": measured_traffic(w.name, "two_call"), "kernel": "pq_decode_kernel",
                "bytes_per_launch": byt["total"], "launch_ms": dec_ms, "peak_kind": peak_kind,
                "timing": "decode-only rotation of graph replays (CUDA events, lead-in replay first)"}
        main = {"code_stream": {"gbs": byt["code_stream"] / (dec_ms / 1e3) / 1e9,
                                "codes_only_gbs": byt["codes"] / (dec_ms / 1e3) / 1e9,
                                "frac_of_peak": byt["code_stream"] / (dec_ms / 1e3) / 1e9 / peak},
                "l2": f"rotating {R} input copies of {per_copy / 1e6:.1f} MB"}
        launches = n_timed * (2 + (1 if splits > 1 else 0))
        del copies, outs
    value = job_value(units, 1, ms / 1e3, world)
    # e2e through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
        e2e = measure_e2e(args, w, api, torch, base, Lmax, ws, units, world, dist)
    prefill = measure_prefill(w, api, torch, base, peak)
    # fp16 comparison kernel on the same shape (cache of the same raw vectors)
    fp16 = None if args.no_fp16 else measure_fp16(args, w, api, torch, base, Lmax, units, T)
    sweep = (measure_layer_sweep(args, w, api, torch, base, Lmax, T)
             if w.layers > 1 and not args.two_call and not args.no_sweep else None)
    mixed = (measure_mixed(args, w, api, torch, T, base, max(1, w.num_kv_heads // 8), local_rank)
             if not args.two_call else None)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "steps_timed": n_timed, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(w), "batch": w.batch, "seq_len": Lmax,
                   "num_q_heads": Hq, "num_kv_heads": Hkv, "num_subspaces": M,
                   "num_codewords": w.num_codewords, "plan": {"splits": splits, "cluster": cluster},
                   "l2": main["l2"],
                   "step": ("append 1 token/request (encode) + PQ decode attention, two launches"
                            if args.two_call else
                            "fused launch: append 1 token/request + PQ decode attention "
                            "(aq_decode_step, programmatic dependent launch)")},
        "roofline": roof,
        "code_stream": main["code_stream"],
        "gpu_launches": launches,
        "clocks": clk,
        "prefill": prefill,
    }
    if e2e:
        line["e2e"] = e2e
    if fp16:
        line["fp16_comparison"] = fp16
    if "e4m3_codebooks" in main:
        line["e4m3_codebooks"] = main["e4m3_codebooks"]
    if sweep:
        line["layer_sweep"] = sweep
    if mixed:
        line["mixed_precision"] = mixed
    if args.two_call:
        line["append"] = {"us_per_step": (ms - roof["launch_ms"]) * 1e3,
                          "how": "step time minus the decode launch's time"}
    del base
    torch.cuda.empty_cache()
    # the other workloads' fused steps, each timed the same way
    if not args.two_call and not args.no_extras and w.name == "page1":
        extra = {}
        for name in ("ragged", "long", "qwen_gqa"):
            wx = W.make(name)
            bx = build_cache(wx, api, torch)
            ex = measure_fused_step(args, wx, api, torch, T, bx, local_rank, dist, world)
            ex.pop("launches_per_step")
            if wx.layers > 1 and not args.no_sweep:
                ex["layer_sweep"] = measure_layer_sweep(args, wx, api, torch, bx, int(wx.seq_lens.max()), T)
            extra[name] = ex
            del bx
            torch.cuda.empty_cache()
        line["workloads"] = extra
    if rank == 0 and not args.no_cpu:
        ost = OracleStep(w)
        units_c, secs_c, n_c = ost.run(args.cpu_budget)
        cores = ost.oracle.num_threads()
        # the same oracle on one thread, a third of the budget
        ost.oracle.set_num_threads(1)
        units_1, secs_1, n_1 = ost.run(args.cpu_budget / 3)
        ost.oracle.set_num_threads(cores)
        line["cpu_baseline"] = {"value": units_c / secs_c, "unit": UNIT,
                                "cores": cores, "kind": "oracle",
                                "sample": ost.describe(n_c) + f", {secs_c:.1f} s",
                                "value_1_thread": units_1 / secs_1,
                                "sample_1_thread": ost.describe(n_1) + f", {secs_1:.1f} s",
                                "host_cpus": os.cpu_count()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_e2e(args, w, api, torch, base, Lmax, ws, units, world, dist):
    """Through the C-ABI call with host buffers (aq_decode_step_host, wrapped by
    api.HostDecodeStep): every step moves its q and new K/V in from pinned host
    memory, runs the fused step and moves its output back, and the host reads
    each step's output.  Steps alternate between two streams, each with its own
    pinned buffers, so the host enqueues step i before it waits for (and
    reads) step i-1; they rotate over cache copies larger than 2 x L2, as the
    device-timed steps do."""
    Hq = w.num_q_heads
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    copies, R, _ = rotation(base, torch, l2)
    R += R % 2                                           # an even rotation: stream i % 2 owns copy i
    while len(copies) < R:
        copies.append({k: (v.clone() if torch.is_tensor(v) and k in ("codebooks", "pages", "q", "new_kv") else v)
                       for k, v in base.items()})
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    q0 = torch.from_numpy(w.queries())
    kv0 = base["new_kv"].cpu()
    steps = []
    for i in range(R):
        c = copies[i]
        hs = api.HostDecodeStep(c["pages"], c["codebooks"], c["req_set"], c["bt"], c["seq_lens"], Lmax, Hq,
                                w.scale, stream=streams[i % 2])
        hs.q_host.copy_(q0)
        hs.kv_host.copy_(kv0)
        hs.out_np = hs.out_host.numpy()
        steps.append(hs)
    torch.cuda.synchronize()
    check = 0.0

    def run(n):
        nonlocal check
        prev = None
        for i in range(n):
            hs = steps[i % R]
            hs.launch()
            if prev is not None:
                prev.sync()
                check += prev.out_np[0, 0, 0]            # the host reads the result
            prev = hs
        prev.sync()
        check += prev.out_np[0, 0, 0]

    run(max(3, args.warmup) * 2)
    t0 = time.perf_counter()
    run(2 * R)
    est = (time.perf_counter() - t0) / (2 * R)
    n = max(args.steps, 2 * math.ceil(MIN_REGION_MS / 1e3 / max(est, 1e-7) / 2))
    if dist:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    run(n)
    secs = time.perf_counter() - t0
    for hs in steps:
        hs.check_status()
    secs = max_over_ranks(secs)
    assert math.isfinite(check)
    q_h, kv_h, out_h = steps[0].q_host, steps[0].kv_host, steps[0].out_host
    del steps, copies
    return {"value": job_value(units, n, secs, world), "unit": UNIT,
            "h2d_bytes_per_step": q_h.numel() * 4 + kv_h.numel() * 2,
            "d2h_bytes_per_step": out_h.numel() * 4, "ms_per_step": 1e3 * secs / n, "steps_timed": n,
            "how": "aq_decode_step_host per step (pinned buffers: a gather kernel reads q and the new K/V from "
                   "host memory, the fused step writes its output into host memory), over rotated cache copies, "
                   "alternating two streams; step i enqueued before the host waits for and reads step i-1"}


def measure_fp16(args, w, api, torch, base, Lmax, units, T):
    """The uncompressed comparison: fp16 pages of the same raw vectors, timed
    like the PQ step (graph replays over rotated copies larger than 2 x L2)."""
    Hq, Hkv = w.num_q_heads, w.num_kv_heads
    kvs = base["kvs"]
    bt = base["bt_np"]
    npages = base["npages"]
    pages = torch.zeros((npages, Hkv, 2, 16, 128), dtype=torch.float16, device="cuda")
    for b, k in enumerate(kvs):
        L = len(k)
        pad = (-L) % 16
        kk = np.concatenate([k, np.zeros((pad, Hkv, 2, 128), np.float16)]) if pad else k
        blk = kk.reshape(-1, 16, Hkv, 2, 128).transpose(0, 2, 3, 1, 4)   # [pg][Hkv][2][16][D]
        idx = torch.from_numpy(bt[b, :blk.shape[0]].astype(np.int64)).cuda()
        pages[idx] = torch.from_numpy(np.ascontiguousarray(blk)).cuda()
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    per = pages.numel() * 2
    R = max(2, min(8, math.ceil(2.2 * l2 / per)))
    pcs = [pages] + [pages.clone() for _ in range(R - 1)]
    splits, _, wsb = api.decode_plan(w.batch, Hq, Hkv, Lmax, fp16=True)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty((w.batch, Hq, 128), dtype=torch.float32, device="cuda")

    def step(i):
        api.decode_attention_fp16(base["q"], pcs[i % R], base["bt"], base["seq_lens"], Lmax, w.scale,
                                  out=out, workspace=ws)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    ms, n_timed, _, _ = time_steps(torch, step, R, args.steps)
    byt = T.fp16_decode_bytes(w.seq_lens, Hq, Hkv)
    peak, _ = measured_peaks()
    del pcs, pages
    return {"value": units / (ms / 1e3), "unit": UNIT, "ms_per_call": ms, "steps_timed": n_timed,
            "gbs": byt["total"] / (ms / 1e3) / 1e9, "frac_of_peak": byt["total"] / (ms / 1e3) / 1e9 / peak,
            "splits": splits}


def measure_layer_sweep(args, w, api, torch, base0, Lmax, T):
    """A multi-layer stack (the 80-layer GQA workload): one fused decode step
    per layer, each on that layer's own cache (its codebooks fitted and its
    tokens encoded from that layer's vectors), run back to back as one sweep.
    Timed eagerly (one launch per layer from Python) and as one captured CUDA
    graph; the caches of all layers together exceed L2, so each step reads
    cold codebooks and codes."""
    Hq, Hkv, M = w.num_q_heads, w.num_kv_heads, w.num_subspaces
    keep = ("q", "new_kv", "pages", "codebooks", "req_set", "bt", "seq_lens")
    layers = [{k: base0[k] for k in keep}]
    for layer in range(1, w.layers):
        c = build_cache(w, api, torch, layer=layer)
        layers.append({k: c[k] for k in keep})
        del c
    splits, cluster, wsb = api.decode_plan(w.batch, Hq, Hkv, Lmax, M)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty((w.batch, Hq, 128), dtype=torch.float32, device="cuda")
    st = api.new_status()

    def sweep():
        # consecutive steps touch different layers' caches: overlapped launches
        # keep the early-read contract
        for c in layers:
            api.decode_step(c["q"], c["new_kv"], c["pages"], c["codebooks"], c["req_set"], c["bt"],
                            c["seq_lens"], Lmax, w.scale, overlap=True, out=out, workspace=ws, status=st)

    for _ in range(3):
        sweep()
    torch.cuda.synchronize()
    n = 20
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        sweep()
    e1.record()
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / n
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sweep()
    g.replay()
    torch.cuda.synchronize()
    # graph replays over a region of >= MIN_REGION_MS, a lead-in replay first
    n = max(5, math.ceil(MIN_REGION_MS / max(eager_ms, 1e-3)))
    g.replay()
    e0.record()
    for _ in range(n):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    graph_ms = e0.elapsed_time(e1) / n
    assert int(st.item()) == 0
    byt = T.pq_step_bytes(w.seq_lens, Hq, Hkv, M)["total"] * w.layers
    units = T.kv_tokens_heads(w.seq_lens, Hkv) * w.layers
    peak, _ = measured_peaks()
    del layers
    return {"layers": w.layers, "eager_ms_per_sweep": eager_ms, "graph_ms_per_sweep": graph_ms,
            "us_per_layer": graph_ms * 1e3 / w.layers, "value": units / (graph_ms / 1e3), "unit": UNIT,
            "gbs": byt / (graph_ms / 1e3) / 1e9, "frac_of_peak": byt / (graph_ms / 1e3) / 1e9 / peak,
            "plan": {"splits": splits, "cluster": cluster}}


def measure_mixed(args, w, api, torch, T, base, n16, local_rank=0):
    """The mixed-precision step (AQPIM blog §6.1 item 4): kv heads [0, n16)
    keep fp16 pages of the same raw vectors, the others the PQ cache; one
    aq_decode_step_mixed per step (the PQ step, then the fp16 heads' append +
    attention as its programmatic dependent; a combine per part that splits),
    timed like the main step over rotated copies larger than 2 x L2."""
    Hq, Hkv, M = w.num_q_heads, w.num_kv_heads, w.num_subspaces
    G = Hq // Hkv
    Lmax = int(w.seq_lens.max())
    bt, npages = base["bt_np"], base["npages"]
    kvp = np.zeros((npages, n16, 2, 16, 128), np.float16)
    for b, k in enumerate(base["kvs"]):
        t = np.arange(len(k))
        kvp[bt[b, t // 16], :, :, t % 16] = k[:, :n16]
    mb = dict(base, codebooks=base["codebooks"][:, n16:].contiguous(), pages=base["pages"][:, n16:].contiguous(),
              kvp=torch.from_numpy(kvp).cuda())
    l2 = torch.cuda.get_device_properties(local_rank).L2_cache_size
    copies, R, per_copy = rotation(mb, torch, l2, keys=("codebooks", "pages", "q", "new_kv", "kvp"))
    out = torch.empty((w.batch, Hq, 128), dtype=torch.float32, device="cuda")
    st = api.new_status()
    w_b = ctypes_workspace(api, w, n16, Lmax, torch)

    def step(i):
        c = copies[i % R]
        api.decode_step_mixed(c["q"], c["new_kv"], n16, c["kvp"], c["pages"], c["codebooks"], c["req_set"], c["bt"],
                              c["seq_lens"], Lmax, num_subspaces=M, scale=w.scale, overlap=True, out=out,
                              workspace=w_b, status=st)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    ms, n_timed, _, _ = time_steps(torch, step, R, args.steps)
    assert int(st.item()) == 0
    pq = T.pq_step_bytes(w.seq_lens, (Hkv - n16) * G, Hkv - n16, M)["total"]
    f16 = T.fp16_decode_bytes(w.seq_lens, n16 * G, n16)
    f16_total = f16["total"] - f16["q"] - f16["out"] + 2 * w.batch * n16 * 2 * 128 * 2   # q/out counted once; the append
    byt = pq + f16_total
    peak, _ = measured_peaks()
    s16 = api.decode_plan(w.batch, n16 * G, n16, Lmax, fp16=True)[0]
    spq = api.decode_plan(w.batch, (Hkv - n16) * G, Hkv - n16, Lmax, M)[0]
    launches = 2 + (s16 > 1) + (spq > 1)
    del copies, mb
    return {"fp16_kv_heads": n16, "pq_kv_heads": Hkv - n16, "ms_per_step": ms, "steps_timed": n_timed,
            "bytes_per_step": byt, "gbs": byt / (ms / 1e3) / 1e9, "frac_of_peak": byt / (ms / 1e3) / 1e9 / peak,
            "value": T.kv_tokens_heads(w.seq_lens, Hkv) / (ms / 1e3), "unit": UNIT,
            "launches_per_step": launches, "l2": f"rotating {R} input copies of {per_copy / 1e6:.1f} MB"}


def ctypes_workspace(api, w, n16, Lmax, torch):
    """The mixed step's workspace (None when it needs none)."""
    import ctypes
    from decode_attention_product_gb300 import _lib
    cfg = _lib.config(w.num_subspaces)
    n = ctypes.c_size_t()
    _lib.check(_lib.load().aq_decode_step_mixed_workspace(ctypes.byref(cfg), w.batch, w.num_q_heads, w.num_kv_heads,
                                                          n16, Lmax, ctypes.byref(n)), "workspace")
    return torch.empty(n.value, dtype=torch.uint8, device="cuda") if n.value else None


def measure_e4m3(args, w, api, torch, base, Lmax, units, T, local_rank=0):
    """The fused step with the same codebooks stored as FP8 E4M3 codes (half
    the codebook bytes; AQPIM blog §4.2), timed like the main step: graph
    replays over rotated copies of codebooks and pages larger than 2 x L2."""
    Hq, Hkv, M = w.num_q_heads, w.num_kv_heads, w.num_subspaces
    # its own pages too: the steps write the new tokens' codes, which differ
    # from the fp16 codebooks' codes where rounding moved a codeword
    b8 = dict(base, codebooks=api.to_e4m3(base["codebooks"]), pages=base["pages"].clone())
    l2 = torch.cuda.get_device_properties(local_rank).L2_cache_size
    copies, R, _ = rotation(b8, torch, l2)
    splits, _, wsb = api.decode_plan(w.batch, Hq, Hkv, Lmax, M)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty((w.batch, Hq, 128), dtype=torch.float32, device="cuda")
    st = api.new_status()

    def step(i):
        c = copies[i % R]
        api.decode_step(c["q"], c["new_kv"], c["pages"], c["codebooks"], c["req_set"], c["bt"],
                        c["seq_lens"], Lmax, w.scale, overlap=True, out=out, workspace=ws, status=st)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    ms, n_timed, _, _ = time_steps(torch, step, R, args.steps)
    assert int(st.item()) == 0
    byt = T.pq_step_bytes_e4m3(w.seq_lens, Hq, Hkv, M)
    peak, _ = measured_peaks()
    del copies, b8
    return {"value": units / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps_timed": n_timed,
            "bytes_per_step": byt["total"],
            "gbs": byt["total"] / (ms / 1e3) / 1e9, "frac_of_peak": byt["total"] / (ms / 1e3) / 1e9 / peak,
            "codebooks": "FP8 E4M3 (same codebooks, rounded to nearest even)"}


def main():
    global MIN_REGION_MS
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="page1", choices=list(W.NAMES))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-fp16", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="page1 only: skip the ragged, long and qwen_gqa step objects")
    ap.add_argument("--two-call", action="store_true",
                    help="time aq_encode_append + aq_decode_attention instead of the fused step")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for cpu_baseline; also caps each step of --impl reference")
    ap.add_argument("--no-sweep", action="store_true", help="qwen_gqa: skip the 80-layer sweep")
    ap.add_argument("--min-region-ms", type=float, default=200.0,
                    help="shortest timed region (repeats of the K steps); lower only for profiler runs")
    args = ap.parse_args()
    MIN_REGION_MS = args.min_region_ms
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = W.make(args.workload)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
