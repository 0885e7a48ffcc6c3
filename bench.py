"""Benchmark of the lightning-indexer hot path on GB300.

One step = one idx_score_topk call (q preparation, the tcgen05 scoring kernel,
then the selection kernel) over the batched-decode workload: T=64 queries, H=64 heads, D=128,
valid lengths uniform in [8192, 32768], 64-entry blocks, per-query block tables
over a 40000-block NVFP4 pool, top_k=512. Inputs are seeded and synthetic and
resident in HBM when timing starts; L2 is flushed (a 256 MB write) before
every timed step, outside the timed events.

Prints one JSON line: scored (query, key) pairs per second (whole job), the
device-timed value, an end-to-end value through the public API with host
buffers (pinned H2D of the step's q, w, block table and valid lengths; D2H of
the top-k indices and scores), the roofline of the scoring kernel against the
measured HBM copy bandwidth, and the float64 CPU oracle timed on a bounded
sample of the same workload.

--impl reference times that oracle alone (the CPU reference arm).
--gpus N (under torchrun): every rank runs its own batch (weak scaling); the
timed region is bracketed by a barrier and synchronisation and the slowest
rank's time is used.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "indexer (query,key) scores+top-k per sec; % of HBM / tensor-core roofline"
UNIT = "pairs/s"
BYTES_PER_PAIR = 64 + 8 + 4.0 / 64 + 4.0 / 64     # nibbles + E4M3 scales + gscale + table entry

# name -> (generator name in workloads, base seed, valid-length description, table description)
WORKLOADS = {
    "batched_decode": ("batched_decode", 1001, "valid_lens~U[8192,32768]", "per-query block tables"),
    "long_decode": ("long_decode", 1002, "valid_lens=262144", "per-query block tables"),
    "prefill": ("prefill", 1003, "valid_lens=(r+28672)//4", "one shared block table"),
}


def make_workload(name: str, seed: int):
    from sparse_attention_top_paged_gb300 import workloads
    return getattr(workloads, WORKLOADS[name][0])(seed)


def workload_config(W):
    _, _, lens, table = WORKLOADS[W.name]
    return {
        "workload": f"{W.name}: T={W.T} H={W.H} D={W.D} {lens} epb={W.epb} "
                    f"P={W.P} top_k={W.top_k} NVFP4 keys, {table}",
        "T": W.T, "H": W.H, "D": W.D, "entries_per_block": W.epb, "pool_blocks": W.P,
        "top_k": W.top_k, "pairs_per_step": W.pairs,
        "l2": "flushed before every timed step (256 MB write, outside the timed events)",
        "seed": W.meta.get("seed"),
    }


def rank_seed(name: str, rank: int) -> int:
    """Each rank scores its own batch (weak scaling): the workload's seed + rank."""
    return WORKLOADS[name][1] + rank


def whole_job(pairs_per_rank, steps: int, seconds_per_rank, dist=None, device=None):
    """Whole-job throughput: all ranks' pairs over the slowest rank's time.

    With ``dist`` the per-rank pair counts are summed and the times maxed
    across the process group; returns ``(pairs_per_second, max_seconds)``."""
    if dist is None:
        return pairs_per_rank * steps / seconds_per_rank, seconds_per_rank
    import torch
    t = torch.tensor([float(seconds_per_rank)], dtype=torch.float64, device=device)
    n = torch.tensor([float(pairs_per_rank)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(n.item()) * steps / float(t.item()), float(t.item())


KERNEL_SOURCES = ("score_tc.cu", "tc_ptx.cuh", "common.cuh", "internal.h")


def kernel_source_hash() -> str:
    """sha256 over the sources the scoring kernel is built from."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "sparse_attention_top_paged_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(name: str):
    """DRAM bytes per launch of the scoring kernel from the committed ncu
    summary, or None when those counters were taken on another workload or
    on other kernel sources."""
    tfile = os.path.join(ROOT, "profiles", "score_tc_kernel.traffic.json")
    if not os.path.exists(tfile):
        return None
    rec = json.load(open(tfile))
    if rec.get("source_sha256") != kernel_source_hash() or rec.get("workload_name") != name:
        return None
    return rec.get("bytes_per_launch")


def launches_per_step(W) -> int:
    """Our kernels per idx_score_topk call on the tensor path: q preparation,
    the scorer, and the selection kernel."""
    return 3


def peaks():
    """(HBM GB/s, dense bf16/f16 tensor TFLOP/s burst, "measured"|"fallback")."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# Dense FP4 (block-scaled) tensor rate over the bf16 rate, nominal: 13.5 / 2.25.
FP4_OVER_BF16 = 6.0


def roofline(W, kern_s, q_format="exact", q_elem_bytes=4):
    """Roofline of the scoring kernel (q preparation + scorer). Decode
    workloads stream every key once: HBM bound, 72.125 B per pair plus q, w
    and the length per query. Prefill shares 128 blocks of keys between 4096
    rows: the 2*H*D flops per pair on the tensor cores bound it (f16 runs at
    the bf16 rate; the NVFP4-q mode's FP4 MMA against the measured bf16 peak
    times the nominal FP4/bf16 ratio)."""
    hbm, tensor, kind = peaks()
    if W.name == "prefill":
        flops = 2.0 * W.H * W.D * W.pairs
        achieved = flops / kern_s / 1e12
        peak = tensor if q_format == "exact" else tensor * FP4_OVER_BF16
        pk = kind if q_format == "exact" else f"{kind} bf16 x {FP4_OVER_BF16:g} (nominal FP4/bf16)"
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None, "kernel": "score_tc_kernel",
                "peak_kind": pk, "algorithmic_flops_per_launch": flops}
    algo_bytes = W.pairs * BYTES_PER_PAIR + W.T * (q_elem_bytes * W.H * W.D + 4 * W.H + 4)
    achieved = algo_bytes / kern_s / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": recorded_traffic(W.name) if q_format == "exact" else None, "kernel": "score_tc_kernel",
            "peak_kind": kind,
            "algorithmic_bytes_per_launch": algo_bytes}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
            return self
        # nvidia-smi takes a moment to start: wait for its first sample so the
        # samples cover the timed region
        t0 = time.perf_counter()
        while not self.lines and time.perf_counter() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0])); mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _oracle_run(W, rows, cap=None):
    """The float64 oracle on query rows ``rows`` of W, each truncated to its
    first ``cap`` keys when cap is given. Returns (pairs, seconds)."""
    import numpy as np
    import oracle
    lens = W.valid_lens if cap is None else np.minimum(W.valid_lens, cap).astype(np.int32)
    t0 = time.perf_counter()
    oracle.score_topk(W.q, W.w, W.block_table, W.bt_stride, W.max_lb, lens, W.epb, W.top_k,
                      rows=list(rows), **W.oracle_kwargs())
    dt = time.perf_counter() - t0
    return int(sum(int(lens[t]) for t in rows)), dt


def _set_threads(threads: int):
    os.environ["OPENBLAS_NUM_THREADS"] = str(threads)
    os.environ["OMP_NUM_THREADS"] = str(threads)


def _oracle_sample(args):
    """Runs in a spawned process: the float64 oracle, one thread, on the first
    n queries."""
    name, seed, n_queries = args
    _set_threads(1)
    W = make_workload(name, seed)
    n = min(n_queries, W.T)
    return _oracle_run(W, range(n)) + (n,)


def _oracle_worker(name, seed, rows, barrier, out):
    """Runs in a spawned process: the float64 oracle, one thread, on ``rows``
    of the workload, started together with the other workers."""
    _set_threads(1)
    W = make_workload(name, seed)
    barrier.wait()
    t0 = time.perf_counter()
    pairs, _ = _oracle_run(W, rows)
    out.put((pairs, t0, time.perf_counter()))


def cpu_baseline(name: str, seed: int, n_queries: int):
    """The float64 oracle on the first n_queries queries of the workload:
    once on one thread, and once with one single-threaded process per host
    core, the queries dealt out between them (the reported value)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    ctx = mp.get_context("spawn")
    with ctx.Pool(1) as pool:
        pairs1, dt1, n = pool.apply(_oracle_sample, ((name, seed, n_queries),))
    procs = max(1, min(cores, n))
    barrier, out = ctx.Barrier(procs), ctx.Queue()
    workers = [ctx.Process(target=_oracle_worker, args=(name, seed, list(range(n))[i::procs], barrier, out))
               for i in range(procs)]
    for wkr in workers:
        wkr.start()
    res = [out.get() for _ in workers]
    for wkr in workers:
        wkr.join()
    pairs = sum(r[0] for r in res)
    dt = max(r[2] for r in res) - min(r[1] for r in res)
    return {"value": pairs / dt, "unit": UNIT, "cores": procs, "kind": "oracle",
            "sample": f"first {n} of the {name} queries ({pairs} pairs), numpy float64, one single-threaded "
                      f"process per core ({procs}), {dt:.2f} s",
            "seconds": dt, "single_thread_value": pairs1 / dt1, "single_thread_seconds": dt1}


REFERENCE_BUDGET_S = 120.0


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm. Every step scores one query row
    (rows taken in turn), truncated to its first n keys, where n is sized from
    a calibration run so that all timed steps together take about two
    minutes of oracle time."""
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0))
    _set_threads(cores)
    name = args.workload
    W = make_workload(name, WORKLOADS[name][1])
    p, dt = _oracle_run(W, [0])                  # calibration, untimed
    per_step = max(256, min(int(W.valid_lens.max()), int(p / dt * REFERENCE_BUDGET_S / max(args.steps, 1))))
    for i in range(args.warmup):
        _oracle_run(W, [i % W.T], per_step)
    times, pairs = [], 0
    for i in range(args.steps):
        p, dt = _oracle_run(W, [i % W.T], per_step)
        times.append(dt)
        pairs += p
    total = sum(times)
    value = pairs / total
    sample = (f"one query row per step (rows in turn), at most its first {per_step} keys "
              f"(rows hold {int(W.valid_lens.min())}..{int(W.valid_lens.max())}), numpy float64")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(W), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


QSA_STEP = ("qsa_qprep (32 heads of one decode query at position 8192) + block_pool (8192 raw bf16 keys -> "
            "512 pooled blocks) + score_topk (32 heads, F32 keys, k=64) + expand_blocks + gather_kv (1024 tokens, "
            "4 kv heads x 128, K and V)")


def _qsa_oracle(Q):
    """The float64 oracle over the whole QSA chain; returns seconds."""
    import numpy as np
    import oracle
    hd = Q.raw_keys.shape[1]
    nh = Q.q_raw_bits.shape[1] // hd
    q_vals = (Q.q_raw_bits.astype(np.uint32) << 16).view(np.float32)
    t0 = time.perf_counter()
    q = oracle.qsa_qprep_rows(q_vals, Q.q_norm_w, 1, Q.raw_keys.shape[0], nh * hd, nh, hd, Q.rot, Q.theta,
                              Q.eps)[0]
    keys = oracle.block_pool(Q.raw_keys, Q.k_norm_w, 0, Q.n_blocks, Q.ratio, Q.rot, Q.theta, Q.eps)
    sc = oracle.qsa_score(q, keys)
    order = np.lexsort((np.arange(sc.size), -sc))[:Q.top_k]
    pos = oracle.expand_blocks(order[None].astype(np.int32), Q.ratio)
    oracle.gather_kv(pos, Q.page_table, Q.page_table.shape[1], Q.page_table.shape[1], Q.block_size,
                     Q.k_cache_bits, Q.v_cache_bits)
    return time.perf_counter() - t0


def run_qsa(args, rank, world):
    """The QSA chain (pooling, block scoring, top-k, expansion, K/V gather) as
    one step, replayed from a CUDA graph of the public API calls:
    latency-bound, reported in pairs/s (512 scored blocks per step) and
    microseconds."""
    import math
    import numpy as np
    import torch
    import sparse_attention_top_paged_gb300 as idx
    from sparse_attention_top_paged_gb300 import workloads
    Q = workloads.qsa(1004 + rank)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt = _qsa_oracle(Q)
        cpu = {"value": Q.n_blocks / dt, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"the whole QSA chain once, numpy float64, {dt:.3f} s", "seconds": dt}
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda")
    hd, nb = Q.raw_keys.shape[1], Q.n_blocks
    raw = torch.from_numpy(Q.raw_keys_bits.view(np.int16)).to(dev)
    nw = torch.from_numpy(Q.k_norm_w).to(dev)
    n_heads = Q.q.shape[0]
    q_raw = torch.from_numpy(Q.q_raw_bits.view(np.int16)).to(dev)
    q_nw = torch.from_numpy(Q.q_norm_w).to(dev)
    q = torch.empty((1, n_heads, hd), device=dev)
    w = torch.full((1, n_heads), 1.0 / math.sqrt(hd), device=dev)
    table = torch.arange(nb // 64, dtype=torch.int32, device=dev).reshape(1, -1)
    lens = torch.tensor([nb], dtype=torch.int32, device=dev)
    kc = torch.from_numpy(Q.k_cache_bits.view(np.int16)).to(dev)
    vc = torch.from_numpy(Q.v_cache_bits.view(np.int16)).to(dev)
    ptab = torch.from_numpy(Q.page_table).to(dev)
    bk = torch.empty((nb, hd), device=dev)
    gi = torch.empty((1, Q.top_k), dtype=torch.int32, device=dev)
    gs = torch.empty((1, Q.top_k), device=dev)
    n_tok = Q.top_k * Q.ratio
    k_out = torch.empty((1, n_tok) + tuple(kc.shape[2:]), dtype=kc.dtype, device=dev)
    v_out = torch.empty_like(k_out)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        idx.qsa_qprep(q_raw, q_nw, n_heads, Q.rot, Q.theta, Q.eps, first_pos=Q.raw_keys.shape[0], out=q)
        idx.block_pool(raw, nw, bk, 0, nb, Q.ratio, Q.rot, Q.theta, Q.eps)
        idx.score_topk(q, w, table, lens, Q.top_k, entries_per_block=64, keys_f32=bk.reshape(nb // 64, 64, hd),
                       out=(gi, gs))
        pos = idx.expand_blocks(gi, Q.ratio)
        idx.gather_kv(pos, ptab, Q.block_size, kc, vc, out=(k_out, v_out))

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    # The six launches of a step are captured once in a CUDA graph: issued
    # from Python one by one they take longer on the host than on the device.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    value, t_total = whole_job(nb, K, sum(ms) / 1e3)
    # end to end: the query's projection row in from pinned host memory, the
    # selected blocks and their scores out
    hq = torch.from_numpy(Q.q_raw_bits.view(np.int16).copy()).pin_memory()
    ho_i = torch.empty((1, Q.top_k), dtype=torch.int32).pin_memory()
    ho_s = torch.empty((1, Q.top_k), dtype=torch.float32).pin_memory()
    E = max(10, K // 10)
    e2e = []
    for _ in range(E):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        q_raw.copy_(hq, non_blocking=True)
        graph.replay()
        ho_i.copy_(gi, non_blocking=True)
        ho_s.copy_(gs, non_blocking=True)
        b.record(stream)
        e2e.append((a, b))
    torch.cuda.synchronize()
    e2e_value, _ = whole_job(nb, E, sum(a.elapsed_time(b) for a, b in e2e) / 1e3)
    # algorithmic bytes: the query row in and prepared q out and back in, raw keys in,
    # pooled keys out and back in, the gathered rows in and out
    row = int(np.prod(kc.shape[2:])) * kc.element_size()
    algo = q_raw.numel() * 2 + 2 * q.numel() * 4 + raw.numel() * 2 + 2 * bk.numel() * 4 + 2 * 2 * n_tok * row
    hbm, _, kind = peaks()
    achieved = algo / (t_total / K) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_total / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": "qsa: " + QSA_STEP, "pairs_per_step": nb, "seed": 1004, "cuda_graph": True,
                       "l2": "flushed before every timed step (256 MB write, outside the timed events)"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": hq.numel() * 2,
                    "d2h_bytes_per_step": ho_i.numel() * 4 + ho_s.numel() * 4},
            "gpu_launches": 6 * K,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": None, "kernel": "whole QSA chain (latency-bound)", "peak_kind": kind,
                         "algorithmic_bytes_per_launch": algo},
            "cpu_baseline": cpu, "clocks": clk.summary()}), flush=True)


def qsa_attn_case(seed: int, rows: int = 512, first_pos: int = 8192, nq: int = 32, nkv: int = 4, hd: int = 128,
                  ratio: int = 16, bs: int = 16, topk: int = 64):
    """Prefill rows at positions first_pos.. over 64 distinct complete blocks
    each (ascending) plus their tails, from bf16 caches behind a shuffled page
    table."""
    import numpy as np
    from sparse_attention_top_paged_gb300 import workloads
    rng = np.random.default_rng(seed)
    pages = (first_pos + rows + bs - 1) // bs
    P = pages + 8
    kbits = workloads._to_bf16_bits(rng.standard_normal((P, bs, nkv, hd)).astype(np.float32))
    vbits = workloads._to_bf16_bits(rng.standard_normal((P, bs, nkv, hd)).astype(np.float32))
    table = rng.permutation(P)[:pages].astype(np.int32)
    ncomp = [(first_pos + r + 1) // ratio for r in range(rows)]
    lists = np.stack([np.sort(rng.choice(ncomp[r], size=topk, replace=False)) for r in range(rows)]).astype(np.int32)
    q = rng.standard_normal((rows, nq, hd)).astype(np.float32)
    tokens = sum(topk * ratio + (first_pos + r + 1) - ncomp[r] * ratio for r in range(rows))
    return dict(q=q, kbits=kbits, vbits=vbits, table=table, lists=lists, first_pos=first_pos, ratio=ratio,
                tokens=tokens, rows=rows, nq=nq, nkv=nkv, hd=hd)


def run_qsa_attn(args, rank, world):
    """QSA prefill attention (idx_qsa_prefill_attn) over 512 rows: (row,
    head, token) scores per second. Both contractions run on the tensor
    cores: 4*hd flops per (row, head, token) (the q.k dot product and the
    weighted V sum) against the bf16 tensor peak. With 8 heads per kv head a
    gathered K or V element feeds 16 flops, so the kernel is bound by the
    gather of K and V rows from L2 (17.8 MB of pages, each row gathered by
    every query row that selects it), far below the tensor peak; the line
    carries those gathered bytes and their rate as context."""
    import math
    import numpy as np
    import torch
    import sparse_attention_top_paged_gb300 as idx
    c = qsa_attn_case(1005 + rank)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        n = 4
        vals = lambda b: (b.astype(np.uint32) << 16).view(np.float32)
        t0 = time.perf_counter()
        oracle.qsa_prefill_attn(c["q"][:n], vals(c["kbits"]), vals(c["vbits"]), c["table"], c["lists"][:n],
                                c["first_pos"], c["ratio"], 1.0 / math.sqrt(c["hd"]))
        dt = time.perf_counter() - t0
        pairs_n = c["tokens"] * n / c["rows"]
        cpu = {"value": pairs_n * c["nq"] / dt, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"first {n} of {c['rows']} rows, all {c['nq']} heads, numpy float64, {dt:.2f} s",
               "seconds": dt}
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda")
    q = torch.from_numpy(c["q"]).to(dev)
    kc = torch.from_numpy(c["kbits"].view(np.int16)).to(dev)
    vc = torch.from_numpy(c["vbits"].view(np.int16)).to(dev)
    table = torch.from_numpy(c["table"]).to(dev)
    lists = torch.from_numpy(c["lists"]).to(dev)
    out = torch.empty_like(q)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        idx.qsa_prefill_attn(q, kc, vc, table, lists, c["first_pos"], c["ratio"], out=out)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    pairs = c["tokens"] * c["nq"]            # (row, head, token) scores per step
    value, t_total = whole_job(pairs, K, sum(a.elapsed_time(b) for a, b in ev) / 1e3)
    hq = torch.from_numpy(c["q"]).pin_memory()
    ho = torch.empty_like(hq).pin_memory()
    E = max(10, K // 10)
    e2e = []
    for _ in range(E):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        q.copy_(hq, non_blocking=True)
        step()
        ho.copy_(out, non_blocking=True)
        b.record(stream)
        e2e.append((a, b))
    torch.cuda.synchronize()
    e2e_value, _ = whole_job(pairs, E, sum(a.elapsed_time(b) for a, b in e2e) / 1e3)
    flops = 4.0 * c["hd"] * pairs
    achieved = flops / (t_total / K) / 1e12
    gathered = c["tokens"] * c["nkv"] * c["hd"] * 2 * 2   # K and V rows, bf16, per (row, kv head, token)
    _, tensor, kind = peaks()
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_total / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"qsa_attn: {c['rows']} prefill rows from position {c['first_pos']}, 64 selected "
                                   f"blocks of 16 tokens + tail each, nq={c['nq']} nkv={c['nkv']} hd={c['hd']}, "
                                   "bf16 paged K/V", "pairs_per_step": pairs, "seed": 1005,
                       "l2": "flushed before every timed step (256 MB write, outside the timed events)"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": hq.numel() * 4,
                    "d2h_bytes_per_step": ho.numel() * 4},
            "gpu_launches": K,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": tensor, "unit": "TFLOP/s",
                         "frac": achieved / tensor, "traffic": None,
                         "kernel": "qsa_prefill_attn_tc_kernel", "peak_kind": kind,
                         "algorithmic_flops_per_launch": flops,
                         "gathered_bytes_per_launch": gathered,
                         "gathered_gbs": gathered / (t_total / K) / 1e9},
            "cpu_baseline": cpu, "clocks": clk.summary()}), flush=True)


def gather_split_case(seed: int):
    """The split-gather workload: 64 queries x 2048 sorted positions of a
    262144-token cache (block 64), 512 E4M3 codes (no NaN code) + an f32
    scale in [0.01, 4) + 64 bf16 rope values per token, one page-table
    permutation per query."""
    import numpy as np
    from sparse_attention_top_paged_gb300 import workloads
    rng = np.random.default_rng(seed)
    T, n, bs, nd, rd, n_tok = 64, 2048, 64, 512, 64, 262144
    P = n_tok // bs
    codes = rng.integers(0, 256, size=(P, bs, nd), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38
    scale = rng.uniform(0.01, 4.0, size=(P, bs)).astype(np.float32)
    rope = workloads._to_bf16_bits(rng.standard_normal((P, bs, rd)).astype(np.float32))
    table = np.stack([rng.permutation(P) for _ in range(T)]).astype(np.int32)
    sel = np.stack([np.sort(rng.choice(n_tok, size=n, replace=False)) for _ in range(T)]).astype(np.int32)
    return {"T": T, "n": n, "bs": bs, "nd": nd, "rd": rd, "n_tok": n_tok, "P": P, "codes": codes, "scale": scale,
            "rope": rope, "table": table, "sel": sel}


def run_gather_split(args, rank, world):
    """The FP8 + BF16 split gather (idx_gather_split): 64 queries x 2048
    selected positions from a 262144-token paged cache, 512 E4M3 + per-token
    scale + 64 bf16 per token, into a dense bf16 tile. HBM bound: gathered
    bytes in, the tile out."""
    import numpy as np
    import torch
    import sparse_attention_top_paged_gb300 as idx
    c = gather_split_case(1006 + rank)
    T, n, bs, nd, rd, n_tok, P = c["T"], c["n"], c["bs"], c["nd"], c["rd"], c["n_tok"], c["P"]
    codes, scale, rope, table, sel = c["codes"], c["scale"], c["rope"], c["table"], c["sel"]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        oracle.gather_split(sel[:2], table[:2], P, P, bs, codes, scale, rope)
        dt = time.perf_counter() - t0
        cpu = {"value": 2 * n / dt, "unit": "rows/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"2 of {T} queries ({2 * n} rows), numpy, {dt:.2f} s", "seconds": dt}
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda")
    d = lambda x: torch.from_numpy(x).to(dev)
    dsel, dtab, dcodes, dscale, drope = d(sel), d(table), d(codes), d(scale), d(rope.view(np.int16))
    out = torch.empty((T, n, nd + rd), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        idx.gather_split(dsel, dtab, bs, dcodes, drope, dscale, out=out)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    rows = T * n
    value, t_total = whole_job(rows, K, sum(a.elapsed_time(b) for a, b in ev) / 1e3)
    hsel = torch.from_numpy(sel).pin_memory()
    hout = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    E = max(10, K // 10)
    e2e = []
    for _ in range(E):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dsel.copy_(hsel, non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)
        b.record(stream)
        e2e.append((a, b))
    torch.cuda.synchronize()
    e2e_value, _ = whole_job(rows, E, sum(a.elapsed_time(b) for a, b in e2e) / 1e3)
    algo = rows * (nd + 4 + 2 * rd + 2 * (nd + rd) + 4)   # nope, scale, rope in; the tile out; sel
    hbm, _, kind = peaks()
    achieved = algo / (t_total / K) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "gathered rows per sec (FP8+BF16 split -> BF16 tile)", "value": value, "unit": "rows/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8->bf16",
            "data": "synthetic",
            "config": {"workload": f"gather_split: T={T} x {n} positions of {n_tok}, 512 e4m3 + scale + 64 bf16 "
                                   "per token, block 64", "rows_per_step": rows, "seed": 1006,
                       "l2": "flushed before every timed step (256 MB write, outside the timed events)"},
            "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": hsel.numel() * 4,
                    "d2h_bytes_per_step": hout.numel() * 2},
            "gpu_launches": K,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": None, "kernel": "gather_split_vec_kernel", "peak_kind": kind,
                         "algorithmic_bytes_per_launch": algo},
            "cpu_baseline": cpu, "clocks": clk.summary()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="auto", choices=["auto", "tensor", "simt"])
    ap.add_argument("--workload", default="batched_decode",
                    choices=sorted(WORKLOADS) + ["qsa", "qsa_attn", "gather_split"])
    ap.add_argument("--cpu-queries", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="batched_decode only: skip the long-decode, prefill and NVFP4-q sub-records")
    ap.add_argument("--q-format", default="exact", choices=["exact", "nvfp4"],
                    help="nvfp4: the opt-in mode scoring NVFP4-quantised queries on the FP4 MMA")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.workload == "qsa":
        return run_qsa(args, rank, world)
    if args.workload == "qsa_attn":
        return run_qsa_attn(args, rank, world)
    if args.workload == "gather_split":
        return run_gather_split(args, rank, world)

    import torch
    import sparse_attention_top_paged_gb300 as idx

    # the CPU baseline runs in spawned processes before any GPU work
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, rank_seed(args.workload, 0), args.cpu_queries)

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    W = make_workload(args.workload, rank_seed(args.workload, rank))
    rec = measure_score(W, args, args.steps, dev, flush, dist, e2e=True, q_format=args.q_format)
    extra = {}
    if args.workload == "batched_decode" and not args.no_extra_workloads and args.q_format == "exact":
        # the other two full-size configurations, device-timed, same warm-up,
        # at most EXTRA_STEPS timed steps each; then the opt-in NVFP4-q mode
        # on batched decode and prefill
        del W
        for name, qf in (("long_decode", "exact"), ("prefill", "exact"), ("batched_decode", "nvfp4"),
                         ("prefill", "nvfp4")):
            W2 = make_workload(name, rank_seed(name, rank))
            r2 = measure_score(W2, args, min(args.steps, EXTRA_STEPS), dev, flush, dist, e2e=False, q_format=qf)
            key = name if qf == "exact" else f"{name}_nvfp4_q"
            extra[key] = {"metric": METRIC, "value": r2["value"], "unit": UNIT, "steps": r2["steps"],
                          "ms_per_step": r2["ms_per_step"], "config": dict(r2["config"], q_format=qf),
                          "roofline": r2["roofline"], "clocks": r2["clocks"]}
            del W2
            torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": rec["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16" if args.q_format == "exact" else "e2m1",
            "data": "synthetic",
            "config": dict(rec["config"], parallelism=f"replicas x{world} (independent batches)",
                           q_format=args.q_format,
                           mma=("tcgen05 kind::f16, f16 x f16 -> f32 (exact for NVFP4 x bf16-valued q)"
                                if args.q_format == "exact" else
                                "tcgen05 kind::mxf4nvf4 block-scaled, e2m1 x e2m1 with e4m3 group scales -> f32 "
                                "(q quantised to NVFP4)")),
            "e2e": rec["e2e"],
            "gpu_launches": rec["gpu_launches"],
            "roofline": rec["roofline"],
            "cpu_baseline": cpu,
            "clocks": rec["clocks"],
            "wall_s": rec["wall_s"],
        }
        if extra:
            line["workloads"] = extra
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


EXTRA_STEPS = 2000


def measure_score(W, args, K, dev, flush, dist, e2e, q_format="exact"):
    """Device-timed idx_score_topk steps over W (L2 flushed before each), and
    optionally the end-to-end leg through the public Python call."""
    import ctypes
    import numpy as np
    import torch
    import sparse_attention_top_paged_gb300 as idx
    q = torch.from_numpy(W.q).to(dev)
    # The workloads' queries are bf16 values (the page's launcher upcasts its
    # bf16 q_I): they go in as bf16 (q_dtype BF16), which the library reads as
    # exactly those float32 values; a float32-only q stays float32.
    if torch.equal(q.to(torch.bfloat16).float(), q):
        q = q.to(torch.bfloat16)
    w = torch.from_numpy(W.w).to(dev)
    bt = torch.from_numpy(W.block_table).to(dev)
    vl = torch.from_numpy(W.valid_lens).to(dev)
    fp4 = torch.from_numpy(W.keys_fp4).to(dev)
    sc = torch.from_numpy(W.key_scale).to(dev)
    gs = torch.from_numpy(W.key_gscale).to(dev)
    k = W.top_k
    out_i = torch.empty((W.T, k), dtype=torch.int32, device=dev)
    out_s = torch.empty((W.T, k), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lib = idx.load_library()
    stream = torch.cuda.current_stream(dev)

    a = idx.make_score_args(q, w, bt, vl, k, entries_per_block=W.epb, bt_stride=W.bt_stride,
                            keys_fp4=fp4, key_scale=sc,
                            key_gscale=gs, topk_idx=out_i, topk_score=out_s, dev_status=status,
                            path=args.path, q_format=q_format)
    ws_bytes = idx.score_topk_workspace_bytes(a)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    sptr = ctypes.c_void_p(stream.cuda_stream)

    def step(events=None):
        if events is not None:
            a.timing_events[0] = events[0].cuda_event
            a.timing_events[1] = events[1].cuda_event
        else:
            a.timing_events[0] = None
            a.timing_events[1] = None
        rc = lib.idx_score_topk(ctypes.byref(a), sptr)
        if rc != 0:
            raise idx.IndexerError("idx_score_topk", rc)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    # The scoring kernel is bracketed by events on every KSAMPLE-th timed step:
    # an event recorded between the scorer and the selection kernel stops the
    # selection's programmatic early launch (about 5 us per step), so
    # bracketing every step would inflate the step time it is part of.
    KSAMPLE = 8
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range((K + KSAMPLE - 1) // KSAMPLE)]
    for pair in kev:          # torch creates the CUDA event on first record; the library records it later
        pair[0].record(stream)
        pair[1].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        wall0 = time.perf_counter()
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            step(kev[i // KSAMPLE] if i % KSAMPLE == 0 else None)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if dist:
        dist.barrier()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    step_ms = [s.elapsed_time(e) for s, e in ev]
    kern_ms = [s.elapsed_time(e) for s, e in kev]
    pairs_step = W.pairs
    value, t_total = whole_job(pairs_step, K, sum(step_ms) / 1e3, dist, dev)
    kern_s = statistics.mean(kern_ms) / 1e3
    rec = {"value": value, "steps": K, "ms_per_step": 1e3 * t_total / K,
           "config": dict(workload_config(W), q_dtype=str(q.dtype).replace("torch.", "")),
           "roofline": dict(roofline(W, kern_s, q_format, q.element_size()), kernel_ms=1e3 * kern_s,
                            kernel_timed_steps=len(kern_ms)),
           "clocks": clk.summary(), "wall_s": wall, "gpu_launches": launches_per_step(W) * K}
    if not e2e:
        return rec

    # ---- end to end through the public Python API with host buffers ----
    # The step's inputs travel as one pinned host block into one device block
    # (q, w, block table, lengths at 256-byte-aligned offsets) and both
    # outputs come back as one block: one copy each way. Each step is timed
    # on the host, from the first host-side call to the return of a
    # synchronize after the copy out (what a caller waits for), once the L2
    # flush before it has finished; the CUDA-event span of the same steps is
    # reported beside it.
    def packed(parts):
        offs, total = [], 0
        for x in parts:
            offs.append(total)
            total += (x.nbytes + 255) // 256 * 256
        return offs, total

    # q travels in the dtype the device-timed leg used
    tdt = {np.dtype(np.float32): torch.float32, np.dtype(np.int32): torch.int32, np.dtype(np.uint16): torch.bfloat16}
    q_host = (q.view(torch.int16).cpu().numpy().view(np.uint16) if q.dtype == torch.bfloat16 else W.q)
    in_parts = [q_host, W.w, W.block_table, W.valid_lens]
    in_offs, in_bytes = packed(in_parts)
    h_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    for x, o in zip(in_parts, in_offs):
        h_in[o:o + x.nbytes].copy_(torch.from_numpy(np.ascontiguousarray(x).view(np.uint8).reshape(-1)))
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    eq, ew, ebt, evl = (d_in[o:o + x.nbytes].view(tdt[x.dtype]).view(x.shape) for x, o in zip(in_parts, in_offs))
    out_bytes = (W.T * k * 4 + 255) // 256 * 256
    d_out = torch.empty(2 * out_bytes, dtype=torch.uint8, device=dev)
    e_i = d_out[:W.T * k * 4].view(torch.int32).view(W.T, k)
    e_s = d_out[out_bytes:out_bytes + W.T * k * 4].view(torch.float32).view(W.T, k)
    h_out = torch.empty(2 * out_bytes, dtype=torch.uint8).pin_memory()
    h2d, d2h = in_bytes, 2 * out_bytes
    E = max(10, K // 10)

    # The call is the public API's prepared form, as a serving loop holds it:
    # a ScoreTopkPlan bound to the input and output blocks (arguments checked
    # and marshalled once), run once per step over the freshly copied inputs.
    plan = idx.ScoreTopkPlan(eq, ew, ebt, evl, k, entries_per_block=W.epb, bt_stride=W.bt_stride, keys_fp4=fp4,
                             key_scale=sc, key_gscale=gs, out=(e_i, e_s), workspace=ws, q_format=q_format)

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        plan.run()
        h_out.copy_(d_out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    host_s, dev_ms = [], []
    for _ in range(E):
        flush.zero_()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        s0.record(stream)
        e2e_step()
        s1.record(stream)
        torch.cuda.synchronize()
        host_s.append(time.perf_counter() - t0)
        dev_ms.append(s0.elapsed_time(s1))
    e2e_value, e2e_t = whole_job(pairs_step, E, sum(host_s), dist, dev)
    e2e_dev, _ = whole_job(pairs_step, E, sum(dev_ms) / 1e3, dist, dev)
    # the host copy holds what the device-timed steps produced
    if not torch.equal(h_out[:W.T * k * 4].view(torch.int32).view(W.T, k), out_i.cpu()):
        raise RuntimeError("end-to-end top-k differs from the device-timed steps")
    rec["e2e"] = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                  "ms_per_step": 1e3 * e2e_t / E,
                  "timing": "host perf_counter around copy in + ScoreTopkPlan.run + copy out + synchronize",
                  "device_value": e2e_dev, "device_ms_per_step": statistics.mean(dev_ms), "steps": E}
    return rec


if __name__ == "__main__":
    main()
