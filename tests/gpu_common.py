"""Shared helpers of the GPU parity tests (imported only by ``-m gpu`` tests)."""

import numpy as np

import oracle
from tests.parity import check_query, check_scores_row


def ensure_built():
    from sparse_attention_top_paged_gb300 import _lib, build
    build.build()
    return _lib.load_library()


def to_device(W):
    import torch
    dev = "cuda"
    d = {
        "q": torch.from_numpy(np.ascontiguousarray(W.q)).to(dev),
        "w": torch.from_numpy(np.ascontiguousarray(W.w)).to(dev),
        "bt": torch.from_numpy(np.ascontiguousarray(W.block_table, dtype=np.int32)).to(dev),
        "vl": torch.from_numpy(np.ascontiguousarray(W.valid_lens, dtype=np.int32)).to(dev),
    }
    if W.keys_f32 is not None:
        d["keys_f32"] = torch.from_numpy(np.ascontiguousarray(W.keys_f32)).to(dev)
    else:
        d["keys_fp4"] = torch.from_numpy(np.ascontiguousarray(W.keys_fp4)).to(dev)
        d["key_scale"] = torch.from_numpy(np.ascontiguousarray(W.key_scale)).to(dev)
        d["key_gscale"] = torch.from_numpy(np.ascontiguousarray(W.key_gscale)).to(dev)
    return d


def run_gpu(W, path="auto", *, scores=False, num_ctas=0, dev=None, q_format="exact"):
    """One idx_score_topk call through the C ABI; returns numpy results."""
    import torch
    import sparse_attention_top_paged_gb300 as idx
    d = dev if dev is not None else to_device(W)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    so = None
    if scores:
        so = torch.full((W.T, W.max_lb * W.epb), float("nan"), dtype=torch.float32, device="cuda")
    keys = {k: d[k] for k in ("keys_fp4", "key_scale", "key_gscale", "keys_f32") if k in d}
    gi, gs = idx.score_topk(d["q"], d["w"], d["bt"], d["vl"], W.top_k, entries_per_block=W.epb,
                            bt_stride=W.bt_stride, scores_out=so, dev_status=st, path=path,
                            num_ctas=num_ctas, q_format=q_format, **keys)
    torch.cuda.synchronize()
    return (gi.cpu().numpy(), gs.cpu().numpy(), int(st.item()),
            None if so is None else so.cpu().numpy())


def oracle_rows(W, rows=None):
    return oracle.score_topk_rows(W.q, W.w, W.block_table, W.bt_stride, W.max_lb, W.valid_lens,
                                  W.epb, rows=rows, **W.oracle_kwargs())


def oracle_rows_nvfp4(W, rows=None):
    """Oracle score rows of the NVFP4-q mode: the exact definition applied to
    the NVFP4-quantised queries."""
    return oracle.score_topk_rows(oracle.nvfp4_q(W.q), W.w, W.block_table, W.bt_stride, W.max_lb, W.valid_lens,
                                  W.epb, rows=rows, **W.oracle_kwargs())


def _oracle_rows_job(args):
    """Runs in a spawned process: the oracle's score rows of one named
    workload (rebuilt from its seed) for the given query rows."""
    name, seed, rows, nvfp4 = args
    from sparse_attention_top_paged_gb300 import workloads as wl
    W = getattr(wl, name)(seed)
    return (oracle_rows_nvfp4 if nvfp4 else oracle_rows)(W, rows)[0]


def oracle_rows_parallel(name, seed, rows, procs=None, nvfp4=False):
    """``oracle_rows`` (``oracle_rows_nvfp4`` with ``nvfp4``) of the named
    workload for many rows, split over spawned processes (each rebuilds the
    workload from its seed)."""
    import multiprocessing as mp
    import os
    rows = list(rows)
    procs = procs or max(1, min(8, len(rows), len(os.sched_getaffinity(0))))
    chunks = [rows[i::procs] for i in range(procs) if rows[i::procs]]
    out = {}
    with mp.get_context("spawn").Pool(len(chunks)) as pool:
        for part in pool.map(_oracle_rows_job, [(name, seed, c, nvfp4) for c in chunks]):
            out.update(part)
    return out


def check_against_oracle(W, gi, gs, ref_rows, so=None, label=""):
    for t, I in ref_rows.items():
        check_query(I, gi[t], gs[t], W.top_k, where=f"{label} query {t}")
        if so is not None and I is not None:
            check_scores_row(I, so[t], where=f"{label} scores row {t}")
