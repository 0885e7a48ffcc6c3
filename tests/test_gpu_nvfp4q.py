"""The opt-in NVFP4 query mode (q_format="nvfp4") against the float64 oracle.

In this mode each head of q is quantised to NVFP4 (E2M1 codes, one E4M3 scale
per 16 elements, one float32 scale per head) and the tensor cores take keys
and queries in FP4 directly (block-scaled MMA). The oracle computes the same
definition on the quantised queries (oracle.nvfp4_q), so:
  * the quantisation itself (idx_quantize_q_nvfp4) must match the oracle's
    bit for bit: codes, scales and the per-head scale;
  * the scores must match the oracle's scores of the quantised queries to
    float32 accumulation (|diff| <= 2e-5 max |I| per query: products of E2M1
    codes and E4M3 scales are exact, only the sums round), and the top-k
    under the usual acceptance rule.
"""

import numpy as np
import pytest

import oracle
from sparse_attention_top_paged_gb300 import workloads as wl
from tests.gpu_common import (check_against_oracle, ensure_built, oracle_rows_nvfp4, oracle_rows_parallel,
                              run_gpu, to_device)
from tests.test_gpu_score import _long_rows, _small, prefill_sample_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TIGHT = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _quantize_gpu(q):
    import sparse_attention_top_paged_gb300 as idx
    c, s, g = idx.quantize_q_nvfp4(torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda())
    torch.cuda.synchronize()
    return c.cpu().numpy(), s.cpu().numpy(), g.cpu().numpy()


def _pack(codes):
    codes = np.asarray(codes, np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _quant_cases():
    rng = np.random.default_rng(31)
    cases = {
        "normal": rng.standard_normal((512, 128)),
        "bf16": torch.from_numpy(rng.standard_normal((256, 128)).astype(np.float32)).bfloat16().float().numpy(),
        "scaled": rng.standard_normal((512, 128)) * np.exp2(rng.integers(-40, 40, size=(512, 1))),
        "heavy": rng.standard_cauchy((256, 128)),
        "sparse": rng.standard_normal((256, 128)) * (rng.random((256, 128)) < 0.05),
        "zero_groups": rng.standard_normal((64, 128)) * np.repeat(rng.random((64, 8)) < 0.5, 16, axis=1),
        "grid": (rng.integers(-12, 13, size=(256, 128)) / 4.0) * np.exp2(rng.integers(-3, 4, size=(256, 1))),
    }
    z = np.zeros((4, 128)); z[1, 5] = 1e-3; z[2, :16] = 448.0; z[3, 100] = -2.0 ** -20
    cases["edge"] = z
    return {k: v.astype(np.float32) for k, v in cases.items()}


@pytest.mark.parametrize("case", list(_quant_cases().keys()))
def test_quantizer_bit_exact(case):
    q = _quant_cases()[case]
    c, s, g = _quantize_gpu(q)
    oc, osc, og = oracle.quantize_q_nvfp4(q)
    assert np.array_equal(g, og), case
    assert np.array_equal(s, osc), case
    assert np.array_equal(c, _pack(oc)), case


def test_quantizer_golden_head():
    import json
    import os
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_q_example.json")))
    x = np.zeros(128, np.float32)
    for off, vals in gold["x_nonzero"].items():
        x[int(off):int(off) + len(vals)] = vals
    c, s, g = _quantize_gpu(x[None])
    want = np.zeros(128, np.uint8)
    for off, vals in gold["codes_nonzero"].items():
        want[int(off):int(off) + len(vals)] = vals
    assert float(g[0]) == gold["gq"] and list(s[0]) == gold["scales"]
    assert np.array_equal(c[0], _pack(want))


def _check_tight(W, so, rows, label):
    for t, I in rows.items():
        if I is None:
            continue
        fin = np.isfinite(I)
        assert np.array_equal(np.isneginf(so[t][:len(I)]), ~fin), f"{label} row {t}: masked keys differ"
        if fin.any():
            tol = TIGHT * float(np.max(np.abs(I[fin])))
            err = float(np.max(np.abs(so[t][:len(I)][fin] - I[fin])))
            assert err <= tol, f"{label} row {t}: max |diff| {err:.3e} > {tol:.3e}"


def _run_and_check(W, label, rows=None):
    gi, gs, st, so = run_gpu(W, "tensor", scores=True, q_format="nvfp4")
    assert st == 0
    ref, _ = oracle_rows_nvfp4(W, rows)
    _check_tight(W, so, ref, label)
    check_against_oracle(W, gi, gs, ref, None, label)


@pytest.mark.parametrize("jitter", [0, 2])
def test_tiny(jitter):
    _run_and_check(wl.tiny_decode(1000 + jitter, gscale_pow2_jitter=jitter), f"tiny{jitter}")


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_small_batched(seed):
    _run_and_check(_small(seed, q_bf16=(seed != 3)), f"small{seed}")


def test_ragged_lengths():
    lens = [0, 1, 15, 16, 63, 64, 65, 127, 128, 129, 199, 200, 201, 1000, 2047, 4095]
    W = wl.decode_workload("ragged", 77, T=len(lens), H=64, valid_lens=lens, max_lb=64, P=1100, top_k=200)
    _run_and_check(W, "ragged")


@pytest.mark.parametrize("H", [1, 12, 96, 128])
def test_head_counts(H):
    W = _small(60 + H, T=5, H=H, lo=2000, hi=5000, k=100, max_lb=80, P=500)
    _run_and_check(W, f"H{H}")


def test_shared_table_row_pairs():
    """Every row reads one table: two rows per decoded tile (N = 128 MMA)."""
    _run_and_check(wl.prefill(5, rows=96, base=4000, ratio=4, n_blocks=24, top_k=256), "shared")


def test_shared_table_odd_rows():
    _run_and_check(wl.prefill(6, rows=37, base=3000, ratio=4, n_blocks=20, top_k=128), "shared-odd")


@pytest.mark.parametrize("num_ctas", [1, 7, 300])
def test_partition_independent(num_ctas):
    W = _small(71, T=6, lo=1000, hi=7000, k=64, max_lb=120, P=800)
    ref = run_gpu(W, "tensor", scores=True, q_format="nvfp4")
    got = run_gpu(W, "tensor", scores=True, q_format="nvfp4", num_ctas=num_ctas)
    assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[3], got[3], equal_nan=True)


def test_unsupported_combinations_raise():
    import sparse_attention_top_paged_gb300 as idx
    W = _small(81, T=2, lo=100, hi=300, k=16, max_lb=8, P=40)
    with pytest.raises(idx.IndexerError):
        run_gpu(W, "simt", q_format="nvfp4")
    W2 = _small(82, T=2, H=200, lo=100, hi=300, k=16, max_lb=8, P=40)
    with pytest.raises(idx.IndexerError):
        run_gpu(W2, "tensor", q_format="nvfp4")


@pytest.mark.parametrize("case", ["batched", "pairs", "split"])
def test_workspace_needs_no_initialisation(case):
    import sparse_attention_top_paged_gb300 as idx
    if case == "batched":
        W = _small(91, T=8, lo=3000, hi=9000, k=256, max_lb=150, P=1300)
    elif case == "pairs":
        W = wl.prefill(7, rows=40, base=3000, ratio=4, n_blocks=20, top_k=128)
    else:
        W = _long_rows(92, T=3, lo=65536, hi=80000, k=512, P=3800)
    d = to_device(W)
    out = (torch.empty((W.T, W.top_k), dtype=torch.int32, device="cuda"),
           torch.empty((W.T, W.top_k), dtype=torch.float32, device="cuda"))
    a = idx.make_score_args(d["q"], d["w"], d["bt"], d["vl"], W.top_k, entries_per_block=W.epb,
                            keys_fp4=d["keys_fp4"], key_scale=d["key_scale"], key_gscale=d["key_gscale"],
                            bt_stride=W.bt_stride, topk_idx=out[0], topk_score=out[1], path="tensor",
                            q_format="nvfp4")
    ws = torch.empty(idx.score_topk_workspace_bytes(a), dtype=torch.uint8, device="cuda")
    ref, _ = oracle_rows_nvfp4(W)
    for rep in range(2):
        g = torch.Generator(device="cpu").manual_seed(200 + rep)
        ws.copy_(torch.randint(0, 256, (ws.numel(),), dtype=torch.uint8, generator=g))
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        gi, gs = idx.score_topk(d["q"], d["w"], d["bt"], d["vl"], W.top_k, entries_per_block=W.epb,
                                bt_stride=W.bt_stride, keys_fp4=d["keys_fp4"], key_scale=d["key_scale"],
                                key_gscale=d["key_gscale"], dev_status=st, path="tensor", workspace=ws, out=out,
                                q_format="nvfp4")
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        check_against_oracle(W, gi.cpu().numpy(), gs.cpu().numpy(), ref, None, f"garbage-ws/{case}/{rep}")


# ----------------------------------------------- full-size workloads ----

def test_batched_decode_full():
    W = wl.batched_decode()
    _run_and_check(W, "batched")


def test_prefill_sampled_rows():
    W = wl.prefill()
    gi, gs, st, so = run_gpu(W, "tensor", scores=True, q_format="nvfp4")
    assert st == 0
    sample = prefill_sample_rows(W.T)
    ref = oracle_rows_parallel("prefill", W.meta["seed"], sample, nvfp4=True)
    _check_tight(W, so, ref, "prefill")
    check_against_oracle(W, gi, gs, ref, None, "prefill")


def test_long_decode_full():
    W = wl.long_decode()
    gi, gs, st, _ = run_gpu(W, "tensor", q_format="nvfp4")
    assert st == 0
    ref = oracle_rows_parallel("long_decode", W.meta["seed"], range(W.T), nvfp4=True)
    check_against_oracle(W, gi, gs, ref, None, "long")
