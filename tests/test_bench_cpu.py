"""The benchmark's host-side arithmetic and its CPU reference arm (no GPU)."""

import json
import os
import subprocess
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _w(name, pairs, T, H=64, D=128):
    return SimpleNamespace(name=name, pairs=pairs, T=T, H=H, D=D)


def test_decode_roofline_counts_bytes_per_pair_and_query():
    W = _w("batched_decode", pairs=1_000_000, T=10)
    r = bench.roofline(W, kern_s=1e-4)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    algo = 1_000_000 * 72.125 + 10 * (4 * 64 * 128 + 4 * 64 + 4)
    assert r["algorithmic_bytes_per_launch"] == pytest.approx(algo)
    assert r["achieved"] == pytest.approx(algo / 1e-4 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])


def test_prefill_roofline_is_tensor_flops():
    W = _w("prefill", pairs=1000, T=4)
    r = bench.roofline(W, kern_s=1e-6)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["algorithmic_flops_per_launch"] == 2.0 * 64 * 128 * 1000
    assert r["achieved"] == pytest.approx(2.0 * 64 * 128 * 1000 / 1e-6 / 1e12)
    assert r["traffic"] is None


def test_traffic_record_only_for_its_workload_and_sources(tmp_path, monkeypatch):
    rec = {"bytes_per_launch": 123, "source_sha256": bench.kernel_source_hash(), "workload_name": "batched_decode"}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "score_tc_kernel.traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["source_sha256"])
    assert bench.recorded_traffic("batched_decode") == 123
    assert bench.recorded_traffic("long_decode") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "other")
    assert bench.recorded_traffic("batched_decode") is None


def test_reference_arm_prints_one_bounded_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "prefill", "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["steps"] == 3 and j["value"] > 0
    assert j["e2e"] == {"value": j["value"], "unit": "pairs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["config"]["workload"].startswith("prefill")


def test_warmup_below_three_is_refused():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "2"], capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert out.returncode != 0 and "warmup" in out.stderr


def test_gather_split_case_matches_its_recipe():
    c = bench.gather_split_case(1006)
    assert c["codes"].shape == (c["P"], c["bs"], c["nd"]) and c["P"] * c["bs"] == c["n_tok"]
    assert not (((c["codes"] & 0x7F) == 0x7F).any())          # no E4M3 NaN code
    assert c["sel"].shape == (c["T"], c["n"])
    for row in c["sel"]:
        assert (row[1:] > row[:-1]).all() and row[0] >= 0 and row[-1] < c["n_tok"]   # sorted, distinct
    for perm in c["table"]:
        assert sorted(perm.tolist()) == list(range(c["P"]))
    assert (c["scale"] >= 0.01).all() and (c["scale"] < 4.0).all()


def test_qsa_attn_case_token_count_is_its_definition():
    c = bench.qsa_attn_case(7, rows=9, first_pos=100, nq=4, nkv=2, hd=64, ratio=16, bs=16, topk=4)
    want = 0
    for r in range(c["rows"]):
        p = c["first_pos"] + r
        ncomp = (p + 1) // c["ratio"]
        blocks = c["lists"][r]
        assert len(set(blocks.tolist())) == len(blocks) and (blocks >= 0).all() and (blocks < ncomp).all()
        want += len(blocks) * c["ratio"] + (p + 1 - ncomp * c["ratio"])
    assert c["tokens"] == want
