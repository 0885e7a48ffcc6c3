"""idx_score_topk_static, called through the C ABI.

Some callers of this library may not call cudaMalloc (an operator inside a host
runtime that owns all device memory and gives it no allocator, or a serving
loop that must not allocate once running). idx_score_topk_static serves them
with a scratch array built into the library instead of a caller workspace.
Here it must return what idx_score_topk returns with a caller-provided
workspace on the same inputs, and what the float64 oracle computes, on two
calls in a row (the second call finds the first call's leftovers in the shared
array), and must refuse, without launching, arguments that need more scratch
than the array holds.
"""

import ctypes

import numpy as np
import pytest

from sparse_attention_top_paged_gb300 import workloads as wl
from tests.gpu_common import check_against_oracle, ensure_built, oracle_rows, run_gpu, to_device
from tests.parity import REL_TOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _workload(seed):
    rng = np.random.default_rng(seed)
    vl = rng.integers(2000, 9000, size=16)
    return wl.decode_workload("no_alloc", seed, T=16, H=64, valid_lens=vl, max_lb=141, P=2300, top_k=512)


def _call_static(lib, W, d):
    import sparse_attention_top_paged_gb300 as idx
    gi = torch.full((W.T, W.top_k), -7, dtype=torch.int32, device="cuda")
    gs = torch.full((W.T, W.top_k), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = idx.make_score_args(d["q"], d["w"], d["bt"], d["vl"], W.top_k, entries_per_block=W.epb,
                            keys_fp4=d["keys_fp4"], key_scale=d["key_scale"], key_gscale=d["key_gscale"],
                            bt_stride=W.bt_stride, topk_idx=gi, topk_score=gs, dev_status=st)
    rc = lib.idx_score_topk_static(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, rc
    torch.cuda.synchronize()
    return gi.cpu().numpy(), gs.cpu().numpy(), int(st.item())


def _assert_same(ref_i, ref_s, gi, gs):
    """Same valid slots, scores within 1e-3 of the query's largest |score|,
    and the same index sets except keys within that tolerance of the k-th."""
    for t in range(ref_i.shape[0]):
        valid = ref_i[t] >= 0
        assert np.array_equal(gi[t] >= 0, valid), t
        assert np.all(np.isneginf(gs[t][~valid]))
        if not valid.any():
            continue
        tol = REL_TOL * float(np.max(np.abs(ref_s[t][valid])))
        assert np.all(np.abs(gs[t][valid] - ref_s[t][valid]) <= tol), t
        kth = float(ref_s[t][valid].min())
        score_of = dict(zip(ref_i[t][valid].tolist(), ref_s[t][valid].tolist()))
        score_of.update(zip(gi[t][valid].tolist(), gs[t][valid].tolist()))
        for i in set(ref_i[t][valid].tolist()) ^ set(gi[t][valid].tolist()):
            assert abs(score_of[i] - kth) <= tol, (t, i)


def test_static_scratch_matches_workspace_entry_point(lib):
    W = _workload(21)
    d = to_device(W)
    ref_i, ref_s, ref_st, _ = run_gpu(W, "auto", dev=d)   # idx_score_topk with a workspace
    assert ref_st == 0
    rows, _ = oracle_rows(W)
    for call in range(2):
        gi, gs, st = _call_static(lib, W, d)
        assert st == 0
        _assert_same(ref_i, ref_s, gi, gs)
        check_against_oracle(W, gi, gs, rows, None, f"static/{call}")
    # a different problem next: nothing of the previous call may leak into it
    W2 = _workload(22)
    d2 = to_device(W2)
    ref2 = run_gpu(W2, "auto", dev=d2)
    gi, gs, st = _call_static(lib, W2, d2)
    _assert_same(ref2[0], ref2[1], gi, gs)
    rows2, _ = oracle_rows(W2)
    check_against_oracle(W2, gi, gs, rows2, None, "static/next")


def test_static_scratch_rejects_oversized_arguments(lib):
    import sparse_attention_top_paged_gb300 as idx
    T, k = 1200, 4096                                   # needs > 8 MiB of candidates
    q = torch.zeros((T, 1, 128), dtype=torch.float32, device="cuda")
    w = torch.zeros((T, 1), dtype=torch.float32, device="cuda")
    bt = torch.zeros((T, 1024), dtype=torch.int32, device="cuda")   # 65536 keys per row
    vl = torch.zeros(T, dtype=torch.int32, device="cuda")
    fp4 = torch.zeros((1, 64, 64), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((1, 64, 8), dtype=torch.uint8, device="cuda")
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    gi = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    gs = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    a = idx.make_score_args(q, w, bt, vl, k, entries_per_block=64, keys_fp4=fp4, key_scale=sc, key_gscale=g,
                            topk_idx=gi, topk_score=gs)
    assert idx.score_topk_workspace_bytes(a) > lib_scratch_bytes()
    rc = lib.idx_score_topk_static(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 3                                      # IDX_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((gi == -7).all())                       # nothing was launched


def lib_scratch_bytes():
    from sparse_attention_top_paged_gb300 import _lib
    return _lib.STATIC_SCRATCH_BYTES
