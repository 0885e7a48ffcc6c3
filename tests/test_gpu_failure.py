"""Failure paths that need a GPU, exercised without faulting it.

Every wait inside the scoring pipeline gives up after a limit, raises the
CTA's abort flag and lets the CTA drain its copies and MMAs before it exits;
the call then reports IDX_STATUS_TIMEOUT in the device status word. Here a
test build of the library (shortened wait limit, and CTA 0 waiting once for a
barrier nothing ever arrives on) takes that path on purpose: the call must
return promptly with the status bit set, and the same CUDA context must then
run the regular library correctly.
"""

import ctypes
import time

import numpy as np
import pytest

from sparse_attention_top_paged_gb300 import workloads as wl
from tests.gpu_common import check_against_oracle, ensure_built, oracle_rows, run_gpu, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def stall_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    from sparse_attention_top_paged_gb300 import _lib, build
    path = build.build_variant("stall", defines=("IDX_TEST_STALL=1", "IDX_WAIT_LIMIT_NS=20000000ull"),
                               sources=("score_tc.cu",))
    return _lib.load_library(path)


def test_stalled_wait_reports_timeout_and_leaves_context_usable(stall_lib):
    import sparse_attention_top_paged_gb300 as idx
    rng = np.random.default_rng(61)
    W = wl.decode_workload("stall", 61, T=6, H=64, valid_lens=rng.integers(3000, 9000, size=6), max_lb=150,
                           P=1000, top_k=256)
    d = to_device(W)
    gi = torch.empty((W.T, W.top_k), dtype=torch.int32, device="cuda")
    gs = torch.empty((W.T, W.top_k), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = idx.make_score_args(d["q"], d["w"], d["bt"], d["vl"], W.top_k, entries_per_block=W.epb,
                            keys_fp4=d["keys_fp4"], key_scale=d["key_scale"], key_gscale=d["key_gscale"],
                            bt_stride=W.bt_stride, topk_idx=gi, topk_score=gs, dev_status=st, path="tensor")
    need = ctypes.c_size_t(0)
    assert stall_lib.idx_score_topk_workspace_size(ctypes.byref(a), ctypes.byref(need)) == 0
    ws = torch.empty(max(need.value, 256), dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    t0 = time.perf_counter()
    rc = stall_lib.idx_score_topk(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert rc == 0
    assert int(st.item()) & idx.STATUS_TIMEOUT
    assert elapsed < 10.0, elapsed
    # the context is intact: the regular library computes the same problem correctly
    ri, rs_, rst, _ = run_gpu(W, "tensor", dev=d)
    assert rst == 0
    rows, _ = oracle_rows(W)
    check_against_oracle(W, ri, rs_, rows, None, "after-timeout")


@pytest.fixture(scope="module")
def stall_attn_lib():
    """The prefill attention's tcgen05 kernel built with a 20 ms wait limit and
    CTA 0's MMA warp waiting once for a barrier nothing arrives on."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    from sparse_attention_top_paged_gb300 import _lib, build
    path = build.build_variant("stall_attn", defines=("IDX_TEST_STALL=1", "IDX_WAIT_LIMIT_NS=20000000ull"),
                               sources=("qsa_attn_tc.cu",))
    return _lib.load_library(path)


def test_attention_stalled_wait_reports_timeout_and_leaves_context_usable(stall_attn_lib):
    """The attention's abort path: CTA 0 gives up without issuing an MMA, its
    producers leave with their copies drained, the call returns promptly with
    IDX_STATUS_TIMEOUT, and the regular library then computes correctly."""
    import math
    import oracle
    import sparse_attention_top_paged_gb300 as idx
    rng = np.random.default_rng(62)
    rows, nq, nkv, hd, bs, ratio, fp, topk = 6, 16, 2, 128, 16, 16, 2000, 64
    pages = (fp + rows + bs - 1) // bs
    kb = wl._to_bf16_bits(rng.standard_normal((pages, bs, nkv, hd)).astype(np.float32))
    vb = wl._to_bf16_bits(rng.standard_normal((pages, bs, nkv, hd)).astype(np.float32))
    table = rng.permutation(pages).astype(np.int32)
    lists = rng.integers(0, (fp + 1) // ratio, size=(rows, topk)).astype(np.int32)
    q = rng.standard_normal((rows, nq, hd)).astype(np.float32)
    d = lambda x: torch.from_numpy(x).cuda()
    dq, dk, dv, dt, dl = d(q), d(kb.view(np.int16)), d(vb.view(np.int16)), d(table), d(lists)
    out = torch.zeros_like(dq)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    rc = stall_attn_lib.idx_qsa_prefill_attn(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dt.data_ptr(), pages, pages,
                                             dl.data_ptr(), out.data_ptr(), rows, fp, topk, ratio, bs, nq, nkv, hd,
                                             1.0 / math.sqrt(hd), st.data_ptr(),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert rc == 0
    assert int(st.item()) & idx.STATUS_TIMEOUT
    assert elapsed < 10.0, elapsed
    vals = lambda b: (b.astype(np.uint32) << 16).view(np.float32)
    got = idx.qsa_prefill_attn(dq, dk, dv, dt, dl, fp, ratio).cpu().numpy()
    ref, ost = oracle.qsa_prefill_attn(q, vals(kb), vals(vb), table, lists, fp, ratio, 1.0 / math.sqrt(hd))
    assert ost == 0 and np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref))


# --------------------------------------------------- debug-bounds build ----

@pytest.fixture(scope="module")
def debug_lib():
    """libidx built with -DIDX_DEBUG_BOUNDS: its index checks OR
    IDX_STATUS_DEBUG_BOUNDS into the status word and skip the access."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    from sparse_attention_top_paged_gb300 import _lib, build
    return _lib.load_library(build.build_variant("debug", defines=("IDX_DEBUG_BOUNDS",)))


def _score_with(lib, W, d, path):
    import sparse_attention_top_paged_gb300 as idx
    gi = torch.empty((W.T, W.top_k), dtype=torch.int32, device="cuda")
    gs = torch.empty((W.T, W.top_k), dtype=torch.float32, device="cuda")
    so = torch.full((W.T, W.max_lb * W.epb), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = idx.make_score_args(d["q"], d["w"], d["bt"], d["vl"], W.top_k, entries_per_block=W.epb,
                            keys_fp4=d["keys_fp4"], key_scale=d["key_scale"], key_gscale=d["key_gscale"],
                            bt_stride=W.bt_stride, topk_idx=gi, topk_score=gs, scores_out=so, dev_status=st,
                            path=path)
    need = ctypes.c_size_t(0)
    assert lib.idx_score_topk_workspace_size(ctypes.byref(a), ctypes.byref(need)) == 0
    ws = torch.empty(max(need.value, 256), dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    assert lib.idx_score_topk(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    torch.cuda.synchronize()
    return gi.cpu().numpy(), gs.cpu().numpy(), so.cpu().numpy(), int(st.item())


def _debug_cases():
    rng = np.random.default_rng(71)
    small = wl.decode_workload("dbg-small", 71, T=8, H=64, valid_lens=rng.integers(1, 6000, size=8), max_lb=100,
                               P=1024, top_k=128)
    ragged = wl.decode_workload("dbg-ragged", 72, T=8, H=12, valid_lens=[0, 1, 63, 64, 65, 127, 129, 4095],
                                max_lb=64, P=600, top_k=100)
    shared = wl.prefill(73, rows=33, base=4000, ratio=4, n_blocks=24, top_k=256)
    wide = wl.decode_workload("dbg-wide", 74, T=3, H=200, valid_lens=[500, 1700, 3000], max_lb=50, P=200, top_k=64)
    bad = wl.decode_workload("dbg-bad", 75, T=4, H=64, valid_lens=[2000, 2500, 3000, 2200], max_lb=50, P=300,
                             top_k=64)
    bad.block_table[0, 3] = bad.P + 5
    bad.valid_lens[2] = bad.max_lb * bad.epb + 1
    return [small, ragged, shared, wide, bad]


@pytest.mark.parametrize("path", ["tensor", "simt"])
def test_debug_bounds_build_flags_nothing_and_matches(debug_lib, path):
    from sparse_attention_top_paged_gb300 import _lib
    import sparse_attention_top_paged_gb300 as idx
    regular = _lib.load_library()
    for W in _debug_cases():
        d = to_device(W)
        ref = _score_with(regular, W, d, path)
        got = _score_with(debug_lib, W, d, path)
        assert got[3] & idx.STATUS_DEBUG_BOUNDS == 0, (W.name, got[3])
        assert got[3] == ref[3], W.name
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1].view(np.uint32), ref[1].view(np.uint32))
        assert np.array_equal(got[2].view(np.uint32), ref[2].view(np.uint32)), W.name


def test_debug_bounds_build_gathers(debug_lib):
    """The gathers through the debug-bounds build, with bad positions and
    table entries in the mix: no index check fires, bytes as the regular
    build."""
    import sparse_attention_top_paged_gb300 as idx
    from sparse_attention_top_paged_gb300 import _lib
    rng = np.random.default_rng(76)
    kc = torch.from_numpy(rng.integers(0, 65536, size=(8, 16, 4, 128), dtype=np.uint16).view(np.int16)).cuda()
    table = torch.from_numpy(np.array([[3, 1, 7, -1, 2, 0, 5, 9]], dtype=np.int32)).cuda()
    sel = torch.from_numpy(rng.integers(-2, 140, size=(1, 96)).astype(np.int32)).cuda()
    outs = []
    for lib in (_lib.load_library(), debug_lib):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        k_out = torch.empty((1, 96, 4, 128), dtype=torch.int16, device="cuda")
        a = _lib.GatherKvArgs()
        a.T, a.n_sel = 1, 96
        a.sel, a.block_table = sel.data_ptr(), table.data_ptr()
        a.max_logical_blocks, a.bt_stride = 8, 8
        a.P, a.block_size = 8, 16
        a.k_cache, a.v_cache = kc.data_ptr(), None
        a.row_bytes = 4 * 128 * 2
        a.k_out, a.v_out = k_out.data_ptr(), None
        a.dev_status = st.data_ptr()
        assert lib.idx_gather_kv(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
        torch.cuda.synchronize()
        outs.append((k_out.cpu().numpy(), int(st.item())))
    assert outs[1][1] & idx.STATUS_DEBUG_BOUNDS == 0
    assert outs[0][1] == outs[1][1] and outs[0][1] != 0      # bad entries reported by both
    assert np.array_equal(outs[0][0], outs[1][0])
