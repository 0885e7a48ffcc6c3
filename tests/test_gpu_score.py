"""GPU parity of idx_score_topk against the float64 oracle (through the C ABI).

Both score paths run: "simt" (CUDA cores, full score rows + row selection) and
"tensor" (tcgen05 tensor cores writing score rows and a per-row score
histogram, then the histogram-guided row selection). Small cases
compare every output with the oracle; the full-size workloads compare every
returned entry of sampled queries, in the launch configuration the benchmark
times.
"""

import numpy as np
import pytest

import oracle
from sparse_attention_top_paged_gb300 import workloads as wl
from tests.gpu_common import (check_against_oracle, ensure_built, oracle_rows, oracle_rows_parallel, run_gpu,
                              to_device)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PATHS = ["simt", "tensor"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("jitter", [0, 2])
def test_tiny_decode(path, jitter):
    W = wl.tiny_decode(1000 + jitter, gscale_pow2_jitter=jitter)
    gi, gs, st, so = run_gpu(W, path, scores=True)
    rows, ost = oracle_rows(W)
    assert st == ost == 0
    check_against_oracle(W, gi, gs, rows, so, f"tiny/{path}")


def _small(seed, T=8, lo=1, hi=6000, H=64, k=128, P=1024, max_lb=100, q_bf16=True):
    rng = np.random.default_rng(seed)
    vl = rng.integers(lo, hi + 1, size=T)
    return wl.decode_workload("small", seed, T=T, H=H, valid_lens=vl, max_lb=max_lb, P=P,
                              top_k=k, q_bf16=q_bf16)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_small_batched(path, seed):
    W = _small(seed, q_bf16=(seed != 3))
    gi, gs, st, so = run_gpu(W, path, scores=True)
    rows, _ = oracle_rows(W)
    assert st == 0
    check_against_oracle(W, gi, gs, rows, so, f"small{seed}/{path}")


@pytest.mark.parametrize("path", PATHS)
def test_ragged_lengths(path):
    k = 200
    lens = [0, 1, 15, 16, 63, 64, 65, 127, 128, 129, 199, 200, 201, 1000, 2047, 4095]
    W = wl.decode_workload("ragged", 77, T=len(lens), H=64, valid_lens=lens, max_lb=64, P=1100, top_k=k)
    gi, gs, st, so = run_gpu(W, path, scores=True)
    rows, _ = oracle_rows(W)
    assert st == 0
    check_against_oracle(W, gi, gs, rows, so, f"ragged/{path}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("k", [1, 4096])
def test_k_extremes(path, k):
    W = _small(40 + k, T=4, lo=3000, hi=9000, k=k, max_lb=150, P=700)
    gi, gs, st, _ = run_gpu(W, path)
    rows, _ = oracle_rows(W)
    check_against_oracle(W, gi, gs, rows, None, f"k{k}/{path}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("H", [1, 12, 200, 256])
def test_head_counts(path, H):
    W = _small(90 + H, T=3, lo=500, hi=3000, H=H, k=64, max_lb=50, P=200)
    gi, gs, st, so = run_gpu(W, path, scores=True)
    rows, _ = oracle_rows(W)
    check_against_oracle(W, gi, gs, rows, so, f"H{H}/{path}")


@pytest.mark.parametrize("path", PATHS)
def test_shared_table_rows(path):
    W = wl.prefill(5, rows=96, base=4000, ratio=4, n_blocks=24, top_k=256)
    gi, gs, st, so = run_gpu(W, path, scores=True)
    rows, _ = oracle_rows(W)
    check_against_oracle(W, gi, gs, rows, so, f"shared/{path}")


@pytest.mark.parametrize("path", PATHS)
def test_all_equal_scores_take_lowest_indices(path):
    W = _small(7, T=3, lo=700, hi=900, k=300, max_lb=20, P=64)
    W.keys_fp4[:] = 0                      # every key decodes to zero -> every score is exactly 0
    gi, gs, st, _ = run_gpu(W, path)
    assert np.array_equal(gi, np.tile(np.arange(300), (3, 1)))
    assert np.all(gs == 0.0) and not np.any(np.signbit(gs))


@pytest.mark.parametrize("path", PATHS)
def test_all_equal_scores_long_rows(path):
    """Rows past the short-row sort where every score ties: the boundary bin
    holds every key, so the selection refines digit by digit on the row."""
    W = _small(17, T=2, lo=5000, hi=6000, k=300, max_lb=100, P=200)
    W.keys_fp4[:] = 0
    gi, gs, st, _ = run_gpu(W, path)
    assert np.array_equal(gi, np.tile(np.arange(300), (2, 1)))
    assert np.all(gs == 0.0) and not np.any(np.signbit(gs))


def _long_rows(seed, T, lo, hi, k, P):
    return _small(seed, T=T, lo=lo, hi=hi, k=k, max_lb=(hi + 63) // 64, P=P)


def test_split_collection_long_rows():
    """Few rows of 64K+ keys: several CTAs per row collect the candidates
    before the selection orders them."""
    W = _long_rows(18, T=3, lo=65536, hi=90000, k=512, P=4400)
    gi, gs, st, _ = run_gpu(W, "tensor")
    assert st == 0
    rows, _ = oracle_rows(W)
    check_against_oracle(W, gi, gs, rows, None, "split")


def test_split_collection_falls_back_and_takes_all():
    """Row 0: every score ties, so no candidate list is made and the selection
    refines on the row itself. Row 1: most blocks are bad, fewer valid keys
    than k remain, all of them taken from the list."""
    W = _long_rows(19, T=2, lo=70000, hi=70000, k=700, P=2300)
    nblk = (70000 + 63) // 64
    W.keys_fp4[W.block_table[0, :nblk]] = 0
    W.block_table[1, 10:nblk] = -1
    gi, gs, st, _ = run_gpu(W, "tensor")
    rows, ost = oracle_rows(W)
    assert st == ost == oracle.STATUS_BAD_BLOCK
    assert np.array_equal(gi[0], np.arange(700)) and np.all(gs[0] == 0.0)
    check_against_oracle(W, gi, gs, {1: rows[1]}, None, "split-take-all")
    assert np.all(gi[1, 640:] == -1) and np.all(np.isneginf(gs[1, 640:]))


def _scaled_copies(W, n_var, high_per_100=100):
    """Every key of the pool a copy of one key (one global scale for all
    blocks) whose eight E4M3 group scales are set to one code: code 0x30 + 2 v
    (v = slot % n_var) for high_per_100 of every 100 pool slots, else 0x08.
    Scores are then that key's score times the scale (the ReLU'd sum is
    positively homogeneous), so each variant's keys tie exactly and variants
    about 20 % apart fall in distinct 12-bit bins."""
    D2 = W.keys_fp4.shape[2]
    flat_k = W.keys_fp4.reshape(-1, D2)
    flat_s = W.key_scale.reshape(-1, W.key_scale.shape[2])
    g = np.arange(flat_k.shape[0])
    flat_k[:] = flat_k[0]
    code = np.where(g % 100 < high_per_100, 0x30 + 2 * (g % n_var), 0x08).astype(np.uint8)
    flat_s[:] = code[:, None]
    W.key_gscale[:] = W.key_gscale[0]
    return W


@pytest.mark.parametrize("n_var", [12, 28])
def test_many_tied_keys_in_few_bins(n_var):
    """4 rows of 6000 keys, k = 2048, 12 or 28 distinct scores: the candidates
    fill 5 or 10 bins of 200-500 keys, ordered by the rows' two CTAs, or, past
    eight such bins, by the first CTA alone (one sort of the buffer)."""
    W = _scaled_copies(_small(21, T=4, lo=6000, hi=6000, k=2048, max_lb=94, P=1024), n_var)
    gi, gs, st, _ = run_gpu(W, "tensor")
    assert st == 0
    rows, _ = oracle_rows(W)
    assert len(np.unique(rows[0])) == n_var
    check_against_oracle(W, gi, gs, rows, None, f"tied{n_var}")


@pytest.mark.parametrize("n_var,high", [(14, 4), (28, 100)])
def test_many_tied_keys_long_rows(n_var, high):
    """3 rows of 70000 keys, k = 2048: 14 high scores on 4 % of the keys (about
    ten bins of ~200 tied keys among the candidates: the collected list ordered
    by the first of a row's four CTAs alone), or 28 scores over all keys (a
    boundary bin past 2048 keys, refined on later digits)."""
    W = _scaled_copies(_long_rows(22, T=3, lo=70000, hi=70000, k=2048, P=3400), n_var, high)
    gi, gs, st, _ = run_gpu(W, "tensor")
    assert st == 0
    rows, _ = oracle_rows(W)
    check_against_oracle(W, gi, gs, rows, None, f"tied-long{n_var}")


@pytest.mark.parametrize("path", PATHS)
def test_bad_inputs_report_status(path):
    W = _small(8, T=4, lo=2000, hi=3000, k=64, max_lb=50, P=300)
    W.block_table[0, 3] = W.P + 5          # query 0 loses keys 192..255
    W.block_table[1, 0] = -3               # query 1 loses keys 0..63
    W.valid_lens[2] = W.max_lb * W.epb + 1  # query 2: bad length -> padding
    W.valid_lens[3] = -1                   # query 3: bad length -> padding
    gi, gs, st, so = run_gpu(W, path, scores=True)
    rows, ost = oracle_rows(W)
    assert st == ost == (oracle.STATUS_BAD_BLOCK | oracle.STATUS_BAD_LEN)
    for t in (0, 1):
        check_against_oracle(W, gi, gs, {t: rows[t]}, so, f"bad/{path}")
    for t in (2, 3):
        assert np.all(gi[t] == -1) and np.all(np.isneginf(gs[t]))


@pytest.mark.parametrize("path", PATHS)
def test_block_permutation_is_bit_exact(path):
    W = _small(9, T=4, lo=3000, hi=5000, k=100, max_lb=80, P=400)
    gi0, gs0, _, _ = run_gpu(W, path)
    pi = np.random.default_rng(1).permutation(W.P)
    W2 = wl.ScoreWorkload("perm", W.q, W.w, pi[W.block_table].astype(np.int32), W.bt_stride,
                          W.valid_lens, W.epb, W.top_k)
    W2.keys_fp4 = np.empty_like(W.keys_fp4); W2.keys_fp4[pi] = W.keys_fp4
    W2.key_scale = np.empty_like(W.key_scale); W2.key_scale[pi] = W.key_scale
    W2.key_gscale = np.empty_like(W.key_gscale); W2.key_gscale[pi] = W.key_gscale
    gi1, gs1, _, _ = run_gpu(W2, path)
    assert np.array_equal(gi0, gi1) and np.array_equal(gs0.view(np.uint32), gs1.view(np.uint32))


def test_paths_agree_on_scores():
    W = _small(10, T=4, lo=2000, hi=4000, k=128)
    _, _, _, so_s = run_gpu(W, "simt", scores=True)
    _, _, _, so_t = run_gpu(W, "tensor", scores=True)
    rows, _ = oracle_rows(W)
    for t, I in rows.items():
        tol = 1e-3 * np.max(np.abs(I))
        assert np.all(np.abs(so_s[t, :len(I)] - so_t[t, :len(I)]) <= tol)


@pytest.mark.parametrize("num_ctas", [1, 7, 300])
def test_tensor_partition_independent(num_ctas):
    W = _small(11, T=6, lo=1000, hi=20000, k=256, max_lb=320, P=2000)
    gi0, gs0, _, _ = run_gpu(W, "tensor")
    gi1, gs1, _, _ = run_gpu(W, "tensor", num_ctas=num_ctas)
    assert np.array_equal(gi0, gi1) and np.array_equal(gs0, gs1)


def test_repeated_calls_are_identical():
    W = _small(12, T=5, lo=3000, hi=8000, k=256, max_lb=130, P=700)
    d = to_device(W)
    a = run_gpu(W, "auto", dev=d)
    b = run_gpu(W, "auto", dev=d)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_f32_keys_qsa_scores():
    """F32 key format (QSA pooled keys) with w = 1/sqrt(hd): qsa_score."""
    rng = np.random.default_rng(13)
    nb, hd, nh = 512, 128, 32
    keys = rng.standard_normal((nb, hd)).astype(np.float32)
    q = rng.standard_normal((1, nh, hd)).astype(np.float32)
    w = np.full((1, nh), 1.0 / np.sqrt(hd), np.float32)
    W = wl.ScoreWorkload("qsa_score", q, w, np.arange(8, dtype=np.int32).reshape(1, 8), 8,
                         np.array([nb], np.int32), 64, 64, keys_f32=keys.reshape(8, 64, hd))
    gi, gs, st, so = run_gpu(W, "auto", scores=True)
    ref = oracle.qsa_score(q[0], keys)
    from tests.parity import check_query, check_scores_row
    check_query(ref, gi[0], gs[0], 64, where="qsa")
    check_scores_row(ref, so[0], where="qsa")
    import sparse_attention_top_paged_gb300 as idx
    with pytest.raises(idx.IndexerError):
        run_gpu(W, "tensor")


# ----------------------------------------------- full-size workloads ----

@pytest.mark.parametrize("path", ["tensor", "simt"])
def test_batched_decode_full(path):
    """Every one of the 64 queries of the benchmark's batch."""
    W = wl.batched_decode()
    gi, gs, st, _ = run_gpu(W, path)
    assert st == 0
    rows, _ = oracle_rows(W)
    check_against_oracle(W, gi, gs, rows, None, f"batched/{path}")


def test_long_decode_full():
    """Every one of the 16 queries of 262,144 keys (the oracle runs in
    parallel processes)."""
    W = wl.long_decode()
    gi, gs, st, _ = run_gpu(W, "auto")
    assert st == 0
    rows = oracle_rows_parallel("long_decode", W.meta["seed"], range(W.T))
    check_against_oracle(W, gi, gs, rows, None, "long")


def prefill_sample_rows(T=4096, seed=3):
    """The first and last 64 rows of the prefill batch and 128 seeded rows
    between them."""
    rng = np.random.default_rng(seed)
    middle = rng.choice(np.arange(64, T - 64), size=128, replace=False)
    return sorted(set(range(64)) | set(range(T - 64, T)) | set(int(x) for x in middle))


def test_prefill_full():
    W = wl.prefill()
    gi, gs, st, _ = run_gpu(W, "auto")
    assert st == 0
    sample = prefill_sample_rows(W.T)
    assert len(sample) == 256
    rows, _ = oracle_rows(W, rows=sample)
    check_against_oracle(W, gi, gs, rows, None, "prefill")


def _garbage(ws, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    ws.copy_(torch.randint(0, 256, (ws.numel(),), dtype=torch.uint8, generator=g))


@pytest.mark.parametrize("case", ["batched", "split"])
def test_workspace_needs_no_initialisation(case):
    """The workspace may hold anything before a call: every call writes each
    scratch word before reading it (score rows, q records, histograms and
    the split collection's candidate counters). Two calls in a row, each on a
    freshly garbage-filled workspace."""
    import sparse_attention_top_paged_gb300 as idx
    if case == "batched":
        W = _small(51, T=8, lo=3000, hi=9000, k=256, max_lb=150, P=1300)
    else:   # few rows of 64K+ keys: the selection's split collection runs
        W = _long_rows(52, T=3, lo=65536, hi=80000, k=512, P=3800)
    d = to_device(W)
    out = (torch.empty((W.T, W.top_k), dtype=torch.int32, device="cuda"),
           torch.empty((W.T, W.top_k), dtype=torch.float32, device="cuda"))
    a = idx.make_score_args(d["q"], d["w"], d["bt"], d["vl"], W.top_k, entries_per_block=W.epb,
                            keys_fp4=d["keys_fp4"], key_scale=d["key_scale"], key_gscale=d["key_gscale"],
                            bt_stride=W.bt_stride, topk_idx=out[0], topk_score=out[1], path="tensor")
    ws = torch.empty(idx.score_topk_workspace_bytes(a), dtype=torch.uint8, device="cuda")
    rows, _ = oracle_rows(W)
    for rep in range(2):
        _garbage(ws, 100 + rep)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        gi, gs = idx.score_topk(d["q"], d["w"], d["bt"], d["vl"], W.top_k, entries_per_block=W.epb,
                                bt_stride=W.bt_stride, keys_fp4=d["keys_fp4"], key_scale=d["key_scale"],
                                key_gscale=d["key_gscale"], dev_status=st, path="tensor", workspace=ws, out=out)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        check_against_oracle(W, gi.cpu().numpy(), gs.cpu().numpy(), rows, None, f"garbage-ws/{case}/{rep}")


def test_tensor_more_ctas_than_tiles():
    """Fewer 128-key tiles than CTAs: empty CTAs sit inside query ranges."""
    W = _small(14, T=3, lo=100, hi=300, k=64, max_lb=8, P=40)
    for g in (152, 400):
        gi, gs, st, so = run_gpu(W, "tensor", scores=True, num_ctas=g)
        rows, _ = oracle_rows(W)
        check_against_oracle(W, gi, gs, rows, so, f"sparse-tiles/{g}")


@pytest.mark.parametrize("num_ctas", [0, 5])
def test_tensor_many_short_queries(num_ctas):
    """Hundreds of short queries: many segments per CTA cycle both segment slots."""
    W = _small(15, T=300, lo=0, hi=700, k=32, max_lb=11, P=3400)
    gi, gs, st, so = run_gpu(W, "tensor", scores=True, num_ctas=num_ctas)
    rows, _ = oracle_rows(W)
    check_against_oracle(W, gi, gs, rows, so, f"short/{num_ctas}")


def test_prepared_plan_matches_the_call():
    """ScoreTopkPlan: arguments marshalled once, run over refilled inputs."""
    import sparse_attention_top_paged_gb300 as idx
    W1 = _small(101, T=6, lo=2000, hi=7000, k=128, max_lb=120, P=800)
    W2 = _small(102, T=6, lo=2000, hi=7000, k=128, max_lb=120, P=800)
    d = to_device(W1)
    plan = idx.ScoreTopkPlan(d["q"], d["w"], d["bt"], d["vl"], W1.top_k, entries_per_block=W1.epb,
                             bt_stride=W1.bt_stride, keys_fp4=d["keys_fp4"], key_scale=d["key_scale"],
                             key_gscale=d["key_gscale"])
    for W in (W1, W2):
        dW = to_device(W)
        for name in ("q", "w", "bt", "vl", "keys_fp4", "key_scale", "key_gscale"):
            d[name].copy_(dW[name])          # refill the bound tensors in place
        gi, gs = plan.run()
        torch.cuda.synchronize()
        ref = run_gpu(W, "tensor")
        assert np.array_equal(gi.cpu().numpy(), ref[0]) and np.array_equal(gs.cpu().numpy(), ref[1])
        rows, _ = oracle_rows(W)
        check_against_oracle(W, gi.cpu().numpy(), gs.cpu().numpy(), rows, None, f"plan/{W.meta['seed']}")


def test_captured_plan_step_with_copies():
    """ScoreTopkPlan.capture: the step's host-to-device copies, the call and the
    copies back as one CUDA graph, replayed over pinned host buffers refilled
    in place; every replay equals a direct call on the same inputs."""
    import sparse_attention_top_paged_gb300 as idx
    Ws = [_small(121 + i, T=6, lo=2000, hi=7000, k=128, max_lb=120, P=800) for i in range(3)]
    d = to_device(Ws[0])
    names = ("q", "w", "bt", "vl")
    host = {n: d[n].cpu().pin_memory() for n in names}
    plan = idx.ScoreTopkPlan(d["q"], d["w"], d["bt"], d["vl"], Ws[0].top_k, entries_per_block=Ws[0].epb,
                             bt_stride=Ws[0].bt_stride, keys_fp4=d["keys_fp4"], key_scale=d["key_scale"],
                             key_gscale=d["key_gscale"])
    hi = torch.empty(plan.topk_idx.shape, dtype=torch.int32).pin_memory()
    hs = torch.empty(plan.topk_score.shape, dtype=torch.float32).pin_memory()

    def before():
        for n in names:
            d[n].copy_(host[n], non_blocking=True)

    def after():
        hi.copy_(plan.topk_idx, non_blocking=True)
        hs.copy_(plan.topk_score, non_blocking=True)

    graph = plan.capture(before, after)
    for W in Ws[1:] + Ws[:1]:
        dW = to_device(W)
        for name in ("keys_fp4", "key_scale", "key_gscale"):
            d[name].copy_(dW[name])
        for n in names:
            host[n].copy_(dW[n].cpu())
        graph.replay()
        torch.cuda.synchronize()
        ref = run_gpu(W, "tensor")
        assert np.array_equal(hi.numpy(), ref[0]) and np.array_equal(hs.numpy(), ref[1])


@pytest.mark.parametrize("q_format", ["exact", "nvfp4"])
@pytest.mark.parametrize("case", ["batched", "pairs"])
def test_bf16_queries_equal_their_float32_upcast(q_format, case):
    """q given as bf16 (q_dtype BF16) gives exactly what its float32 upcast
    gives, on the tensor path; the CUDA-core path refuses it."""
    import sparse_attention_top_paged_gb300 as idx
    if case == "batched":
        W = _small(111, T=6, lo=2000, hi=7000, k=128, max_lb=120, P=800)
    else:
        W = wl.prefill(8, rows=40, base=3000, ratio=4, n_blocks=20, top_k=128)
    d = to_device(W)
    q16 = d["q"].to(torch.bfloat16)
    assert torch.equal(q16.float(), d["q"])      # the workloads' q values are bf16
    kw = dict(entries_per_block=W.epb, bt_stride=W.bt_stride, keys_fp4=d["keys_fp4"], key_scale=d["key_scale"],
              key_gscale=d["key_gscale"], q_format=q_format, path="tensor")
    s32 = torch.full((W.T, W.max_lb * W.epb), float("nan"), dtype=torch.float32, device="cuda")
    s16 = s32.clone()
    i32, v32 = idx.score_topk(d["q"], d["w"], d["bt"], d["vl"], W.top_k, scores_out=s32, **kw)
    i16, v16 = idx.score_topk(q16, d["w"], d["bt"], d["vl"], W.top_k, scores_out=s16, **kw)
    torch.cuda.synchronize()
    assert torch.equal(i32, i16) and torch.equal(v32, v16)
    assert torch.equal(torch.nan_to_num(s32, nan=7.0), torch.nan_to_num(s16, nan=7.0))
    with pytest.raises(idx.IndexerError):
        idx.score_topk(q16, d["w"], d["bt"], d["vl"], W.top_k, **dict(kw, path="simt", q_format="exact"))
