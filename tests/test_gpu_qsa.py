"""GPU parity of the QSA pieces and the K/V gather against the float64 oracle:
idx_block_pool, idx_qsa_qprep, idx_qsa_prefill_attn, idx_gather_kv and idx_gather_split
(bit-exact), idx_expand_blocks (exact),
idx_valid_lens_from_blocks (exact), and the QSA workload end to end
(pool -> score -> top-k -> expand -> gather)."""

import math

import numpy as np
import pytest

import oracle
from sparse_attention_top_paged_gb300 import workloads as wl
from tests.gpu_common import ensure_built
from tests.parity import check_query

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

POOL_REL_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _idx():
    import sparse_attention_top_paged_gb300 as idx
    return idx


def _pool_gpu(Q, first_block, n_new, out=None):
    raw = torch.from_numpy(Q.raw_keys_bits.view(np.int16)).cuda()
    w = torch.from_numpy(Q.k_norm_w).cuda()
    if out is None:
        out = torch.full((Q.n_blocks, raw.shape[1]), float("nan"), device="cuda")
    _idx().block_pool(raw, w, out, first_block, n_new, Q.ratio, Q.rot, Q.theta, Q.eps)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_block_pool_all_blocks():
    Q = wl.qsa()
    got = _pool_gpu(Q, 0, Q.n_blocks)
    ref = oracle.block_pool(Q.raw_keys, Q.k_norm_w, 0, Q.n_blocks, Q.ratio, Q.rot, Q.theta, Q.eps)
    tol = POOL_REL_TOL * np.max(np.abs(ref))
    assert np.max(np.abs(got - ref)) <= tol


@pytest.mark.parametrize("rows,first_pos,extra", [(1, 131071, 0), (7, 1000, 256)])
def test_qsa_qprep_rows(rows, first_pos, extra):
    """Query preparation: one decode query at a far position, and prefill
    rows read from a wider projection (extra columns after the q heads)."""
    rng = np.random.default_rng(20 + rows)
    nh, hd, rot, theta, eps = 32, 128, 64, 1e6, 1e-6
    qkw = nh * hd + extra
    x = rng.standard_normal((rows, qkw)).astype(np.float32)
    bits = wl._to_bf16_bits(x)
    vals = wl._to_bf16_values(x)
    w = (rng.standard_normal(hd) * 0.1).astype(np.float32)
    got = _idx().qsa_qprep(torch.from_numpy(bits.view(np.int16)).cuda(), torch.from_numpy(w).cuda(), nh, rot,
                           theta, eps, first_pos=first_pos).cpu().numpy()
    ref = oracle.qsa_qprep_rows(vals, w, rows, first_pos, qkw, nh, hd, rot, theta, eps)
    assert got.shape == (rows, nh, hd)
    assert np.max(np.abs(got - ref)) <= POOL_REL_TOL * np.max(np.abs(ref))


def test_block_pool_incremental_rows_only():
    Q = wl.qsa(seed=7)
    got = _pool_gpu(Q, 100, 7)
    ref = oracle.block_pool(Q.raw_keys, Q.k_norm_w, 100, 7, Q.ratio, Q.rot, Q.theta, Q.eps)
    assert np.max(np.abs(got[100:107] - ref)) <= POOL_REL_TOL * np.max(np.abs(ref))
    assert np.all(np.isnan(got[:100])) and np.all(np.isnan(got[107:]))
    got0 = _pool_gpu(Q, 3, 0)                     # n_new == 0 launches nothing
    assert np.all(np.isnan(got0))


def _gather_case(seed=3, T=3, n=200, P=40, bs=16, nkv=4, hd=128):
    rng = np.random.default_rng(seed)
    kc = rng.integers(0, 65536, size=(P, bs, nkv, hd), dtype=np.uint16)
    vc = rng.integers(0, 65536, size=(P, bs, nkv, hd), dtype=np.uint16)
    max_lb = 12
    table = np.stack([rng.permutation(P)[:max_lb] for _ in range(T)]).astype(np.int32)
    sel = rng.integers(0, max_lb * bs, size=(T, n)).astype(np.int32)
    sel[0, :5] = -1
    return kc, vc, table, sel, bs, max_lb


def _gather_gpu(kc, vc, table, sel, bs, with_v=True):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k_out, v_out = _idx().gather_kv(torch.from_numpy(sel).cuda(), torch.from_numpy(table).cuda(), bs,
                                    torch.from_numpy(kc.view(np.int16)).cuda(),
                                    torch.from_numpy(vc.view(np.int16)).cuda() if with_v else None,
                                    dev_status=st)
    torch.cuda.synchronize()
    return (k_out.cpu().numpy().view(np.uint16),
            None if v_out is None else v_out.cpu().numpy().view(np.uint16), int(st.item()))


def test_gather_bit_exact():
    kc, vc, table, sel, bs, max_lb = _gather_case()
    k, v, st = _gather_gpu(kc, vc, table, sel, bs)
    rk, rv, rst = oracle.gather_kv(sel, table, max_lb, max_lb, bs, kc, vc)
    assert st == rst == 0
    assert np.array_equal(k, rk) and np.array_equal(v, rv)


def test_gather_bad_rows_and_k_only():
    kc, vc, table, sel, bs, max_lb = _gather_case(seed=4)
    sel[1, 7] = max_lb * bs + 3        # logical block past the table
    table[2, 0] = kc.shape[0] + 1      # physical block out of range
    sel[2, :4] = [0, 1, 2, 15]         # ... and positions that use it
    k, v, st = _gather_gpu(kc, vc, table, sel, bs)
    rk, rv, rst = oracle.gather_kv(sel, table, max_lb, max_lb, bs, kc, vc)
    assert st == rst == (oracle.STATUS_BAD_SEL | oracle.STATUS_BAD_BLOCK)
    assert np.array_equal(k, rk) and np.array_equal(v, rv)
    k2, v2, _ = _gather_gpu(kc, vc, table, sel, bs, with_v=False)
    assert v2 is None and np.array_equal(k2, rk)


@pytest.mark.parametrize("nb", [1, 64, 256, 257, 1000])
def test_expand_blocks_exact(nb):
    """Up to 256 selected blocks (one thread ranks each id) and more (a sorting
    network), with unselected (-1) entries and repeated ids."""
    rng = np.random.default_rng(5 + nb)
    blocks = np.stack([rng.permutation(4 * nb)[:nb] for _ in range(3)]).astype(np.int32)
    blocks[1, nb // 6:] = -1
    blocks[2, : nb // 2] = blocks[2, nb // 2: 2 * (nb // 2)]   # each id of the second half twice
    got = _idx().expand_blocks(torch.from_numpy(blocks).cuda(), 16).cpu().numpy()
    assert np.array_equal(got, oracle.expand_blocks(blocks, 16))


def test_valid_lens_exact():
    bl = np.array([0, 1, 7, 4096], np.int32)
    got = _idx().valid_lens_from_blocks(torch.from_numpy(bl).cuda(), 64).cpu().numpy()
    assert np.array_equal(got, oracle.valid_lens_from_blocks(bl, 64))


def test_qsa_end_to_end():
    """The QSA workload: pool 8192 raw keys in blocks of 16, score the 512
    block keys with 32 heads (w = 1/sqrt(128)), keep the top 64 blocks,
    expand to 1024 positions and gather K/V (4 kv heads, 16-token pages)."""
    Q = wl.qsa()
    idx = _idx()
    hd = Q.raw_keys.shape[1]
    raw = torch.from_numpy(Q.raw_keys_bits.view(np.int16)).cuda()
    bk = torch.empty((Q.n_blocks, hd), device="cuda")
    idx.block_pool(raw, torch.from_numpy(Q.k_norm_w).cuda(), bk, 0, Q.n_blocks, Q.ratio, Q.rot, Q.theta, Q.eps)
    nb = Q.n_blocks
    q = torch.from_numpy(Q.q[None]).cuda()
    w = torch.full((1, Q.q.shape[0]), 1.0 / math.sqrt(hd), device="cuda")
    table = torch.arange(nb // 64, dtype=torch.int32, device="cuda").reshape(1, -1)
    gi, gs = idx.score_topk(q, w, table, torch.tensor([nb], dtype=torch.int32, device="cuda"), Q.top_k,
                            entries_per_block=64, keys_f32=bk.reshape(nb // 64, 64, hd))
    pos = idx.expand_blocks(gi, Q.ratio)
    kc = torch.from_numpy(Q.k_cache_bits.view(np.int16)).cuda()
    vc = torch.from_numpy(Q.v_cache_bits.view(np.int16)).cuda()
    k_out, v_out = idx.gather_kv(pos, torch.from_numpy(Q.page_table).cuda(), Q.block_size, kc, vc)
    torch.cuda.synchronize()

    ref_keys = oracle.block_pool(Q.raw_keys, Q.k_norm_w, 0, nb, Q.ratio, Q.rot, Q.theta, Q.eps)
    ref_scores = oracle.qsa_score(Q.q, ref_keys)
    gi_np, gs_np = gi.cpu().numpy(), gs.cpu().numpy()
    check_query(ref_scores, gi_np[0], gs_np[0], Q.top_k, where="qsa e2e")
    pos_np = pos.cpu().numpy()
    assert np.array_equal(pos_np, oracle.expand_blocks(gi_np, Q.ratio))
    rk, rv, st = oracle.gather_kv(pos_np, Q.page_table, Q.page_table.shape[1], Q.page_table.shape[1],
                                  Q.block_size, Q.k_cache_bits, Q.v_cache_bits)
    assert st == 0
    assert np.array_equal(k_out.cpu().numpy().view(np.uint16), rk)
    assert np.array_equal(v_out.cpu().numpy().view(np.uint16), rv)


def _attn_case(seed, hd, nq, nkv, rows=6, first_pos=3000, ratio=16, bs=16, topk=64, bad_page=None):
    rng = np.random.default_rng(seed)
    n_tok = first_pos + rows + 50
    pages = (n_tok + bs - 1) // bs
    P = pages + 3
    kbits = wl._to_bf16_bits(rng.standard_normal((P, bs, nkv, hd)).astype(np.float32))
    vbits = wl._to_bf16_bits(rng.standard_normal((P, bs, nkv, hd)).astype(np.float32))
    table = rng.permutation(P)[:pages].astype(np.int32)
    if bad_page is not None:
        table[bad_page] = -1
    lists = np.stack([rng.integers(-1, (first_pos + r + 1) // ratio + 3, size=topk) for r in range(rows)])
    lists = lists.astype(np.int32)
    q = rng.standard_normal((rows, nq, hd)).astype(np.float32)
    return q, kbits, vbits, table, lists, first_pos, ratio


def _attn_gpu(q, kbits, vbits, table, lists, first_pos, ratio):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _idx().qsa_prefill_attn(torch.from_numpy(q).cuda(), torch.from_numpy(kbits.view(np.int16)).cuda(),
                                  torch.from_numpy(vbits.view(np.int16)).cuda(), torch.from_numpy(table).cuda(),
                                  torch.from_numpy(lists).cuda(), first_pos, ratio, dev_status=st)
    return got.cpu().numpy(), int(st.item())


def _bf16_vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("hd,nq,nkv", [(128, 32, 4), (64, 8, 8), (256, 4, 1), (64, 4, 2), (128, 16, 4),
                                       (64, 16, 2), (128, 4, 2), (128, 4, 4), (64, 8, 2), (128, 6, 2)])
def test_qsa_prefill_attn(hd, nq, nkv):
    """Prefill rows over 64 listed blocks (some invalid or incomplete, i.e.
    skipped) plus their tails: 1, 2, 3, 4 and 8 query heads per kv head,
    three head sizes."""
    q, kb, vb, table, lists, fp, ratio = _attn_case(30 + hd, hd, nq, nkv)
    got, st = _attn_gpu(q, kb, vb, table, lists, fp, ratio)
    ref, ost = oracle.qsa_prefill_attn(q, _bf16_vals(kb), _bf16_vals(vb), table, lists, fp, ratio,
                                       1.0 / math.sqrt(hd))
    assert st == ost == 0
    assert np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref))


def _at_8_past_16(bits):
    """The cache as a device tensor starting 8 bytes past a 16-byte boundary."""
    flat = torch.zeros(bits.size + 4, dtype=torch.int16, device="cuda")
    flat[4:] = torch.from_numpy(bits.view(np.int16).reshape(-1)).cuda()
    t = flat[4:].view(bits.shape)
    assert t.data_ptr() % 16 == 8
    return t


@pytest.mark.parametrize("which", ["k", "v"])
def test_qsa_prefill_attn_cache_8_byte_aligned(which):
    """A K or V cache that starts 8 bytes past a 16-byte boundary (the
    per-head kernel's 8-byte loads instead of the tiled kernel's 16-byte
    copies) gives the same attention."""
    q, kb, vb, table, lists, fp, ratio = _attn_case(77, 128, 16, 2)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc = _at_8_past_16(kb) if which == "k" else torch.from_numpy(kb.view(np.int16)).cuda()
    vc = _at_8_past_16(vb) if which == "v" else torch.from_numpy(vb.view(np.int16)).cuda()
    got = _idx().qsa_prefill_attn(torch.from_numpy(q).cuda(), kc, vc, torch.from_numpy(table).cuda(),
                                  torch.from_numpy(lists).cuda(), fp, ratio, dev_status=st)
    ref, ost = oracle.qsa_prefill_attn(q, _bf16_vals(kb), _bf16_vals(vb), table, lists, fp, ratio,
                                       1.0 / math.sqrt(128))
    assert int(st.item()) == ost == 0
    assert np.max(np.abs(got.cpu().numpy() - ref)) <= 1e-4 * np.max(np.abs(ref))


@pytest.mark.parametrize("scale,topk,ratio,first_pos", [(6.0, 64, 16, 3000), (6.0, 300, 4, 2000), (1.0, 5, 16, 700),
                                                        (12.0, 129, 8, 1200), (0.0, 64, 16, 3000)])
def test_qsa_prefill_attn_tensor_core_tiles(scale, topk, ratio, first_pos):
    """8 query heads per kv head at hd 128 (the tcgen05 kernel's 128-token
    tiles): peaked scores that move the lazy reference maximum between tiles,
    up to 10 tiles a row with a ragged last tile, a single partial tile, and
    constant scores (q = 0: plain means of V)."""
    q, kb, vb, table, lists, fp, ratio = _attn_case(90 + topk, 128, 32, 4, rows=7, first_pos=first_pos,
                                                    ratio=ratio, topk=topk)
    q = (q * scale).astype(np.float32)
    got, st = _attn_gpu(q, kb, vb, table, lists, fp, ratio)
    ref, ost = oracle.qsa_prefill_attn(q, _bf16_vals(kb), _bf16_vals(vb), table, lists, fp, ratio,
                                       1.0 / math.sqrt(128))
    assert st == ost == 0
    assert np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref))


@pytest.mark.parametrize("nq,hd", [(8, 128), (4, 128), (2, 128), (1, 128), (4, 64)])
def test_qsa_prefill_attn_tail_only_and_empty_rows(nq, hd):
    """No selected blocks (topk = 0): every row attends to its tail alone, and
    a row whose tail is empty (its position completes a block) gives zeros
    (hd 128: the tcgen05 kernel's items without a step; hd 64: the tile
    kernel)."""
    rng = np.random.default_rng(55)
    rows, fp, ratio, bs, nkv = 13, 7, 4, 16, 2
    pages = (fp + rows + bs - 1) // bs
    kb = wl._to_bf16_bits(rng.standard_normal((pages + 1, bs, nkv, hd)).astype(np.float32))
    vb = wl._to_bf16_bits(rng.standard_normal((pages + 1, bs, nkv, hd)).astype(np.float32))
    table = rng.permutation(pages + 1)[:pages].astype(np.int32)
    lists = np.zeros((rows, 0), dtype=np.int32)
    q = rng.standard_normal((rows, nq * nkv, hd)).astype(np.float32)
    got, st = _attn_gpu(q, kb, vb, table, lists, fp, ratio)
    ref, ost = oracle.qsa_prefill_attn(q, _bf16_vals(kb), _bf16_vals(vb), table, lists, fp, ratio,
                                       1.0 / math.sqrt(hd))
    assert st == ost == 0
    empty = [r for r in range(rows) if (fp + r + 1) % ratio == 0]
    assert empty and np.all(got[empty] == 0.0)
    assert np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref))


@pytest.mark.parametrize("nq", [8, 2])
def test_qsa_prefill_attn_tail_only_many_items(nq):
    """Tail-only rows (topk = 0) over more items than SMs: a CTA's items
    alternate between one short step and none (every fourth row's tail is
    empty), so outputs written after a later item, or at the end of an item
    without steps, and both tensor-memory O slots are exercised."""
    rng = np.random.default_rng(56)
    rows, fp, ratio, bs, nkv, hd = 613, 7, 4, 16, 2, 128
    pages = (fp + rows + bs - 1) // bs
    kb = wl._to_bf16_bits(rng.standard_normal((pages + 1, bs, nkv, hd)).astype(np.float32))
    vb = wl._to_bf16_bits(rng.standard_normal((pages + 1, bs, nkv, hd)).astype(np.float32))
    table = rng.permutation(pages + 1)[:pages].astype(np.int32)
    lists = np.zeros((rows, 0), dtype=np.int32)
    q = rng.standard_normal((rows, nq * nkv, hd)).astype(np.float32)
    got, st = _attn_gpu(q, kb, vb, table, lists, fp, ratio)
    ref, ost = oracle.qsa_prefill_attn(q, _bf16_vals(kb), _bf16_vals(vb), table, lists, fp, ratio,
                                       1.0 / math.sqrt(hd))
    assert st == ost == 0
    empty = [r for r in range(rows) if (fp + r + 1) % ratio == 0]
    assert len(empty) > 100 and np.all(got[empty] == 0.0)
    assert np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref))


@pytest.mark.parametrize("nq", [8, 1])
def test_qsa_prefill_attn_one_and_two_step_items(nq):
    """700 rows over 8 listed blocks of 16 tokens: items of one step (rows whose
    tail is empty) and of two, several per CTA, with 8 and 1 q heads per kv
    head; every row against the oracle."""
    q, kb, vb, table, lists, fp, ratio = _attn_case(57 + nq, 128, nq, 1, rows=700, first_pos=1000, topk=8)
    got, st = _attn_gpu(q, kb, vb, table, lists, fp, ratio)
    ref, ost = oracle.qsa_prefill_attn(q, _bf16_vals(kb), _bf16_vals(vb), table, lists, fp, ratio,
                                       1.0 / math.sqrt(128))
    assert st == ost == 0
    assert np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref))


@pytest.mark.parametrize("nq", [16, 8, 4, 2])
@pytest.mark.parametrize("hd", [128, 64])
def test_qsa_prefill_attn_q_4_byte_aligned(nq, hd):
    """q starting 4 bytes past an 8-byte boundary (the tensor-core kernel reads
    q in float pairs, so the 32-token tile kernel serves it) gives the same
    attention, at 8, 4, 2 and 1 q heads per kv head and hd 128 and 64."""
    q, kb, vb, table, lists, fp, ratio = _attn_case(78 + hd, hd, nq, 2)
    flat = torch.zeros(q.size + 1, dtype=torch.float32, device="cuda")
    flat[1:] = torch.from_numpy(q.reshape(-1)).cuda()
    qd = flat[1:].view(q.shape)
    assert qd.data_ptr() % 8 == 4
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _idx().qsa_prefill_attn(qd, torch.from_numpy(kb.view(np.int16)).cuda(), torch.from_numpy(vb.view(np.int16)).cuda(),
                                  torch.from_numpy(table).cuda(), torch.from_numpy(lists).cuda(), fp, ratio, dev_status=st)
    ref, ost = oracle.qsa_prefill_attn(q, _bf16_vals(kb), _bf16_vals(vb), table, lists, fp, ratio, 1.0 / math.sqrt(hd))
    assert int(st.item()) == ost == 0
    assert np.max(np.abs(got.cpu().numpy() - ref)) <= 1e-4 * np.max(np.abs(ref))


@pytest.mark.parametrize("nq,nkv,bs,ratio", [(64, 8, 16, 16), (16, 2, 64, 16), (16, 2, 16, 64), (8, 1, 32, 8),
                                             (32, 8, 16, 16), (8, 2, 64, 16), (4, 1, 32, 8), (16, 8, 16, 16),
                                             (2, 1, 64, 16), (8, 8, 16, 16), (3, 3, 32, 8)])
@pytest.mark.parametrize("hd", [128, 64])
def test_qsa_prefill_attn_tensor_core_geometry(nq, nkv, bs, ratio, hd):
    """The tcgen05 kernel (8, 4, 2 or 1 q heads per kv head, hd 128) and the
    tile kernel (hd 64) over 1, 2, 3 and 8 kv heads, pages of 16, 32 and 64
    tokens and blocks shorter or longer than a page."""
    q, kb, vb, table, lists, fp, ratio = _attn_case(150 + nkv + bs + ratio + hd, hd, nq, nkv, rows=5,
                                                    first_pos=2500, ratio=ratio, bs=bs, topk=48)
    got, st = _attn_gpu(q, kb, vb, table, lists, fp, ratio)
    ref, ost = oracle.qsa_prefill_attn(q, _bf16_vals(kb), _bf16_vals(vb), table, lists, fp, ratio,
                                       1.0 / math.sqrt(hd))
    assert st == ost == 0
    assert np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref))


@pytest.mark.parametrize("nq", [8, 16])
def test_qsa_prefill_attn_missing_page_and_first_rows(nq):
    """A page missing from the table drops its tokens (reported); rows at
    positions 0.. attend to their tails alone (4 and 8 query heads per kv
    head)."""
    q, kb, vb, table, lists, fp, ratio = _attn_case(41, 128, nq, 2, rows=20, first_pos=0, bad_page=0)
    got, st = _attn_gpu(q, kb, vb, table, lists, fp, ratio)
    ref, ost = oracle.qsa_prefill_attn(q, _bf16_vals(kb), _bf16_vals(vb), table, lists, fp, ratio,
                                       1.0 / math.sqrt(128))
    assert st == ost == oracle.STATUS_BAD_BLOCK
    assert np.max(np.abs(got - ref)) <= 1e-4 * max(np.max(np.abs(ref)), 1.0)
    q, kb, vb, table, lists, fp, ratio = _attn_case(42, 128, nq, 2, rows=40, first_pos=0, bad_page=1)
    got, st = _attn_gpu(q, kb, vb, table, lists, fp, ratio)
    ref, ost = oracle.qsa_prefill_attn(q, _bf16_vals(kb), _bf16_vals(vb), table, lists, fp, ratio,
                                       1.0 / math.sqrt(128))
    assert st == ost == oracle.STATUS_BAD_BLOCK
    assert np.max(np.abs(got - ref)) <= 1e-4 * max(np.max(np.abs(ref)), 1.0)


@pytest.mark.parametrize("with_scale", [True, False])
@pytest.mark.parametrize("nd,rd,n", [(512, 64, 200), (512, 64, 201), (36, 6, 101)])
def test_gather_split_bit_exact(with_scale, nd, rd, n):
    """The FP8 + BF16 split gather: dequantised rows bit-exact against the
    oracle, -1 and out-of-table positions zero, a bad table entry reported.
    Full-size rows, an odd row count and a short row whose parts are not
    multiples of 8."""
    rng = np.random.default_rng(50 + with_scale + nd + n)
    P, bs, T, mlb = 40, 16, 3, 32
    codes = rng.integers(0, 256, size=(P, bs, nd)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38                       # no NaN codes
    scale = rng.uniform(0.01, 4.0, size=(P, bs)).astype(np.float32) if with_scale else None
    rope = wl._to_bf16_bits(rng.standard_normal((P, bs, rd)).astype(np.float32))
    table = np.stack([rng.permutation(P)[:mlb] for _ in range(T)]).astype(np.int32)
    table[2, 5] = P + 7
    sel = rng.integers(-1, mlb * bs + 20, size=(T, n)).astype(np.int32)
    sel[2, 0] = 5 * bs + 3                                     # lands in the bad entry
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = lambda x: torch.from_numpy(x).cuda()
    got = _idx().gather_split(d(sel), d(table), bs, d(codes), d(rope.view(np.int16)),
                              d(scale) if with_scale else None, dev_status=st)
    ref, ost = oracle.gather_split(sel, table, mlb, mlb, bs, codes, scale, rope)
    assert int(st.item()) == ost == (oracle.STATUS_BAD_BLOCK | oracle.STATUS_BAD_SEL)
    assert np.array_equal(got.cpu().view(torch.int16).numpy().view(np.uint16), ref)


def _bench():
    import importlib
    import os
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    return importlib.import_module("bench")


def test_qsa_prefill_attn_bench_size_every_row():
    """The benchmark's attention workload (512 rows from position 8192, 64
    selected blocks of 16 tokens plus the tail, 32 q heads over 4 kv heads,
    hd 128) in the launch the benchmark times; every row against the oracle,
    within 1e-4 of the row's largest output."""
    c = _bench().qsa_attn_case(1005)
    got, st = _attn_gpu(c["q"], c["kbits"], c["vbits"], c["table"], c["lists"], c["first_pos"], c["ratio"])
    assert st == 0
    ref, ost = oracle.qsa_prefill_attn(c["q"], _bf16_vals(c["kbits"]), _bf16_vals(c["vbits"]), c["table"],
                                       c["lists"], c["first_pos"], c["ratio"], 1.0 / math.sqrt(c["hd"]))
    assert ost == 0
    err = np.max(np.abs(got - ref), axis=(1, 2))
    scale = np.max(np.abs(ref), axis=(1, 2))
    bad = np.nonzero(err > 1e-4 * scale)[0]
    assert bad.size == 0, (bad[:8], err[bad[:8]], scale[bad[:8]])


def test_gather_split_bench_size_every_query():
    """The benchmark's split-gather workload (64 queries x 2048 positions of a
    262144-token cache) in one launch; every query bit-exact against the
    oracle."""
    c = _bench().gather_split_case(1006)
    d = lambda x: torch.from_numpy(x).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _idx().gather_split(d(c["sel"]), d(c["table"]), c["bs"], d(c["codes"]), d(c["rope"].view(np.int16)),
                              d(c["scale"]), dev_status=st)
    assert int(st.item()) == 0
    got = got.cpu().view(torch.int16).numpy().view(np.uint16)
    ref, ost = oracle.gather_split(c["sel"], c["table"], c["P"], c["P"], c["bs"], c["codes"], c["scale"], c["rope"])
    assert ost == 0
    bad = [t for t in range(c["T"]) if not np.array_equal(got[t], ref[t])]
    assert not bad, bad[:8]
