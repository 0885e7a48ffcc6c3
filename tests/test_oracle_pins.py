"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each ``pin_*`` helper returns True when the oracle agrees with an independent
source: a value the pages print (fixtures under ``tests/golden/``), a library
routine computing the same quantity another way, a closed form, a layout
probe whose answer is known by construction, or an exact invariance. The
mutation tests at the end plant plausible mistakes in the oracle (on the CPU)
and check that some pin then fails.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
import oracle.indexer as oi
from sparse_attention_top_paged_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_table(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b = line.split()
        rows.append((int(a, 0), float(b)))
    return rows


def _load_case(name):
    c = json.load(open(os.path.join(GOLDEN, name)))
    c["expected_score"] = [[-math.inf if v == "-inf" else v for v in r] for r in c["expected_score"]]
    return c


def _run_case(c):
    arr = lambda x, dt: np.asarray(x, dtype=dt)
    idx, sc, status, rows = oracle.score_topk(
        arr(c["q"], np.float32), arr(c["w"], np.float32), arr(c["block_table"], np.int32),
        c["bt_stride"], len(c["block_table"][0]), arr(c["valid_lens"], np.int32), c["epb"], c["k"],
        keys_fp4=arr(c["keys_fp4"], np.uint8), key_scale=arr(c["key_scale"], np.uint8),
        key_gscale=arr(c["key_gscale"], np.float32))
    return idx, sc, status, rows


# ----------------------------------------------------------------- pins ----

def pin_e2m1_printed_table():
    """Oracle E2M1 decode == the table printed in commits 79ef87f / e74c844."""
    tab = _load_table("e2m1_table.txt")
    codes = np.array([c for c, _ in tab])
    want = np.array([v for _, v in tab])
    got = oracle.e2m1_decode(codes)
    return np.array_equal(got, want) and np.array_equal(np.signbit(got), np.signbit(want))


def bitlevel_e2m1(code):
    """Bit-level E2M1 decode as commit 79ef87f describes it (bias 1;
    exponent field 0 is subnormal with 0b001 = 0.5), written without the
    lookup table."""
    sign = -1.0 if code & 8 else 1.0
    e, m = (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return sign * mag


def pin_e2m1_bitlevel():
    got = oracle.e2m1_decode(np.arange(16))
    want = np.array([bitlevel_e2m1(c) for c in range(16)])
    return np.array_equal(got, want)


def pin_e4m3_library():
    """All 256 E4M3 codes vs torch's float8_e4m3fn -> float32 (a library routine)."""
    import torch
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(np.arange(256))
    nan_ok = np.array_equal(np.isnan(got), np.isnan(lib))
    fin = ~np.isnan(lib)
    return nan_ok and np.array_equal(got[fin], lib[fin]) and np.array_equal(np.signbit(got[fin]), np.signbit(lib[fin]))


def pin_e4m3_anchors():
    ok = True
    for code, v in _load_table("e4m3_anchors.txt"):
        g = float(oracle.e4m3_decode(code))
        ok &= (math.isnan(g) and math.isnan(v)) or (g == v and math.copysign(1, g) == math.copysign(1, v))
    return ok


def pin_golden(name):
    c = _load_case(name)
    idx, sc, status, rows = _run_case(c)
    ok = status == 0
    for t, want in enumerate(c["scores"]):
        ok &= np.array_equal(rows[t], np.asarray(want, dtype=np.float64))
    ok &= np.array_equal(idx, np.asarray(c["expected_idx"]))
    ok &= np.array_equal(sc, np.asarray(c["expected_score"], dtype=np.float64))
    return bool(ok)


def _onehot_pool(d, code, P=3, epb=16, D=128):
    """Pool whose only non-zero element is ``code`` at element ``d`` of
    (phys 2, slot 5); every group scale is 448 (0x7E) except group d//16 of
    that row, which is 1.0 (0x38); gscale 1/4."""
    fp4 = np.zeros((P, epb, D // 2), dtype=np.uint8)
    fp4[2, 5, d // 2] = (code << 4) if d % 2 else code
    sc = np.full((P, epb, D // 16), 0x7E, dtype=np.uint8)
    sc[2, 5, d // 16] = 0x38
    g = np.full(P, 0.25, dtype=np.float32)
    return fp4, sc, g


def pin_onehot_layout():
    """q = +-e_d probes every element position through the table: with the
    single non-zero code placed at logical key 21 (logical block 1 -> phys 2,
    slot 5), I[s] must be ReLU(+-value * 1.0 * 0.25) at s=21 and 0 elsewhere,
    the value taken from the printed E2M1 table."""
    tab = dict(_load_table("e2m1_table.txt"))
    bt = np.array([[0, 2, 1]], dtype=np.int32)
    ok = True
    for d in range(0, 128, 7):
        for code in (3, 7, 13):
            fp4, sc, g = _onehot_pool(d, code)
            for sign in (1.0, -1.0):
                q = np.zeros((1, 1, 128), dtype=np.float32)
                q[0, 0, d] = sign
                rows, status = oracle.score_topk_rows(q, np.ones((1, 1), np.float32), bt, 3, 3,
                                                      np.array([48], np.int32), 16,
                                                      keys_fp4=fp4, key_scale=sc, key_gscale=g)
                want = np.zeros(48)
                want[21] = max(sign * tab[code] * 1.0 * 0.25, 0.0)
                ok &= np.array_equal(rows[0], want)
                # the same code probed at every other element gives zero
                q2 = np.zeros_like(q)
                q2[0, 0, (d + 1) % 128] = 1.0
                rows2, _ = oracle.score_topk_rows(q2, np.ones((1, 1), np.float32), bt, 3, 3,
                                                  np.array([48], np.int32), 16,
                                                  keys_fp4=fp4, key_scale=sc, key_gscale=g)
                ok &= not rows2[0].any()
    return bool(ok)


def pin_closed_form():
    """All nibbles code c, all scales byte e, global scale g, q = 1: every key
    decodes to 128 copies of LUT[c]*E4M3[e]*g, so I = sum_h w_h ReLU(128 *
    LUT[c] * E4M3[e] * g) for every s (values from the printed tables)."""
    tab = dict(_load_table("e2m1_table.txt"))
    anchors = dict(_load_table("e4m3_anchors.txt"))
    ok = True
    rng = np.random.default_rng(5)
    w = rng.standard_normal((1, 4)).astype(np.float32)
    for c in (1, 5, 7, 9, 15):
        for e in (0x01, 0x30, 0x3C, 0x7E):
            fp4 = np.full((2, 64, 64), c | (c << 4), dtype=np.uint8)
            sc = np.full((2, 64, 8), e, dtype=np.uint8)
            g = np.array([0.125, 0.125], np.float32)
            q = np.ones((1, 4, 128), np.float32)
            rows, _ = oracle.score_topk_rows(q, w, np.array([[1, 0]], np.int32), 2, 2,
                                             np.array([100], np.int32), 64,
                                             keys_fp4=fp4, key_scale=sc, key_gscale=g)
            dot = 128 * tab[c] * anchors[e] * 0.125
            want = sum(float(w[0, h]) * max(dot, 0.0) for h in range(4))
            ok &= np.allclose(rows[0], want, rtol=1e-15, atol=0)
    return bool(ok)


def pin_block_permutation():
    """Moving the physical blocks and rewriting the table to match leaves
    every score bit-identical."""
    W = wl.tiny_decode(11, gscale_pow2_jitter=2)
    rows0, _ = oracle.score_topk_rows(W.q, W.w, W.block_table, W.bt_stride, W.max_lb, W.valid_lens,
                                      W.epb, **W.oracle_kwargs())
    pi = np.random.default_rng(3).permutation(W.P)
    fp4 = np.empty_like(W.keys_fp4); fp4[pi] = W.keys_fp4
    sc = np.empty_like(W.key_scale); sc[pi] = W.key_scale
    g = np.empty_like(W.key_gscale); g[pi] = W.key_gscale
    bt = pi[W.block_table].astype(np.int32)
    rows1, _ = oracle.score_topk_rows(W.q, W.w, bt, W.bt_stride, W.max_lb, W.valid_lens, W.epb,
                                      keys_fp4=fp4, key_scale=sc, key_gscale=g)
    return all(np.array_equal(rows0[t], rows1[t]) for t in rows0)


def pin_pow2_scaling():
    """w -> 2^j w and gscale -> 2^j gscale scale every score by exactly 2^j."""
    W = wl.tiny_decode(12)
    base, _ = oracle.score_topk_rows(W.q, W.w, W.block_table, W.bt_stride, W.max_lb, W.valid_lens,
                                     W.epb, **W.oracle_kwargs())
    ok = True
    for j in (-3, 5):
        r, _ = oracle.score_topk_rows(W.q, W.w * 2.0 ** j, W.block_table, W.bt_stride, W.max_lb,
                                      W.valid_lens, W.epb, **W.oracle_kwargs())
        ok &= all(np.array_equal(r[t], base[t] * 2.0 ** j) for t in base)
        kw = W.oracle_kwargs()
        kw["key_gscale"] = (W.key_gscale * 2.0 ** j).astype(np.float32)
        r, _ = oracle.score_topk_rows(W.q, W.w, W.block_table, W.bt_stride, W.max_lb,
                                      W.valid_lens, W.epb, **kw)
        ok &= all(np.array_equal(r[t], base[t] * 2.0 ** j) for t in base)
    return bool(ok)


def pin_positive_scaling_topk():
    """w -> c w (c > 0) scales scores by c and leaves the top-k indices alone."""
    W = wl.tiny_decode(13)
    i0, s0, _, _ = oracle.score_topk(W.q, W.w, W.block_table, W.bt_stride, W.max_lb, W.valid_lens,
                                     W.epb, W.top_k, **W.oracle_kwargs())
    i1, s1, _, _ = oracle.score_topk(W.q, (W.w.astype(np.float64) * 3.7), W.block_table, W.bt_stride,
                                     W.max_lb, W.valid_lens, W.epb, W.top_k, **W.oracle_kwargs())
    return np.array_equal(i0, i1) and np.allclose(s1, 3.7 * s0, rtol=1e-12)


def pin_topk_vs_lexsort():
    """Top-k == first k of numpy.lexsort on (index, -score), including ties."""
    rng = np.random.default_rng(9)
    ok = True
    for n, k in ((50, 8), (300, 300), (40, 64), (1000, 17)):
        s = rng.integers(-5, 5, size=n).astype(np.float64)   # many ties
        idx, sc = oracle.topk_sorted(s, k)
        order = np.lexsort((np.arange(n), -s))[:k]
        m = min(n, k)
        ok &= np.array_equal(idx[:m], order) and np.array_equal(sc[:m], s[order])
        ok &= bool(np.all(idx[m:] == -1) and np.all(np.isneginf(sc[m:])))
    return bool(ok)


def pin_topk_bruteforce():
    """Top-k == repeated selection of the best remaining entry (tiny inputs)."""
    rng = np.random.default_rng(10)
    ok = True
    for _ in range(20):
        n = int(rng.integers(0, 12)); k = int(rng.integers(1, 10))
        s = rng.integers(-3, 3, size=n).astype(np.float64)
        left = list(range(n)); want = []
        for _ in range(min(n, k)):
            best = left[0]
            for j in left:
                if s[j] > s[best] or (s[j] == s[best] and j < best):
                    best = j
            want.append(best); left.remove(best)
        idx, _ = oracle.topk_sorted(s, k)
        ok &= list(idx[:len(want)]) == want
    return bool(ok)


def pin_mask():
    """Keys at or past valid_len, made huge, never appear."""
    W = wl.tiny_decode(14)
    fp4 = W.keys_fp4.copy(); sc = W.key_scale.copy()
    L = 1000                                   # mid-block: 15 blocks + 40 slots
    for t in range(W.T):
        for lb in range(W.max_lb):
            phys = W.block_table[t, lb]
            lo = max(0, L - lb * W.epb)
            if lo < W.epb:
                fp4[phys, lo:] = 0x77; sc[phys, lo:] = 0x7E
    vl = np.full(W.T, L, np.int32)
    idx, _, _, rows = oracle.score_topk(W.q, W.w, W.block_table, W.bt_stride, W.max_lb, vl, W.epb,
                                        W.top_k, keys_fp4=fp4, key_scale=sc, key_gscale=W.key_gscale)
    return bool(np.all(idx < L)) and all(len(rows[t]) == L for t in rows)


def pin_bad_inputs():
    """Out-of-range table entries drop their keys and set bit 1; an
    out-of-range valid length pads the whole query and sets bit 2."""
    c = _load_case("tiny_score_a.json")
    c2 = dict(c); c2["block_table"] = [[1, 7]]           # logical block 1 -> phys 7 (P=2)
    idx, sc, status, _ = _run_case(c2)
    ok = status == oracle.STATUS_BAD_BLOCK and list(idx[0]) == [0, 1, -1, -1]
    c3 = dict(c); c3["valid_lens"] = [5]                 # > max_lb * epb = 4
    idx, sc, status, _ = _run_case(c3)
    ok &= status == oracle.STATUS_BAD_LEN and bool(np.all(idx == -1))
    return bool(ok)


def pin_valid_lens_from_blocks():
    """compute_valid_lens of commit c2f705a: block count * entries per block."""
    return list(oracle.valid_lens_from_blocks([0, 1, 3], 64)) == [0, 64, 192]


def pin_gather_library():
    """Gather == numpy fancy indexing over the flattened paged view."""
    rng = np.random.default_rng(4)
    P, bs, nkv, hd, T, n = 9, 4, 2, 8, 2, 13
    kc = rng.integers(0, 65535, size=(P, bs, nkv, hd), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(P, bs, nkv, hd), dtype=np.uint16)
    table = np.stack([rng.permutation(P)[:6] for _ in range(T)]).astype(np.int32)
    sel = rng.integers(0, 6 * bs, size=(T, n)); sel[0, 3] = -1
    k_out, v_out, st = oracle.gather_kv(sel, table, 6, 6, bs, kc, vc)
    flat_k = kc.reshape(P * bs, nkv, hd); flat_v = vc.reshape(P * bs, nkv, hd)
    rows = table[np.arange(T)[:, None], np.clip(sel, 0, None) // bs] * bs + np.clip(sel, 0, None) % bs
    want_k = np.where((sel >= 0)[..., None, None], flat_k[rows], 0)
    want_v = np.where((sel >= 0)[..., None, None], flat_v[rows], 0)
    return st == 0 and np.array_equal(k_out, want_k) and np.array_equal(v_out, want_v)


def pin_pool_special_cases():
    rng = np.random.default_rng(6)
    raw = rng.standard_normal((64, 16))
    w = rng.standard_normal(16) * 0.1
    ok = True
    # block 0 sits at position 0: rope is the identity there
    a = oracle.block_pool(raw, w, 0, 1, 4, 8, 1e6, 1e-6)
    b = oracle.block_pool(raw, w, 0, 1, 4, 0, 1e6, 1e-6)
    ok &= np.allclose(a, b, rtol=0, atol=0)
    # rope preserves the norm of every rotated pair
    a = oracle.block_pool(raw, w, 3, 5, 4, 8, 1e4, 1e-6)
    b = oracle.block_pool(raw, w, 3, 5, 4, 0, 1e4, 1e-6)
    for j in range(4):
        ok &= np.allclose(a[:, j] ** 2 + a[:, j + 4] ** 2, b[:, j] ** 2 + b[:, j + 4] ** 2, rtol=1e-12)
    ok &= np.array_equal(a[:, 8:], b[:, 8:])
    # ratio 1, w = 0, rot = 0: plain RMS normalisation of each row -> RMS 1, same direction
    c = oracle.block_pool(raw, np.zeros(16), 0, 64, 1, 0, 1e6, 0.0)
    ok &= np.allclose(np.sqrt(np.mean(c * c, axis=1)), 1.0, rtol=1e-12)
    ok &= np.allclose(c * np.linalg.norm(raw, axis=1, keepdims=True) / np.linalg.norm(c, axis=1, keepdims=True), raw)
    # closed form: hd 4, rot 2, ratio 2, rows [1,1,1,1],[3,3,3,3] -> mean 2, RMS-normalised 1;
    # block 1 sits at position 2 -> the pair (0,1) turns by 2 rad (frequency theta^0)
    r2 = np.array([[1, 1, 1, 1], [3, 3, 3, 3], [1, 1, 1, 1], [3, 3, 3, 3.0]])
    out = oracle.block_pool(r2, np.zeros(4), 1, 1, 2, 2, 1e6, 0.0)
    want = [math.cos(2) - math.sin(2), math.cos(2) + math.sin(2), 1, 1]
    ok &= np.allclose(out[0], want, rtol=1e-14, atol=1e-15)
    # second pair frequency: hd 4, rot 4, position 8 -> pair (1,3) turns by 8 * theta^(-1/2)
    out = oracle.block_pool(np.ones((16, 4)), np.zeros(4), 1, 1, 8, 4, 100.0, 0.0)
    ang = 8 * 100.0 ** -0.5
    ok &= np.allclose(out[0, [1, 3]], [math.cos(ang) - math.sin(ang), math.cos(ang) + math.sin(ang)], atol=1e-14)
    return bool(ok)


def pin_qprep_rows():
    """qsa.rs qsa_qprep / qsa_qprep_rows: the block pooling's normalisation
    and rope applied to single rows of the projection at first_pos + row."""
    rng = np.random.default_rng(8)
    hd, nh, rows = 16, 3, 5
    x = rng.standard_normal((rows, nh * hd))
    w = rng.standard_normal(hd) * 0.1
    ok = True
    # a one-row "block" at position p is the query row at position p (ratio 1)
    for h in range(nh):
        want = oracle.block_pool(x[:, h * hd:(h + 1) * hd], w, 0, rows, 1, 8, 1e4, 1e-6)
        got = oracle.qsa_qprep_rows(x, w, rows, 0, nh * hd, nh, hd, 8, 1e4, 1e-6)[:, h]
        ok &= np.allclose(got, want, rtol=1e-15, atol=0)
    # head h reads columns h*hd .. h*hd+hd-1 of a wider row; the rest is ignored
    wide = np.concatenate([x, rng.standard_normal((rows, 7)) * 1e3], axis=1)
    a = oracle.qsa_qprep_rows(wide, w, rows, 0, nh * hd + 7, nh, hd, 8, 1e4, 1e-6)
    b = oracle.qsa_qprep_rows(x, w, rows, 0, nh * hd, nh, hd, 8, 1e4, 1e-6)
    ok &= np.array_equal(a, b)
    # row r sits at first_pos + r
    c = oracle.qsa_qprep_rows(x[2:], w, rows - 2, 2, nh * hd, nh, hd, 8, 1e4, 1e-6)
    ok &= np.allclose(c, b[2:], rtol=1e-15, atol=0)
    # closed form: hd 4, rot 2, q = [2,2,2,2] (RMS 2) at position 3, w = 0:
    # [1,1,1,1] with the pair (0,1) turned by 3 rad
    out = oracle.qsa_qprep_rows(np.full((1, 4), 2.0), np.zeros(4), 1, 3, 4, 1, 4, 2, 1e6, 0.0)
    ok &= np.allclose(out[0, 0], [math.cos(3) - math.sin(3), math.cos(3) + math.sin(3), 1, 1], atol=1e-15)
    return bool(ok)


def pin_prefill_attn():
    """qsa.rs qsa_prefill_attn: softmax attention over the selected complete
    blocks plus the tail, through the page table, one kv head per group."""
    rng = np.random.default_rng(9)
    P, bs, nkv, hd = 6, 4, 2, 8
    kc = rng.standard_normal((P, bs, nkv, hd))
    vc = rng.standard_normal((P, bs, nkv, hd))
    table = np.array([3, 0, 5, 1, 4, 2])
    ok = True
    # position 0, no complete block: one token (the tail is position 0 alone) -> its V
    q = rng.standard_normal((1, 4, hd))
    out, st = oracle.qsa_prefill_attn(q, kc, vc, table, np.full((1, 2), -1), 0, 8, 0.5)
    ok &= st == 0 and np.allclose(out[0, 0], vc[3, 0, 0], rtol=0, atol=1e-15)
    # equal scores (K = 0) -> the mean of V over the attended tokens:
    # position 9, ratio 4: blocks 0, 1 complete; list [1, 7 (incomplete), 1 (again)]; tail 8, 9
    z = np.zeros_like(kc)
    out, st = oracle.qsa_prefill_attn(q, z, vc, table, np.array([[1, 7, 1]]), 9, 4, 0.5)
    toks = [4, 5, 6, 7, 4, 5, 6, 7, 8, 9]
    want = np.mean([vc[table[t // bs], t % bs, 0] for t in toks], axis=0)
    ok &= st == 0 and np.allclose(out[0, 0], want, rtol=1e-13)
    # two tokens, closed form: q.k = 2 for token 0 and 0 for token 1 (scale 0.5)
    # -> weights e^1 / (e^1 + 1) and 1 / (e^1 + 1)
    k2 = np.zeros_like(kc); k2[3, 0, 0, 0] = 2.0
    q2 = np.zeros((1, 2, hd)); q2[0, 0, 0] = 1.0
    out, _ = oracle.qsa_prefill_attn(q2, k2, vc, table, np.zeros((1, 0), int), 1, 8, 0.5)
    a = math.e / (math.e + 1)
    ok &= np.allclose(out[0, 0], a * vc[3, 0, 0] + (1 - a) * vc[3, 1, 0], rtol=1e-13)
    # query heads 0,1 read kv head 0 and heads 2,3 kv head 1 (V zero / one per kv head)
    v01 = np.zeros_like(vc); v01[:, :, 1] = 1.0
    out, _ = oracle.qsa_prefill_attn(q, kc, v01, table, np.array([[0, 1]]), 9, 4, 0.5)
    ok &= np.allclose(out[0, :2], 0.0) and np.allclose(out[0, 2:], 1.0)
    # the order of the list does not matter; a missing page is left out and reported
    lst = np.array([[0, 1], [1, 0]])
    q3 = np.repeat(q[:, None], 2, axis=0).reshape(2, 4, hd)
    o1, _ = oracle.qsa_prefill_attn(q3[:1], kc, vc, table, lst[:1], 9, 4, 0.5)
    o2, _ = oracle.qsa_prefill_attn(q3[1:], kc, vc, table, lst[1:], 9, 4, 0.5)
    ok &= np.allclose(o1, o2, rtol=1e-13)
    bad = table.copy(); bad[2] = -1       # tokens 8..11 have no page
    o3, st = oracle.qsa_prefill_attn(q3[:1], kc, vc, bad, lst[:1], 9, 4, 0.5)
    o4, _ = oracle.qsa_prefill_attn(q3[:1], kc, vc, table, lst[:1], 7, 4, 0.5)   # same blocks, no tail
    ok &= st == oracle.STATUS_BAD_BLOCK and np.allclose(o3, o4, rtol=1e-13)
    return bool(ok)


def pin_gather_split_library():
    """commit c2f705a's split gather: the FP8 part through torch's float8 decode,
    a float32 multiply and torch's bfloat16 cast; the bf16 part unchanged; rows
    resolved by fancy indexing; -1 gives zeros, a bad table entry zeros + status."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(10)
    P, bs, nd, rd, T, n = 6, 4, 8, 4, 3, 5
    codes = rng.integers(0, 256, size=(P, bs, nd)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C                       # no NaN codes
    scale = rng.uniform(0.01, 3.0, size=(P, bs)).astype(np.float32)
    rope = rng.integers(0, 65536, size=(P, bs, rd)).astype(np.uint16)
    table = rng.permutation(P)[:4].astype(np.int32).reshape(1, 4).repeat(T, 0)
    sel = rng.integers(-1, 16, size=(T, n)).astype(np.int32)
    out, st = oracle.gather_split(sel, table, 4, 4, bs, codes, scale, rope)
    deq = (torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32)
           * torch.from_numpy(scale)[:, :, None]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    rows = np.concatenate([deq, rope], axis=2)
    pos = np.clip(sel, 0, None)
    want = np.where((sel >= 0)[..., None], rows[table[np.arange(T)[:, None], pos // bs], pos % bs], 0)
    ok = st == 0 and np.array_equal(out, want)
    # ties round to even: 1 + 2^-8 -> 1.0, 1 + 3*2^-8 -> 1 + 2^-6
    ok &= np.array_equal(oracle.bf16_round(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8], np.float32)), [0x3F80, 0x3F82])
    bad = table.copy(); bad[1, 0] = P + 2
    sel2 = np.zeros((T, n), np.int32); sel2[1, 0] = 1
    out2, st2 = oracle.gather_split(sel2, bad, 4, 4, bs, codes, None, rope)
    ok &= st2 == oracle.STATUS_BAD_BLOCK and not out2[1, 0].any()
    return bool(ok)


def pin_qsa_score_handcase():
    """qsa.rs qsa_score on a hand-summed case: heads [1,0,..] and [0,-1,..],
    keys [2,3,..] and [-1,1,..], hd=4 -> score0 = (2 + 0)/2 = 1,
    score1 = (0 + 0)/2 = 0 (both dots of key 1 are <= 0: -1 and -1)."""
    q = np.array([[1, 0, 0, 0], [0, -1, 0, 0]], float)
    k = np.array([[2, 3, 0, 0], [-1, 1, 0, 0]], float)
    return np.array_equal(oracle.qsa_score(q, k), [1.0, 0.0])


def pin_expand_blocks():
    got = oracle.expand_blocks(np.array([[5, -1, 2]]), 3)
    return list(got[0]) == [6, 7, 8, 15, 16, 17, -1, -1, -1]



# ------------------------------------------------- NVFP4 queries (opt-in) ----

def _golden_vec(d, n=128):
    v = np.zeros(n)
    for off, vals in d.items():
        v[int(off):int(off) + len(vals)] = vals
    return v


def pin_nvfp4_q_golden():
    """The hand-worked head of tests/golden/nvfp4_q_example.json: every code,
    scale and dequantised value."""
    c = json.load(open(os.path.join(GOLDEN, "nvfp4_q_example.json")))
    x = _golden_vec(c["x_nonzero"]).astype(np.float32)
    codes, scales, gq = oracle.quantize_q_nvfp4(x)
    ok = float(gq) == c["gq"] and list(scales) == c["scales"]
    ok &= np.array_equal(codes, _golden_vec(c["codes_nonzero"]).astype(np.uint8))
    ok &= np.array_equal(oracle.dequantize_q_nvfp4(codes, scales, gq), _golden_vec(c["q_hat_nonzero"]))
    return bool(ok)


def pin_e4m3_encode_library():
    """The E4M3 encoder against torch's float8_e4m3fn cast (round to nearest
    even) on random values and on every midpoint between neighbouring codes;
    every code round-trips; values above 448 saturate."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    grid = oracle.e4m3_decode(np.arange(0x7F))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    x = np.concatenate([rng.uniform(0, 448, 3000), 2.0 ** rng.uniform(-12, 8.7, 3000), mids]).astype(np.float32)
    x = x[x <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ok = np.array_equal(oracle.e4m3_encode(x), want)
    ok &= np.array_equal(oracle.e4m3_encode(grid), np.arange(0x7F))
    ok &= np.array_equal(oracle.e4m3_encode(np.array([449.0, 480.0, 1e6])), [0x7E] * 3)
    return bool(ok)


def pin_e2m1_encode_ties():
    """E2M1 rounding at every midpoint of the table (ties to the even code),
    next to them, past 6 and below zero; against a threshold search over the
    table's midpoints for a dense sweep."""
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    want_tie = [0, 2, 2, 4, 4, 6, 6]
    ok = list(oracle.e2m1_encode(np.array(ties))) == want_tie
    ok &= list(oracle.e2m1_encode(np.array([-0.2, -0.3, -7.0, 6.5, 100.0]))) == [0, 9, 15, 7, 7]
    y = np.linspace(-8, 8, 64001)
    mag = np.abs(y)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    c = np.searchsorted(mids, mag, side="left")          # count of midpoints strictly below |y|
    at_mid = np.isin(mag, mids)
    c = np.where(at_mid & (c % 2 == 1), c + 1, c)         # a midpoint goes to the even neighbour
    want = np.where((y < 0) & (c != 0), c | 8, c)
    ok &= np.array_equal(oracle.e2m1_encode(y), want)
    return bool(ok)


def pin_nvfp4_q_invariants():
    """On random heads: each non-zero group's largest |x| lands on +-6 * gq * s;
    every element is within gq * s of its value (half the widest E2M1 gap);
    scaling q by 2^k scales gq by 2^k and changes no code or scale; -q flips
    exactly the signs; a zero head quantises to zeros."""
    rng = np.random.default_rng(9)
    q = (rng.standard_normal((64, 128)) * np.exp2(rng.integers(-6, 6, size=(64, 1)))).astype(np.float32)
    q[3] = 0
    q[5, 16:32] = 0
    codes, scales, gq = oracle.quantize_q_nvfp4(q)
    qh = oracle.dequantize_q_nvfp4(codes, scales, gq)
    s = oracle.e4m3_decode(scales) * gq[:, None].astype(np.float64)            # [64, 8]
    xg = q.reshape(64, 8, 16).astype(np.float64)
    hg = qh.reshape(64, 8, 16)
    ok = True
    arg = np.abs(xg).argmax(axis=-1)
    top = np.take_along_axis(hg, arg[..., None], -1)[..., 0]
    nz = np.abs(xg).max(-1) > 0
    ok &= np.allclose(np.abs(top[nz]), 6 * s[nz], rtol=0, atol=0)
    ok &= bool(np.all(np.abs(xg - hg) <= s[..., None] * (1 + 1e-6)))
    for k in (-3, 5):
        c2, s2, g2 = oracle.quantize_q_nvfp4(q * np.float32(2.0 ** k))
        ok &= np.array_equal(c2, codes) and np.array_equal(s2, scales) and np.array_equal(g2, gq * np.float32(2.0 ** k))
    c3, s3, g3 = oracle.quantize_q_nvfp4(-q)
    ok &= np.array_equal(s3, scales) and np.array_equal(g3, gq)
    ok &= np.array_equal(c3, np.where(codes != 0, codes ^ 8, 0))
    ok &= not codes[3].any() and not scales[3].any() and gq[3] == 0
    ok &= not scales[5, 1] and not codes[5, 16:32].any()
    return bool(ok)


def pin_nvfp4_q_scores_bound():
    """Scores from NVFP4 queries stay within sum_h |w_h| sum_d |q - q_hat| |K|
    of the exact scores (ReLU is 1-Lipschitz), on a small decode batch."""
    W = wl.tiny_decode(1000)
    rows = list(range(W.T))
    exact, _ = oracle.score_topk_rows(W.q, W.w, W.block_table, W.bt_stride, W.max_lb, W.valid_lens, W.epb,
                                      rows=rows, **W.oracle_kwargs())
    qh = oracle.nvfp4_q(W.q)
    approx, _ = oracle.score_topk_rows(qh, W.w, W.block_table, W.bt_stride, W.max_lb, W.valid_lens, W.epb,
                                       rows=rows, **W.oracle_kwargs())
    ok = True
    for t in rows:
        phys, slot, okm = oracle.resolve_slots(oi._table_row(W.block_table, W.bt_stride, W.max_lb, t),
                                               int(W.valid_lens[t]), W.epb, W.keys_fp4.shape[0])
        K = oracle.dequant_rows(W.keys_fp4, W.key_scale, W.key_gscale, phys[okm], slot[okm])
        dq = np.abs(np.asarray(W.q[t], np.float64) - qh[t])                      # [H, D]
        bound = np.abs(K) @ dq.T @ np.abs(np.asarray(W.w[t], np.float64))        # [n]
        diff = np.abs(exact[t][okm] - approx[t][okm])
        ok &= bool(np.all(diff <= bound * (1 + 1e-9) + 1e-12)) and bool(np.any(diff > 0))
    return bool(ok)

PINS = [pin_e2m1_printed_table, pin_e2m1_bitlevel, pin_e4m3_library, pin_e4m3_anchors,
        lambda: pin_golden("tiny_score_a.json"), lambda: pin_golden("tiny_score_ties.json"),
        lambda: pin_golden("tiny_score_shared.json"), pin_onehot_layout, pin_closed_form,
        pin_block_permutation, pin_pow2_scaling, pin_positive_scaling_topk, pin_topk_vs_lexsort,
        pin_topk_bruteforce, pin_mask, pin_bad_inputs, pin_valid_lens_from_blocks,
        pin_gather_library, pin_gather_split_library, pin_pool_special_cases, pin_qprep_rows, pin_prefill_attn,
        pin_qsa_score_handcase,
        pin_expand_blocks, pin_nvfp4_q_golden, pin_e4m3_encode_library, pin_e2m1_encode_ties,
        pin_nvfp4_q_invariants, pin_nvfp4_q_scores_bound]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: getattr(f, "__name__", "golden"))
def test_pin(pin):
    assert pin()


def test_integer_decode_is_a_negative_control():
    """The integer decode shipped before commit 79ef87f differs from E2M1 on
    every non-zero magnitude code: the bug report that commit describes."""
    integer = np.arange(8, dtype=np.float64)
    e2m1 = oracle.e2m1_decode(np.arange(8))
    assert list(np.nonzero(integer != e2m1)[0]) == [1, 2, 3, 4, 5, 6, 7]


# ------------------------------------------------------- planted mistakes ----

def _all_pins_pass():
    return all(p() for p in PINS)


MUTATIONS = {
    "integer_fp4_decode": ("e2m1_decode", lambda c: np.where(np.asarray(c) & 8, -1.0, 1.0) * (np.asarray(c) & 7)),
    "nibble_order_swapped": ("unpack_nibbles", lambda p: (lambda a: np.stack([(a >> 4) & 0xF, a & 0xF], -1).reshape(a.shape[:-1] + (-1,)))(np.asarray(p, np.int64))),
    "e4m3_bias_8": ("e4m3_decode", lambda b: (lambda x: np.where((x >> 3) & 15 == 0, (x & 7) / 8 * 2.0 ** -7, (1 + (x & 7) / 8) * np.exp2(((x >> 3) & 15) - 8.0)) * np.where(x & 128, -1, 1))(np.asarray(b, np.int64) & 255)),
}


def _mut_index_scores_no_relu(q_t, w_t, K):
    return (np.asarray(K, np.float64) @ np.asarray(q_t, np.float64).T) @ np.asarray(w_t, np.float64)


def _mut_group_by_8(keys_fp4, key_scale, key_gscale, phys, slot):
    codes = oi.unpack_nibbles(np.asarray(keys_fp4)[phys, slot])
    vals = oi.e2m1_decode(codes)
    scales = oi.e4m3_decode(np.asarray(key_scale)[phys, slot])
    grp = np.minimum(np.arange(vals.shape[-1]) // 8, scales.shape[-1] - 1)
    return vals * scales[:, grp] * np.asarray(key_gscale, np.float64)[phys][:, None]


def _mut_slot_swapped(table_row, valid_len, epb, n_phys):
    s = np.arange(int(valid_len))
    logical = np.minimum(s % epb, len(table_row) - 1)
    slot = np.minimum(s // epb, epb - 1)
    phys = np.asarray(table_row, np.int64)[logical]
    return phys, slot, (phys >= 0) & (phys < n_phys)


def _mut_ties_high_index_first(scores, k, index=None):
    sc = np.asarray(scores, np.float64)
    ix = np.arange(len(sc)) if index is None else np.asarray(index)
    order = np.lexsort((-ix, -sc))
    out_i = np.full(k, -1); out_s = np.full(k, -np.inf)
    n = min(k, len(sc)); out_i[:n] = ix[order][:n]; out_s[:n] = sc[order][:n]
    return out_i, out_s


def _mut_weight_inside_relu(q_t, w_t, K):
    dots = np.asarray(K, np.float64) @ np.asarray(q_t, np.float64).T
    return np.maximum(dots * np.asarray(w_t, np.float64), 0.0).sum(axis=1)


def _mut_qprep_ignores_first_pos(qk, q_norm_w, rows, first_pos, qkw, n_heads, hd, rot, theta, eps, **kw):
    return _real_qprep(qk, q_norm_w, rows, 0, qkw, n_heads, hd, rot, theta, eps, **kw)


def _mut_qprep_head_stride_qkw(qk, q_norm_w, rows, first_pos, qkw, n_heads, hd, rot, theta, eps, **kw):
    qk = np.asarray(qk, np.float64).reshape(rows, qkw)
    cols = np.concatenate([qk[:, h * qkw // n_heads:h * qkw // n_heads + hd] for h in range(n_heads)], axis=1)
    return _real_qprep(cols, q_norm_w, rows, first_pos, n_heads * hd, n_heads, hd, rot, theta, eps, **kw)


_real_qprep = oracle.qsa_qprep_rows
_real_attn = oracle.qsa_prefill_attn


def _mut_bf16_truncate(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _mut_attn_tail_excludes_own_position(q, k_cache, v_cache, block_table, lists, first_pos, ratio, inv_sqrt_d):
    # attends like the real one but one position earlier (the row's own token dropped)
    q = np.asarray(q, np.float64)
    outs, st = [], 0
    for r in range(q.shape[0]):
        if first_pos + r == 0:
            outs.append(np.zeros(q.shape[1:]))
            continue
        o, s_ = _real_attn(q[r:r + 1], k_cache, v_cache, block_table, np.asarray(lists)[r:r + 1],
                           first_pos + r - 1, ratio, inv_sqrt_d)
        outs.append(o[0]); st |= s_
    return np.array(outs), st


def _mut_attn_kv_head_modulo(q, k_cache, v_cache, block_table, lists, first_pos, ratio, inv_sqrt_d):
    q = np.asarray(q, np.float64)
    nq, nkv = q.shape[1], np.asarray(k_cache).shape[2]
    outs = []
    for h in range(nq):   # head h reads kv head h % nkv
        kv = h % nkv
        kc = np.asarray(k_cache)[:, :, kv:kv + 1]; vc = np.asarray(v_cache)[:, :, kv:kv + 1]
        o, st = _real_attn(q[:, h:h + 1], kc, vc, block_table, lists, first_pos, ratio, inv_sqrt_d)
        outs.append(o[:, 0])
    return np.stack(outs, axis=1), st


def _mut_e4m3_encode_truncates(x):
    grid = oracle.e4m3_decode(np.arange(0x7F))
    return (np.searchsorted(grid, np.asarray(x, np.float64), side="right") - 1).clip(0, 0x7E).astype(np.uint8)


def _mut_e2m1_ties_away(y):
    y = np.asarray(y, np.float64)
    mags = np.asarray(oracle.E2M1_MAGNITUDES)
    d = np.abs(np.abs(y)[..., None] - mags)
    best = d == d.min(-1, keepdims=True)
    c = (best * np.arange(8)).max(-1)                       # the larger magnitude of a tie
    return np.where((y < 0) & (c != 0), c | 8, c).astype(np.uint8)


def _mut_quantize_groups_of_32(q):
    """The same steps with one E4M3 scale per 32 elements (returned twice)."""
    f32 = np.float32
    x = np.asarray(q, np.float32)
    lead = x.shape[:-1]
    xg = x.reshape(lead + (4, 32))
    amax = np.abs(x).max(-1)
    gq = np.where(amax > 0, amax / f32(2688), f32(0)).astype(np.float32)
    ag = np.abs(xg).max(-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        s_f = np.where(ag > 0, (ag / (f32(6) * gq)[..., None]).astype(np.float32), f32(0))
    sc = oracle.e4m3_encode(s_f)
    sv = oracle.e4m3_decode(sc).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (xg / (gq[..., None] * sv)[..., None]).astype(np.float32)
    codes = np.where((sv > 0)[..., None], oracle.e2m1_encode(y), 0).astype(np.uint8)
    return codes.reshape(lead + (128,)), np.repeat(sc, 2, -1), gq


@pytest.mark.parametrize("name,target,fn", [
    *[(k, v[0], v[1]) for k, v in MUTATIONS.items()],
    ("qprep_ignores_first_pos", "qsa_qprep_rows", _mut_qprep_ignores_first_pos),
    ("qprep_head_stride_qkw", "qsa_qprep_rows", _mut_qprep_head_stride_qkw),
    ("attn_tail_excludes_own_position", "qsa_prefill_attn", _mut_attn_tail_excludes_own_position),
    ("attn_kv_head_modulo", "qsa_prefill_attn", _mut_attn_kv_head_modulo),
    ("bf16_truncates", "bf16_round", _mut_bf16_truncate),
    ("relu_dropped", "index_scores", _mut_index_scores_no_relu),
    ("weight_inside_relu", "index_scores", _mut_weight_inside_relu),
    ("group_of_8", "dequant_rows", _mut_group_by_8),
    ("block_and_slot_swapped", "resolve_slots", _mut_slot_swapped),
    ("ties_high_index_first", "topk_sorted", _mut_ties_high_index_first),
    ("nvfp4_q_range_448", "NVFP4_Q_RANGE", 448.0),
    ("e4m3_encode_truncates", "e4m3_encode", _mut_e4m3_encode_truncates),
    ("e2m1_ties_away_from_zero", "e2m1_encode", _mut_e2m1_ties_away),
    ("nvfp4_q_scale_per_32", "quantize_q_nvfp4", _mut_quantize_groups_of_32),
])
def test_planted_mistake_is_caught(monkeypatch, name, target, fn):
    monkeypatch.setattr(oi, target, fn, raising=hasattr(oi, target) or not hasattr(oracle, target))
    monkeypatch.setattr(oracle, target, fn, raising=False)
    assert not _all_pins_pass(), f"planted mistake {name!r} in {target} went unnoticed"
