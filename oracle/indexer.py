"""Lightning-indexer score + top-k, written out as its plain definition in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

The method (header comment of "indexer_score_topk.cu", CSA lightning indexer,
eq. 16) scores every valid compressed key ``s`` of query ``t``:

    I[t, s] = sum_h  w[t, h] * ReLU( q[t, h, :] . K[s, :] )

and keeps ``TopK(I[t, :], k)``. One key row per ``s`` is shared by all heads:
the kernel body of that page ("Main kernel" section) reads ``K`` at
``block_entry`` with no head index, so the ``K[s, h]`` written in the header is
read as ``K[s]``.

Keys live in a paged NVFP4 pool ("Main kernel" argument list and the
"PyTorch binding" section of the same page):

* ``keys_fp4  [P, epb, D/2] uint8``  two E2M1 codes per byte, low nibble is
  the even element (``lane 0 = low nibble`` in the FP4 dequantization
  section; ``d0 = g*16 + 2*b`` reads the low nibble in the main loop);
* ``key_scale [P, epb, D/16] uint8`` one FP8 E4M3 scale per 16 elements;
* ``key_gscale [P] float32``          one global scale per physical block.

Everything below is float64 numpy; a library primitive (matmul, stable sort)
serves as a step where the definition has one, with no blocking or
reordering beyond the definition.
"""

from __future__ import annotations

import numpy as np

# Status bits a call reports instead of faulting (shared meaning with the
# library's device status word; the values are part of the public contract).
STATUS_BAD_BLOCK = 1  # a block-table entry outside [0, P)
STATUS_BAD_LEN = 2    # a valid length outside [0, max_logical_blocks * epb]
STATUS_BAD_SEL = 4    # a gather position whose logical block is outside the table

# E2M1 magnitudes for the three magnitude bits, as the lookup table of commit
# e74c844 ("Clean up E2M1 dequant: use LUT approach") lists them.
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_decode(codes) -> np.ndarray:
    """Decode 4-bit E2M1 codes to float64.

    Magnitude from the lookup table of commit e74c844 (index = low three
    bits); bit 3 is the sign ("bit3=sign, bits[2:0]=magnitude", FP4
    dequantization section of indexer_score_topk.cu). Code 8 is -0.0.
    """
    c = np.asarray(codes, dtype=np.int64)
    mag = np.asarray(E2M1_MAGNITUDES, dtype=np.float64)[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def e4m3_decode(raw) -> np.ndarray:
    """Decode FP8 E4M3 (OCP "e4m3fn": bias 7, no infinities) bytes to float64.

    indexer_score_topk.cu decodes each group scale through ``__nv_fp8_e4m3``
    ("Read group scale (FP8 E4M3)" in the main loop). Written out:
    exponent field ``e = bits 6..3``, mantissa ``m = bits 2..0``;
    ``e == 0`` is subnormal ``m/8 * 2^-6``; otherwise ``(1 + m/8) * 2^(e-7)``;
    ``e == 15, m == 7`` is NaN; bit 7 is the sign.
    """
    b = np.asarray(raw, dtype=np.int64) & 0xFF
    sign = (b >> 7) & 1
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    subnormal = (m / 8.0) * 2.0 ** -6
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    val = np.where(e == 0, subnormal, normal)
    val = np.where((e == 15) & ((b & 7) == 7), np.nan, val)
    return np.where(sign == 1, -val, val)


def unpack_nibbles(packed) -> np.ndarray:
    """``[..., D/2]`` bytes -> ``[..., D]`` E2M1 codes; element ``2j`` is the low
    nibble of byte ``j`` and ``2j+1`` the high nibble (FP4 dequantization
    section: lane 0 = low nibble; main loop: ``d0 = g*16 + 2*b``, ``d1 = d0+1``).
    """
    p = np.asarray(packed, dtype=np.int64)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int64)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = (p >> 4) & 0xF
    return out


def resolve_slots(table_row, valid_len: int, epb: int, n_phys: int):
    """Slot resolution of the "Main kernel" section of indexer_score_topk.cu.

    For ``s < valid_len``: ``logical_block = s // epb``, ``slot = s % epb``,
    ``phys = table_row[logical_block]``. Returns ``(phys, slot, ok)`` with
    ``ok`` false where ``phys`` lies outside ``[0, n_phys)``.
    """
    s = np.arange(int(valid_len), dtype=np.int64)
    logical = s // epb
    slot = s % epb
    phys = np.asarray(table_row, dtype=np.int64)[logical]
    ok = (phys >= 0) & (phys < n_phys)
    return phys, slot, ok


def dequant_rows(keys_fp4, key_scale, key_gscale, phys, slot) -> np.ndarray:
    """NVFP4 key rows ``K[n, D]`` in float64.

    ``K[s, d] = e2m1(code[s, d]) * e4m3(scale[s, d // 16]) * gscale[phys]``:
    16-element groups with one FP8 scale each and one FP32 global scale per
    physical block (main loop of indexer_score_topk.cu: ``group_s =
    fp8_s * global_s`` applied to the 8 packed bytes of group ``g``), with the
    E2M1 values of commit 79ef87f instead of the integer decode that commit
    replaced.
    """
    phys = np.asarray(phys, dtype=np.int64)
    slot = np.asarray(slot, dtype=np.int64)
    codes = unpack_nibbles(np.asarray(keys_fp4)[phys, slot])          # [n, D]
    vals = e2m1_decode(codes)                                          # [n, D]
    scales = e4m3_decode(np.asarray(key_scale)[phys, slot])            # [n, D/16]
    d = vals.shape[-1]
    group_of = np.arange(d) // 16
    g = np.asarray(key_gscale, dtype=np.float64)[phys]                 # [n]
    return vals * scales[:, group_of] * g[:, None]


def index_scores(q_t, w_t, K) -> np.ndarray:
    """``I[s] = sum_h w[h] * max(q[h] . K[s], 0)`` for the rows of ``K``.

    Eq. 16 in the header of indexer_score_topk.cu; the ReLU-then-weight step is
    the "ReLU + weighted sum" lines of its main loop (``if (dot > 0) score +=
    w[h] * dot``).
    """
    q_t = np.asarray(q_t, dtype=np.float64)
    w_t = np.asarray(w_t, dtype=np.float64)
    dots = np.asarray(K, dtype=np.float64) @ q_t.T                     # [n, H]
    return np.maximum(dots, 0.0) @ w_t                                 # [n]


def topk_sorted(scores, k: int, index=None):
    """The ``k`` best entries under (score descending, index ascending).

    Ordering and padding follow indexer_score_topk.cu: its selection sort emits
    higher scores first and the lower index on equal scores ("Write top-k
    indices" section); unfilled slots keep ``-1`` / ``-inf`` (heap initialised
    to ``-INFINITY`` / ``-1``). ``index`` gives the logical index of each score
    (default ``0..n-1``). A stable sort on the negated score is the full sort
    the definition calls for.
    """
    sc = np.asarray(scores, dtype=np.float64)
    ix = np.arange(sc.shape[0], dtype=np.int64) if index is None else np.asarray(index, dtype=np.int64)
    order = np.argsort(ix, kind="stable")          # ascending index first ...
    sc, ix = sc[order], ix[order]
    order = np.argsort(-sc, kind="stable")         # ... then score descending, ties keep index order
    sc, ix = sc[order], ix[order]
    out_i = np.full(k, -1, dtype=np.int64)
    out_s = np.full(k, -np.inf, dtype=np.float64)
    n = min(k, sc.shape[0])
    out_i[:n] = ix[:n]
    out_s[:n] = sc[:n]
    return out_i, out_s


def valid_lens_from_blocks(block_lens, epb: int) -> np.ndarray:
    """``valid_lens = block_lens * entries_per_block``: the compute_valid_lens
    step of commit c2f705a (all entries of an allocated block are valid)."""
    return np.asarray(block_lens, dtype=np.int64) * int(epb)


def _table_row(block_table, bt_stride: int, max_lb: int, t: int):
    flat = np.asarray(block_table).reshape(-1)
    start = t * int(bt_stride)
    return flat[start:start + max_lb]


def score_topk_rows(q, w, block_table, bt_stride, max_lb, valid_lens, epb, *,
                    keys_fp4=None, key_scale=None, key_gscale=None, keys_f32=None,
                    rows=None):
    """Full score rows ``I[t, :valid_len[t]]`` for the queries in ``rows``.

    Returns ``(scores, status)``; ``scores[t]`` is a float64 array of length
    ``valid_lens[t]`` (``None`` when that length is outside
    ``[0, max_lb * epb]``), with ``-inf`` at keys whose block-table entry is
    outside ``[0, P)``. ``keys_f32 [P, epb, D]`` replaces the NVFP4 pool for
    the unquantised (QSA) key format.
    """
    q = np.asarray(q)
    T = q.shape[0]
    rows = range(T) if rows is None else rows
    n_phys = (np.asarray(keys_f32).shape[0] if keys_f32 is not None
              else np.asarray(keys_fp4).shape[0])
    status = 0
    out = {}
    for t in rows:
        L = int(valid_lens[t])
        if L < 0 or L > max_lb * epb:
            status |= STATUS_BAD_LEN
            out[t] = None
            continue
        phys, slot, ok = resolve_slots(_table_row(block_table, bt_stride, max_lb, t), L, epb, n_phys)
        if not ok.all():
            status |= STATUS_BAD_BLOCK
        I = np.full(L, -np.inf, dtype=np.float64)
        if ok.any():
            if keys_f32 is not None:
                K = np.asarray(keys_f32, dtype=np.float64)[phys[ok], slot[ok]]
            else:
                K = dequant_rows(keys_fp4, key_scale, key_gscale, phys[ok], slot[ok])
            I[ok] = index_scores(q[t], np.asarray(w)[t], K)
        out[t] = I
    return out, status


def score_topk(q, w, block_table, bt_stride, max_lb, valid_lens, epb, k, *,
               keys_fp4=None, key_scale=None, key_gscale=None, keys_f32=None,
               rows=None):
    """``TopK(I[t, :], k)`` per query: indices, scores and the status bits.

    Keys with an out-of-range block-table entry are not candidates; a query
    whose valid length is out of range yields only padding. Returns
    ``(idx [R, k] int64, score [R, k] float64, status, scores)`` for the ``R``
    queries in ``rows`` (default: all), ``scores`` being the per-query rows of
    :func:`score_topk_rows`.
    """
    scores, status = score_topk_rows(q, w, block_table, bt_stride, max_lb, valid_lens, epb,
                                     keys_fp4=keys_fp4, key_scale=key_scale,
                                     key_gscale=key_gscale, keys_f32=keys_f32, rows=rows)
    ts = list(scores.keys())
    idx = np.full((len(ts), k), -1, dtype=np.int64)
    sc = np.full((len(ts), k), -np.inf, dtype=np.float64)
    for r, t in enumerate(ts):
        I = scores[t]
        if I is None:
            continue
        cand = np.nonzero(~np.isneginf(I))[0]   # excluded keys carry -inf
        idx[r], sc[r] = topk_sorted(I[cand], k, index=cand)
    return idx, sc, status, scores


# ---------------------------------------------------------------------------
# NVFP4 queries: the opt-in mode in which the dot products take q in NVFP4.
#
# The header comment of indexer_score_topk.cu plans a second phase that swaps
# the FP32 dot products for the FP4 tensor-core MMA, which takes both operands
# in FP4; the "Main kernel" argument list already calls the query inputs
# "dequantized from FP4", and commit c2f705a's CSAIndexer keeps a placeholder
# projection "until Nvfp4Linear with FP4 output". The pages give no recipe for
# quantising q; this mode applies the NVFP4 scheme of the keys (E2M1 elements,
# one E4M3 scale per 16 consecutive elements, "FP4 dequantization (NVFP4
# scheme)") plus one float32 scale per (query, head) that maps the head's
# largest |q| onto the top of the E2M1 x E4M3 range, 6 * 448 = 2688. Every
# rounding decision is taken in float32, in this order:
#     amax = max_d |x_d|,                gq = fl32(amax / 2688)  (0 if amax == 0)
#     per group g of 16 elements:        s_g = E4M3(fl32(ag / fl32(6 * gq)))
#     per element (code 0 if s_g == 0):  c_d = E2M1(fl32(x_d / fl32(gq * s_g)))
#     dequantised:                       q_hat_d = gq * s_g * e2m1(c_d)
# where E4M3() and E2M1() round to the nearest representable value, ties to
# the even code, saturating at the largest finite value (448, 6); a value that
# rounds to zero gets code 0 (no negative zero).

NVFP4_Q_RANGE = 2688.0   # 6 (largest E2M1) * 448 (largest finite E4M3)


def _nearest_even_code(x, grid):
    """Index of the grid value nearest to each x (float64 distances), the even
    index on a tie; values beyond the grid's end take its last entry."""
    x = np.asarray(x, dtype=np.float64)
    d = np.abs(x[..., None] - np.asarray(grid, dtype=np.float64))
    best = d == d.min(axis=-1, keepdims=True)
    pref = best * np.where(np.arange(len(grid)) % 2 == 0, 2, 1)   # prefer the even code of a tie
    return np.argmax(pref, axis=-1)


def e4m3_encode(x) -> np.ndarray:
    """Non-negative values to E4M3 bytes: nearest finite value (codes 0..0x7E),
    ties to the even code, saturating at 448."""
    grid = e4m3_decode(np.arange(0x7F))
    return _nearest_even_code(x, grid).astype(np.uint8)


def e2m1_encode(y) -> np.ndarray:
    """Values to E2M1 codes: nearest magnitude of the E2M1 table, ties to the
    even code, saturating at 6; bit 3 set for a negative value that does not
    round to zero."""
    y = np.asarray(y, dtype=np.float64)
    c = _nearest_even_code(np.abs(y), E2M1_MAGNITUDES)
    return np.where((y < 0) & (c != 0), c | 8, c).astype(np.uint8)


def quantize_q_nvfp4(q):
    """``q [..., 128]`` (taken as float32) -> ``(codes [..., 128] uint8,
    scales [..., 8] uint8 E4M3, gq [...] float32)`` by the steps above."""
    x = np.asarray(q, dtype=np.float32)
    lead = x.shape[:-1]
    xg = x.reshape(lead + (8, 16))
    f32 = np.float32
    amax = np.abs(x).max(axis=-1)
    gq = np.where(amax > 0, amax / f32(NVFP4_Q_RANGE), f32(0)).astype(np.float32)
    ag = np.abs(xg).max(axis=-1)                                              # [..., 8]
    with np.errstate(divide="ignore", invalid="ignore"):
        s_f = (ag / (f32(6) * gq)[..., None]).astype(np.float32)
    s_f = np.where(ag > 0, s_f, f32(0))
    scales = e4m3_encode(s_f)
    s_val = e4m3_decode(scales).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (xg / (gq[..., None] * s_val)[..., None]).astype(np.float32)
    codes = np.where((s_val > 0)[..., None], e2m1_encode(y), 0).astype(np.uint8)
    return codes.reshape(lead + (128,)), scales, gq


def dequantize_q_nvfp4(codes, scales, gq) -> np.ndarray:
    """``q_hat = gq * s_g * e2m1(code)`` in float64 (exact)."""
    codes = np.asarray(codes)
    lead = codes.shape[:-1]
    v = e2m1_decode(codes).reshape(lead + (8, 16))
    s = e4m3_decode(scales)[..., None]
    return (v * s * np.asarray(gq, dtype=np.float64)[..., None, None]).reshape(lead + (128,))


def nvfp4_q(q) -> np.ndarray:
    """The queries the NVFP4-q mode scores with: ``dequantize(quantize(q))``."""
    return dequantize_q_nvfp4(*quantize_q_nvfp4(q))
