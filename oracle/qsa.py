"""QSA key pooling, QSA query preparation, QSA block score, the selected-row
K/V gather and the prefill attention over the selected blocks, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "metrale_model_layers/layers/ops/qsa.rs" (doc comments of
``qsa_block_pool``, ``qsa_qprep``, ``qsa_qprep_rows``, ``qsa_score``,
``qsa_gather`` and ``qsa_prefill_attn``) and the gather described
in commit c2f705a of "Commit graph, dsv4/kernels/indexer" (dense tile from the
paged pool through the block table).
"""

from __future__ import annotations

import math

import numpy as np

from .indexer import STATUS_BAD_BLOCK, STATUS_BAD_SEL, e4m3_decode


def block_pool(raw_keys, k_norm_w, first_block: int, n_new: int, ratio: int,
               rot: int, theta: float, eps: float, *, interleaved: bool = False) -> np.ndarray:
    """Pool ``n_new`` newly complete blocks starting at ``first_block``.

    qsa.rs, ``qsa_block_pool``: the mean of ``ratio`` raw keys, then RMSNorm
    scaled by ``1 + w``, then rope at the block's first token position.
    Returns ``[n_new, hd]``; row ``i`` is block ``first_block + i``, pooled
    from raw rows ``[(first_block+i)*ratio, (first_block+i+1)*ratio)`` at
    position ``(first_block+i)*ratio``.

    Readings where the page is silent: RMSNorm is
    ``m / sqrt(mean(m^2) + eps) * (1 + w)``; rope rotates the first ``rot``
    dimensions, pairing ``i`` with ``i + rot/2`` (half split; ``interleaved``
    pairs ``2i`` with ``2i+1`` instead) at angle ``pos * theta^(-2i/rot)``.
    Parity unpinned for the pairing convention.
    """
    raw = np.asarray(raw_keys, dtype=np.float64)
    w = np.asarray(k_norm_w, dtype=np.float64)
    hd = raw.shape[1]
    out = np.zeros((n_new, hd), dtype=np.float64)
    half = rot // 2
    for i in range(n_new):
        b = first_block + i
        m = raw[b * ratio:(b + 1) * ratio].mean(axis=0)
        y = m / math.sqrt(float(np.mean(m * m)) + eps) * (1.0 + w)
        pos = b * ratio
        z = y.copy()
        for j in range(half):
            ang = pos * theta ** (-2.0 * j / rot)
            c, s = math.cos(ang), math.sin(ang)
            a_i, b_i = (2 * j, 2 * j + 1) if interleaved else (j, j + half)
            x1, x2 = y[a_i], y[b_i]
            z[a_i] = x1 * c - x2 * s
            z[b_i] = x2 * c + x1 * s
        out[i] = z
    return out


def qsa_qprep_rows(qk, q_norm_w, rows: int, first_pos: int, qkw: int, n_heads: int, hd: int, rot: int,
                   theta: float, eps: float, *, interleaved: bool = False) -> np.ndarray:
    """Query preparation for QSA scoring, ``[rows, n_heads, hd]``.

    qsa.rs, ``qsa_qprep`` (one decode query: per head, RMSNorm scaled by
    ``1 + w``, then partial rope at ``pos``) and ``qsa_qprep_rows`` (the same
    for ``rows`` prefill rows at positions ``first_pos + row``, reading q from
    rows of the indexer projection ``qk``). Readings where the page is silent:
    row ``r`` of ``qk`` has ``qkw`` values and head ``h``'s q is its columns
    ``h*hd .. h*hd+hd-1``; RMSNorm and rope as in :func:`block_pool`.
    """
    qk = np.asarray(qk, dtype=np.float64).reshape(rows, qkw)
    w = np.asarray(q_norm_w, dtype=np.float64)
    out = np.zeros((rows, n_heads, hd), dtype=np.float64)
    half = rot // 2
    for r in range(rows):
        pos = first_pos + r
        for h in range(n_heads):
            x = qk[r, h * hd:(h + 1) * hd]
            y = x / math.sqrt(float(np.mean(x * x)) + eps) * (1.0 + w)
            z = y.copy()
            for j in range(half):
                ang = pos * theta ** (-2.0 * j / rot)
                c, s = math.cos(ang), math.sin(ang)
                a_i, b_i = (2 * j, 2 * j + 1) if interleaved else (j, j + half)
                z[a_i] = y[a_i] * c - y[b_i] * s
                z[b_i] = y[b_i] * c + y[a_i] * s
            out[r, h] = z
    return out


def qsa_prefill_attn(q, k_cache, v_cache, block_table, lists, first_pos: int, ratio: int,
                     inv_sqrt_d: float):
    """Prefill attention over the selected blocks plus the incomplete tail.

    qsa.rs, ``qsa_prefill_attn``: per (row, q head), attention over exactly the
    selected blocks in ``lists`` plus the incomplete tail, read from the paged
    cache. Readings where the page is silent: row ``r`` is at position
    ``p = first_pos + r``; blocks ``b < (p+1) // ratio`` are complete and only
    those entries of the row's list count (others are skipped, duplicates are
    not merged); the tail is tokens ``((p+1)//ratio)*ratio .. p``; query head
    ``h`` reads kv head ``h // (nq // nkv)``; token ``t`` is at page
    ``block_table[t // block_size]``, slot ``t % block_size``; one softmax of
    ``(q . k) * inv_sqrt_d`` weights V. A token whose page is missing or out
    of range is left out and reported; a row with no token gives zeros.

    q ``[rows, nq, hd]``; caches ``[P, block_size, nkv, hd]`` (values);
    block_table ``[n_pages]``; lists ``[rows, topk]``. Returns
    ``(out [rows, nq, hd], status)``.
    """
    q = np.asarray(q, dtype=np.float64)
    kc = np.asarray(k_cache, dtype=np.float64)
    vc = np.asarray(v_cache, dtype=np.float64)
    table = np.asarray(block_table).reshape(-1)
    lists = np.asarray(lists).reshape(q.shape[0], -1)
    rows, nq, hd = q.shape
    P, block_size, nkv, _ = kc.shape
    out = np.zeros((rows, nq, hd), dtype=np.float64)
    status = 0
    for r in range(rows):
        p = first_pos + r
        ncomp = (p + 1) // ratio
        tokens = []
        for b in lists[r]:
            if 0 <= b < ncomp:
                tokens.extend(range(int(b) * ratio, int(b) * ratio + ratio))
        tokens.extend(range(ncomp * ratio, p + 1))
        keep = []
        for t in tokens:
            pg = t // block_size
            page = int(table[pg]) if pg < len(table) else -1
            if 0 <= page < P:
                keep.append((page, t % block_size))
            else:
                status |= STATUS_BAD_BLOCK
        if not keep:
            continue
        pages = np.array([k[0] for k in keep])
        slots = np.array([k[1] for k in keep])
        for h in range(nq):
            kv = h // (nq // nkv)
            K = kc[pages, slots, kv]              # [n_tokens, hd]
            V = vc[pages, slots, kv]
            s = (K @ q[r, h]) * inv_sqrt_d
            e = np.exp(s - s.max())
            out[r, h] = (e / e.sum()) @ V
    return out, status


def qsa_score(q, block_keys) -> np.ndarray:
    """qsa.rs, ``qsa_score``: ``scores[b] = sum_h relu(q_h . k_b) / sqrt(hd)``."""
    q = np.asarray(q, dtype=np.float64)            # [n_heads, hd]
    kb = np.asarray(block_keys, dtype=np.float64)  # [n_blocks, hd]
    return np.maximum(kb @ q.T, 0.0).sum(axis=1) / math.sqrt(q.shape[1])


def expand_blocks(blocks, ratio: int) -> np.ndarray:
    """Token positions of selected blocks, for the gather.

    qsa.rs, ``qsa_gather``: slot ``i`` of the scratch holds position
    ``sel[i]``. The page does not fix the order of the selected blocks; the
    reading taken is ascending block order, each block expanded to its
    ``ratio`` positions in ascending order, ``-1`` after the last selected
    block. ``blocks``: ``[T, nb]`` block indices, ``-1`` for none.
    """
    blocks = np.asarray(blocks, dtype=np.int64)
    T, nb = blocks.shape
    out = np.full((T, nb * ratio), -1, dtype=np.int64)
    for t in range(T):
        sel = sorted(int(b) for b in blocks[t] if b >= 0)
        pos = [b * ratio + r for b in sel for r in range(ratio)]
        out[t, :len(pos)] = pos
    return out


def gather_kv(sel, block_table, bt_stride: int, max_lb: int, block_size: int,
              k_cache, v_cache):
    """Copy the selected rows of a paged K/V cache into a dense tile.

    qsa.rs, ``qsa_gather`` (slot ``i`` holds position ``sel[i]``) and commit
    c2f705a's gather (rows resolved through the block table). For position
    ``p``: ``phys = table[t][p // block_size]``, row ``p % block_size``.
    ``p < 0`` gives a zero row; a logical block outside the table or a
    physical block outside ``[0, P)`` also gives a zero row and sets a status
    bit. ``k_cache``/``v_cache``: ``[P, block_size, ...]`` of any dtype; the
    copy is of the stored elements, unchanged.
    """
    sel = np.asarray(sel, dtype=np.int64)
    kc, vc = np.asarray(k_cache), np.asarray(v_cache)
    T, n = sel.shape
    n_phys = kc.shape[0]
    flat = np.asarray(block_table, dtype=np.int64).reshape(-1)
    k_out = np.zeros((T, n) + kc.shape[2:], dtype=kc.dtype)
    v_out = np.zeros((T, n) + vc.shape[2:], dtype=vc.dtype)
    status = 0
    for t in range(T):
        for i in range(n):
            p = int(sel[t, i])
            if p < 0:
                continue
            lb = p // block_size
            if lb >= max_lb:
                status |= STATUS_BAD_SEL
                continue
            phys = int(flat[t * bt_stride + lb])
            if phys < 0 or phys >= n_phys:
                status |= STATUS_BAD_BLOCK
                continue
            k_out[t, i] = kc[phys, p % block_size]
            v_out[t, i] = vc[phys, p % block_size]
    return k_out, v_out, status


def bf16_round(x) -> np.ndarray:
    """float32 values -> bf16 bit patterns, rounded to nearest, ties to even
    (finite inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def gather_split(sel, block_table, bt_stride: int, max_lb: int, block_size: int, nope, nope_scale, rope):
    """The dense-tile gather of commit c2f705a (gather_kv.cu): rows of a paged
    cache split into an FP8 part and a BF16 part, FP8 dequantised to BF16.

    Layout reading (the commit gives none): per token ``nope_dim`` E4M3
    bytes, an optional float32 scale, ``rope_dim`` bf16 values; output row =
    ``bf16_rn(float32(e4m3) * scale)`` followed by the rope part unchanged.
    Positions resolve as in :func:`gather_kv`. Returns ``(out bf16 bits
    [T, n_sel, nope_dim + rope_dim], status)``.
    """
    nope = np.asarray(nope, dtype=np.uint8)
    rope = np.asarray(rope, dtype=np.uint16)
    P, bs, nope_dim = nope.shape
    rope_dim = rope.shape[2]
    scale = np.ones((P, bs), np.float32) if nope_scale is None else np.asarray(nope_scale, np.float32)
    # every (phys, row) dequantised once: float32 product, then bf16 rounding
    deq = bf16_round(e4m3_decode(nope).astype(np.float32) * scale[:, :, None])
    rows = np.concatenate([deq, rope], axis=2)          # [P, bs, nope_dim + rope_dim] bf16 bits
    out, _, status = gather_kv(sel, block_table, bt_stride, max_lb, block_size, rows, rows)
    return out, status
