"""GB300-native lightning indexer over a paged NVFP4 key pool.

Python face of libidx (``include/idx.h``). Each function checks and marshals
its torch arguments and calls the library; outputs are allocated with torch on
the inputs' device, and work is queued on the current CUDA stream.

* :func:`score_topk`   -> ``idx_score_topk``   (scores, top-k indices and scores)
* :func:`gather_kv`    -> ``idx_gather_kv``    (selected K/V rows -> dense tile)
* :func:`gather_split` -> ``idx_gather_split`` (FP8 + BF16 split rows -> dense BF16 tile)
* :func:`block_pool`   -> ``idx_block_pool``   (QSA mean -> RMSNorm(1+w) -> RoPE)
* :func:`qsa_qprep`    -> ``idx_qsa_qprep``    (QSA query: RMSNorm(1+w) -> RoPE)
* :func:`qsa_prefill_attn` -> ``idx_qsa_prefill_attn`` (attention over selected blocks + tail)
* :func:`expand_blocks` -> ``idx_expand_blocks`` (selected blocks -> positions)
* :func:`valid_lens_from_blocks` -> ``idx_valid_lens_from_blocks``
"""

from __future__ import annotations

import ctypes

from . import _lib
from ._lib import (IndexerError, KEYS_F32, KEYS_NVFP4, PATHS, STATUS_BAD_BLOCK,  # noqa: F401
                   STATUS_BAD_LEN, STATUS_BAD_SEL, STATUS_DEBUG_BOUNDS, STATUS_TIMEOUT, load_library)

_workspaces: dict = {}


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype=None, dims=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {t.dim()}")


def _stream(device):
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _raise(where, code):
    if code != _lib.IDX_OK:
        raise IndexerError(where, code)


def _workspace(device, nbytes):
    """A workspace of at least ``nbytes`` on ``device``, reused across calls
    (the library needs no initialised contents)."""
    torch = _torch()
    key = (str(device),)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def make_score_args(q, w, block_table, valid_lens, top_k, *, entries_per_block, keys_fp4=None,
                    key_scale=None, key_gscale=None, keys_f32=None, bt_stride=None,
                    topk_idx=None, topk_score=None, scores_out=None, dev_status=None,
                    path="auto", num_ctas=0, q_format="exact"):
    """Build an ``idx_score_topk_args`` from torch tensors (no device work).
    ``q_format="nvfp4"`` selects the opt-in NVFP4 query mode."""
    torch = _torch()
    _check(q, "q", None, 3)
    if q.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("q must be float32 or bfloat16")
    _check(w, "w", torch.float32, 2)
    _check(block_table, "block_table", torch.int32, 2)
    _check(valid_lens, "valid_lens", torch.int32, 1)
    T, H, D = q.shape
    a = _lib.ScoreTopkArgs()
    a.T, a.H, a.D = T, H, D
    a.q, a.w = q.data_ptr(), w.data_ptr()
    if keys_f32 is not None:
        _check(keys_f32, "keys_f32", torch.float32, 3)
        a.key_format = KEYS_F32
        a.keys_f32 = keys_f32.data_ptr()
        a.P = keys_f32.shape[0]
    else:
        _check(keys_fp4, "keys_fp4", torch.uint8, 3)
        _check(key_scale, "key_scale", torch.uint8, 3)
        _check(key_gscale, "key_gscale", torch.float32, 1)
        a.key_format = KEYS_NVFP4
        a.keys_fp4, a.key_scale, a.key_gscale = keys_fp4.data_ptr(), key_scale.data_ptr(), key_gscale.data_ptr()
        a.P = keys_fp4.shape[0]
    a.entries_per_block = entries_per_block
    a.block_table = block_table.data_ptr()
    a.max_logical_blocks = block_table.shape[1]
    a.bt_stride = block_table.shape[1] if bt_stride is None else bt_stride
    a.valid_lens = valid_lens.data_ptr()
    a.top_k = top_k
    if topk_idx is not None:
        a.topk_idx = topk_idx.data_ptr()
    if topk_score is not None:
        a.topk_score = topk_score.data_ptr()
    if scores_out is not None:
        _check(scores_out, "scores_out", torch.float32, 2)
        a.scores_out = scores_out.data_ptr()
        a.ld_scores = scores_out.shape[1]
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32)
        a.dev_status = dev_status.data_ptr()
    a.path = PATHS[path]
    a.num_ctas = num_ctas
    a.q_format = _lib.Q_FORMATS[q_format]
    a.q_dtype = _lib.Q_BF16 if q.dtype == torch.bfloat16 else _lib.Q_F32
    return a


def score_topk(q, w, block_table, valid_lens, top_k, *, entries_per_block, keys_fp4=None,
               key_scale=None, key_gscale=None, keys_f32=None, bt_stride=None, scores_out=None,
               dev_status=None, path="auto", num_ctas=0, out=None, workspace=None, q_format="exact"):
    """Top-k lightning-indexer keys per query: ``(topk_idx [T,k] int32,
    topk_score [T,k] float32)``. ``bt_stride=0`` shares table row 0 across
    queries. ``scores_out`` (``[T, ld]`` float32) also receives every score.
    ``q_format="nvfp4"``: score with q quantised to NVFP4 (opt-in; see
    :func:`quantize_q_nvfp4`)."""
    torch = _torch()
    T = q.shape[0]
    if out is None:
        topk_idx = torch.empty((T, top_k), dtype=torch.int32, device=q.device)
        topk_score = torch.empty((T, top_k), dtype=torch.float32, device=q.device)
    else:
        topk_idx, topk_score = out
    a = make_score_args(q, w, block_table, valid_lens, top_k, entries_per_block=entries_per_block,
                        keys_fp4=keys_fp4, key_scale=key_scale, key_gscale=key_gscale,
                        keys_f32=keys_f32, bt_stride=bt_stride, topk_idx=topk_idx,
                        topk_score=topk_score, scores_out=scores_out, dev_status=dev_status,
                        path=path, num_ctas=num_ctas, q_format=q_format)
    lib = load_library()
    with torch.cuda.device(q.device):
        need = ctypes.c_size_t(0)
        _raise("idx_score_topk_workspace_size", lib.idx_score_topk_workspace_size(ctypes.byref(a), ctypes.byref(need)))
        ws = workspace if workspace is not None else _workspace(q.device, need.value)
        a.workspace = ws.data_ptr()
        a.workspace_bytes = ws.numel() * ws.element_size()
        _raise("idx_score_topk", lib.idx_score_topk(ctypes.byref(a), _stream(q.device)))
    return topk_idx, topk_score


class ScoreTopkPlan:
    """A prepared ``idx_score_topk`` call for a serving loop: the arguments
    are checked and marshalled once, the outputs and the workspace allocated
    once, and every :meth:`run` is one library call on the current stream
    over whatever the bound tensors then hold (refill them in place between
    runs). :meth:`capture` records a step with its copies as one CUDA graph.
    Arguments as for :func:`score_topk`."""

    def __init__(self, q, w, block_table, valid_lens, top_k, *, entries_per_block, keys_fp4=None,
                 key_scale=None, key_gscale=None, keys_f32=None, bt_stride=None, scores_out=None,
                 dev_status=None, path="auto", num_ctas=0, out=None, workspace=None, q_format="exact"):
        torch = _torch()
        T = q.shape[0]
        if out is None:
            out = (torch.empty((T, top_k), dtype=torch.int32, device=q.device),
                   torch.empty((T, top_k), dtype=torch.float32, device=q.device))
        self.topk_idx, self.topk_score = out
        self._keep = (q, w, block_table, valid_lens, keys_fp4, key_scale, key_gscale, keys_f32, scores_out,
                      dev_status)
        self.args = make_score_args(q, w, block_table, valid_lens, top_k, entries_per_block=entries_per_block,
                                    keys_fp4=keys_fp4, key_scale=key_scale, key_gscale=key_gscale,
                                    keys_f32=keys_f32, bt_stride=bt_stride, topk_idx=self.topk_idx,
                                    topk_score=self.topk_score, scores_out=scores_out, dev_status=dev_status,
                                    path=path, num_ctas=num_ctas, q_format=q_format)
        self.device = q.device
        self._lib = load_library()
        with torch.cuda.device(q.device):
            need = ctypes.c_size_t(0)
            _raise("idx_score_topk_workspace_size",
                   self._lib.idx_score_topk_workspace_size(ctypes.byref(self.args), ctypes.byref(need)))
            self.workspace = workspace if workspace is not None else torch.empty(
                max(need.value, 256), dtype=torch.uint8, device=q.device)
        if self.workspace.numel() * self.workspace.element_size() < need.value:
            raise ValueError("workspace smaller than idx_score_topk_workspace_size")
        self.args.workspace = self.workspace.data_ptr()
        self.args.workspace_bytes = self.workspace.numel() * self.workspace.element_size()
        self._args_ref = ctypes.byref(self.args)

    def run(self, stream=None):
        """One call on ``stream`` (a torch.cuda.Stream; default: the current
        stream of the plan's device). Returns (topk_idx, topk_score)."""
        torch = _torch()
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        _raise("idx_score_topk", self._lib.idx_score_topk(self._args_ref, ctypes.c_void_p(s.cuda_stream)))
        return self.topk_idx, self.topk_score

    def capture(self, before=None, after=None):
        """Record one serving step as a CUDA graph: ``before()`` (e.g. the
        step's host-to-device copies into the bound inputs, from pinned
        buffers), this plan's call, then ``after()`` (e.g. the copies of the
        outputs back to pinned host buffers). Returns the torch CUDAGraph;
        each ``replay()`` runs the step on the current stream over whatever
        the pinned and bound buffers then hold, with one host launch."""
        torch = _torch()
        with torch.cuda.device(self.device):
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):   # one call outside the capture sets the kernels' attributes
                self.run()
            torch.cuda.current_stream().wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                if before is not None:
                    before()
                self.run()
                if after is not None:
                    after()
        return graph


def quantize_q_nvfp4(q):
    """The NVFP4 query quantisation of ``q_format="nvfp4"`` on its own:
    ``q [..., 128]`` float32 -> ``(codes [..., 64] uint8, scales [..., 8]
    uint8 E4M3, gscale [...] float32)``; codes pack element 2j in the low
    nibble of byte j."""
    torch = _torch()
    if q.dtype != torch.float32 or q.shape[-1] != 128 or not q.is_cuda:
        raise ValueError("q must be a CUDA float32 tensor with a last dimension of 128")
    q = q.contiguous()
    lead = tuple(q.shape[:-1])
    rows = q.numel() // 128
    codes = torch.empty(lead + (64,), dtype=torch.uint8, device=q.device)
    scales = torch.empty(lead + (8,), dtype=torch.uint8, device=q.device)
    gscale = torch.empty(lead, dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        _raise("idx_quantize_q_nvfp4", load_library().idx_quantize_q_nvfp4(
            q.data_ptr(), rows, codes.data_ptr(), scales.data_ptr(), gscale.data_ptr(), _stream(q.device)))
    return codes, scales, gscale


def score_topk_workspace_bytes(args) -> int:
    need = ctypes.c_size_t(0)
    _raise("idx_score_topk_workspace_size",
           load_library().idx_score_topk_workspace_size(ctypes.byref(args), ctypes.byref(need)))
    return need.value


def gather_kv(sel, block_table, block_size, k_cache, v_cache=None, *, bt_stride=None,
              dev_status=None, out=None):
    """Dense ``[T, n_sel, ...]`` copies of the K (and V) cache rows at the
    positions ``sel [T, n_sel]`` (-1: zero row). Caches: ``[P, block_size, ...]``."""
    torch = _torch()
    _check(sel, "sel", torch.int32, 2)
    _check(block_table, "block_table", torch.int32, 2)
    _check(k_cache, "k_cache")
    if v_cache is not None:
        _check(v_cache, "v_cache")
    T, n = sel.shape
    row_shape = tuple(k_cache.shape[2:])
    if out is None:
        k_out = torch.empty((T, n) + row_shape, dtype=k_cache.dtype, device=k_cache.device)
        v_out = None if v_cache is None else torch.empty((T, n) + row_shape, dtype=v_cache.dtype, device=v_cache.device)
    else:
        k_out, v_out = out
    a = _lib.GatherKvArgs()
    a.T, a.n_sel = T, n
    a.sel, a.block_table = sel.data_ptr(), block_table.data_ptr()
    a.max_logical_blocks = block_table.shape[1]
    a.bt_stride = block_table.shape[1] if bt_stride is None else bt_stride
    a.P, a.block_size = k_cache.shape[0], block_size
    a.k_cache = k_cache.data_ptr()
    a.v_cache = v_cache.data_ptr() if v_cache is not None else None
    a.row_bytes = k_cache[0, 0].numel() * k_cache.element_size()
    a.k_out = k_out.data_ptr()
    a.v_out = v_out.data_ptr() if v_out is not None else None
    a.dev_status = dev_status.data_ptr() if dev_status is not None else None
    lib = load_library()
    with torch.cuda.device(k_cache.device):
        _raise("idx_gather_kv", lib.idx_gather_kv(ctypes.byref(a), _stream(k_cache.device)))
    return k_out, v_out


def gather_split(sel, block_table, block_size, nope, rope, nope_scale=None, *, bt_stride=None, dev_status=None,
                 out=None):
    """Dense bf16 ``[T, n_sel, nope_dim + rope_dim]`` rows at positions ``sel``
    (-1: zero row) from a paged cache split into FP8 E4M3 ``nope``
    (uint8 ``[P, block_size, nope_dim]``, optional float32 per-token
    ``nope_scale`` ``[P, block_size]``) and bf16 ``rope``
    (``[P, block_size, rope_dim]``)."""
    torch = _torch()
    _check(sel, "sel", torch.int32, 2)
    _check(block_table, "block_table", torch.int32, 2)
    _check(nope, "nope", torch.uint8, 3)
    _check(rope, "rope", dims=3)
    if rope.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError("rope must hold bf16 bit patterns (bfloat16 or 16-bit int)")
    if nope_scale is not None:
        _check(nope_scale, "nope_scale", torch.float32, 2)
    T, n = sel.shape
    P, bs, nope_dim = nope.shape
    rope_dim = rope.shape[2]
    o = out if out is not None else torch.empty((T, n, nope_dim + rope_dim), dtype=torch.bfloat16, device=sel.device)
    _check(o, "out", dims=3)
    a = _lib.GatherSplitArgs()
    a.T, a.n_sel = T, n
    a.sel, a.block_table = sel.data_ptr(), block_table.data_ptr()
    a.max_logical_blocks = block_table.shape[1]
    a.bt_stride = block_table.shape[1] if bt_stride is None else bt_stride
    a.P, a.block_size = P, block_size
    a.nope, a.rope = nope.data_ptr(), rope.data_ptr()
    a.nope_scale = nope_scale.data_ptr() if nope_scale is not None else None
    a.nope_dim, a.rope_dim = nope_dim, rope_dim
    a.out = o.data_ptr()
    if dev_status is not None:
        a.dev_status = dev_status.data_ptr()
    lib = load_library()
    with torch.cuda.device(sel.device):
        _raise("idx_gather_split", lib.idx_gather_split(ctypes.byref(a), _stream(sel.device)))
    return o


def block_pool(raw_keys, k_norm_w, block_keys, first_block, n_new, ratio, rot, theta, eps):
    """Pool blocks ``first_block .. first_block+n_new-1`` of ``raw_keys``
    (bf16 ``[n_tok, hd]``) into rows of ``block_keys`` (float32 ``[nb, hd]``)."""
    torch = _torch()
    _check(raw_keys, "raw_keys", dims=2)
    if raw_keys.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError("raw_keys must hold bf16 bit patterns (bfloat16 or 16-bit int)")
    _check(k_norm_w, "k_norm_w", torch.float32, 1)
    _check(block_keys, "block_keys", torch.float32, 2)
    hd = raw_keys.shape[1]
    if (first_block + n_new) * ratio > raw_keys.shape[0] or first_block + n_new > block_keys.shape[0]:
        raise ValueError("block range exceeds raw_keys or block_keys")
    lib = load_library()
    with torch.cuda.device(raw_keys.device):
        _raise("idx_block_pool", lib.idx_block_pool(
            _ptr(raw_keys), _ptr(k_norm_w), _ptr(block_keys), first_block, n_new, ratio, hd, rot,
            ctypes.c_float(theta), ctypes.c_float(eps), _stream(raw_keys.device)))
    return block_keys


def qsa_qprep(qk, q_norm_w, n_heads, rot, theta, eps, *, first_pos=0, out=None):
    """QSA query preparation: rows of the indexer projection ``qk`` (bf16
    ``[rows, qkw]``, head h's q at columns ``h*hd``) -> float32
    ``[rows, n_heads, hd]``, RMSNorm scaled by ``1 + q_norm_w`` then rope at
    positions ``first_pos + row``. A decode query is one row."""
    torch = _torch()
    _check(qk, "qk", dims=2)
    if qk.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError("qk must hold bf16 bit patterns (bfloat16 or 16-bit int)")
    _check(q_norm_w, "q_norm_w", torch.float32, 1)
    rows, qkw = qk.shape
    hd = q_norm_w.shape[0]
    q_out = out if out is not None else torch.empty((rows, n_heads, hd), dtype=torch.float32, device=qk.device)
    _check(q_out, "out", torch.float32, 3)
    lib = load_library()
    with torch.cuda.device(qk.device):
        _raise("idx_qsa_qprep", lib.idx_qsa_qprep(_ptr(qk), _ptr(q_norm_w), _ptr(q_out), rows, first_pos, qkw,
                                                  n_heads, hd, rot, theta, eps, _stream(qk.device)))
    return q_out


def qsa_prefill_attn(q, k_cache, v_cache, block_table, lists, first_pos, ratio, *, inv_sqrt_d=None,
                     dev_status=None, out=None):
    """Attention of prefill rows (``q`` float32 ``[rows, nq, hd]``, row r at
    position ``first_pos + r``) over the selected blocks ``lists`` (int32
    ``[rows, topk]``) plus the incomplete tail, from paged bf16 caches
    ``[P, block_size, nkv, hd]`` through ``block_table`` (int32 ``[n_pages]``).
    Returns float32 ``[rows, nq, hd]``."""
    import math
    torch = _torch()
    _check(q, "q", torch.float32, 3)
    for name, c in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check(c, name, dims=4)
        if c.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
            raise TypeError(f"{name} must hold bf16 bit patterns (bfloat16 or 16-bit int)")
    _check(block_table, "block_table", torch.int32, 1)
    _check(lists, "lists", torch.int32, 2)
    rows, nq, hd = q.shape
    P, block_size, nkv, _ = k_cache.shape
    topk = lists.shape[1]
    scale = 1.0 / math.sqrt(hd) if inv_sqrt_d is None else inv_sqrt_d
    attn = out if out is not None else torch.empty((rows, nq, hd), dtype=torch.float32, device=q.device)
    _check(attn, "out", torch.float32, 3)
    lib = load_library()
    with torch.cuda.device(q.device):
        _raise("idx_qsa_prefill_attn", lib.idx_qsa_prefill_attn(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[0], P,
            _ptr(lists) if topk > 0 else None, _ptr(attn), rows, first_pos, topk, ratio, block_size, nq, nkv, hd,
            scale, _ptr(dev_status), _stream(q.device)))
    return attn


def expand_blocks(blocks, ratio):
    """``[T, nb]`` selected block ids (-1 none) -> ``[T, nb*ratio]`` ascending positions."""
    torch = _torch()
    _check(blocks, "blocks", torch.int32, 2)
    T, nb = blocks.shape
    pos = torch.empty((T, nb * ratio), dtype=torch.int32, device=blocks.device)
    lib = load_library()
    with torch.cuda.device(blocks.device):
        _raise("idx_expand_blocks", lib.idx_expand_blocks(_ptr(blocks), T, nb, ratio, _ptr(pos),
                                                          _stream(blocks.device)))
    return pos


def valid_lens_from_blocks(block_lens, entries_per_block):
    torch = _torch()
    _check(block_lens, "block_lens", torch.int32, 1)
    out = torch.empty_like(block_lens)
    lib = load_library()
    with torch.cuda.device(block_lens.device):
        _raise("idx_valid_lens_from_blocks", lib.idx_valid_lens_from_blocks(
            _ptr(block_lens), block_lens.shape[0], entries_per_block, _ptr(out), _stream(block_lens.device)))
    return out
