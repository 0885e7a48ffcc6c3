"""Seeded synthetic inputs for the indexer, the QSA pooling and the K/V gather.

This module only draws random inputs of the documented shapes and value
distributions; it computes nothing of the method itself. Both the CUDA path
(tests, benchmark) and the float64 oracle take the arrays it returns.

Workloads (sizes as named; ``seed`` selects the draw):

* ``tiny_decode``: T=4, H=8, D=128, 2048 keys per query, 64 entries per
  block, 32 logical blocks per query taken from one seeded permutation of
  128 physical blocks, top_k=64; q, w ~ N(0,1) float32; global scale 1/2688.
* ``batched_decode``: T=64, H=64, valid lengths uniform in [8192, 32768],
  per-query tables (disjoint slices of one permutation) over 40000 blocks,
  top_k=512; q = bf16(N(0,1)) held as float32, w ~ N(0,1)/8.
* ``long_decode``: T=16, H=64, 262144 keys per query, disjoint tables over
  70000 blocks, top_k=2048; values as ``batched_decode``.
* ``prefill``: 4096 rows of one sequence sharing one table (row stride 0)
  of 128 blocks, row r scores (r + 28672) // 4 keys, H=64, top_k=2048.
* ``qsa``: 8192 raw bf16 keys (hd=128), pooling ratio 16, rot 64,
  theta 1e6, eps 1e-6, norm weight ~ N(0, 0.1); 32 query heads, top_k=64
  blocks; bf16 K/V caches [512 pages, 16, 4 kv heads, 128].

NVFP4 keys everywhere: each packed byte uniform over 0..255 (both nibbles
uniform over the 16 E2M1 codes); E4M3 group scales drawn uniform in
[2^-4, 2^2] and rounded to the nearest E4M3 value by torch's float8 cast.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

D_FP4 = 128
GSCALE = 1.0 / 2688.0


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def _to_bf16_values(x: np.ndarray) -> np.ndarray:
    """float32 array holding the bf16-rounded values of ``x``."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.to(torch.float32).numpy().copy()


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 array with the bf16 encodings of ``x`` (round to nearest even)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def nvfp4_pool(rng: np.random.Generator, P: int, epb: int, D: int = D_FP4,
               gscale=GSCALE, gscale_pow2_jitter: int = 0):
    """A paged NVFP4 key pool: ``keys_fp4 [P,epb,D/2] u8``, ``key_scale
    [P,epb,D/16] u8`` (E4M3), ``key_gscale [P] f32``. With
    ``gscale_pow2_jitter = j`` each block's global scale is ``gscale * 2^u``,
    ``u`` uniform in ``[-j, j]``."""
    keys_fp4 = rng.integers(0, 256, size=(P, epb, D // 2), dtype=np.uint8)
    key_scale = _to_e4m3_bytes(rng.uniform(2.0 ** -4, 2.0 ** 2, size=(P, epb, D // 16)))
    g = np.full(P, gscale, dtype=np.float64)
    if gscale_pow2_jitter:
        g = g * np.exp2(rng.integers(-gscale_pow2_jitter, gscale_pow2_jitter + 1, size=P))
    return keys_fp4, key_scale, g.astype(np.float32)


@dataclass
class ScoreWorkload:
    """Inputs of one score + top-k call (numpy, host memory)."""
    name: str
    q: np.ndarray            # [T, H, D] float32
    w: np.ndarray            # [T, H] float32
    block_table: np.ndarray  # [rows, max_lb] int32
    bt_stride: int           # elements between consecutive queries' rows (0: shared)
    valid_lens: np.ndarray   # [T] int32
    epb: int
    top_k: int
    keys_fp4: np.ndarray | None = None   # [P, epb, D/2] uint8
    key_scale: np.ndarray | None = None  # [P, epb, D/16] uint8
    key_gscale: np.ndarray | None = None  # [P] float32
    keys_f32: np.ndarray | None = None   # [P, epb, D] float32
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return self.q.shape[0]

    @property
    def H(self) -> int:
        return self.q.shape[1]

    @property
    def D(self) -> int:
        return self.q.shape[2]

    @property
    def max_lb(self) -> int:
        return self.block_table.shape[1]

    @property
    def P(self) -> int:
        return (self.keys_f32 if self.keys_f32 is not None else self.keys_fp4).shape[0]

    @property
    def pairs(self) -> int:
        """Scored (query, key) pairs: the sum of the valid lengths."""
        return int(np.asarray(self.valid_lens, dtype=np.int64).sum())

    def oracle_kwargs(self) -> dict:
        return dict(keys_fp4=self.keys_fp4, key_scale=self.key_scale,
                    key_gscale=self.key_gscale, keys_f32=self.keys_f32)


def decode_workload(name: str, seed: int, *, T: int, H: int, valid_lens, max_lb: int,
                    P: int, top_k: int, epb: int = 64, D: int = D_FP4,
                    q_bf16: bool = True, w_scale: float = 1.0 / 8.0,
                    gscale_pow2_jitter: int = 0) -> ScoreWorkload:
    """Per-query block tables: disjoint slices of one seeded permutation of the
    ``P`` physical blocks (needs ``T * max_lb <= P``)."""
    rng = _rng(seed)
    valid_lens = np.asarray(valid_lens, dtype=np.int32)
    assert T * max_lb <= P, "disjoint per-query tables need T * max_lb <= P"
    perm = rng.permutation(P).astype(np.int32)
    block_table = perm[:T * max_lb].reshape(T, max_lb).copy()
    keys_fp4, key_scale, key_gscale = nvfp4_pool(rng, P, epb, D, gscale_pow2_jitter=gscale_pow2_jitter)
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    if q_bf16:
        q = _to_bf16_values(q)
    w = (rng.standard_normal((T, H)) * w_scale).astype(np.float32)
    return ScoreWorkload(name, q, w, block_table, max_lb, valid_lens, epb, top_k,
                         keys_fp4, key_scale, key_gscale, meta={"seed": seed})


def tiny_decode(seed: int = 1000, *, gscale_pow2_jitter: int = 0) -> ScoreWorkload:
    rng = _rng(seed)
    T, H, D, epb, P, nlb = 4, 8, D_FP4, 64, 128, 32
    perm = rng.permutation(P).astype(np.int32)
    block_table = perm.reshape(T, nlb).copy()     # query t uses perm[32t : 32t+32]
    keys_fp4, key_scale, key_gscale = nvfp4_pool(rng, P, epb, D, gscale_pow2_jitter=gscale_pow2_jitter)
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    w = rng.standard_normal((T, H)).astype(np.float32)
    valid_lens = np.full(T, nlb * epb, dtype=np.int32)
    return ScoreWorkload("tiny_decode", q, w, block_table, nlb, valid_lens, epb, 64,
                         keys_fp4, key_scale, key_gscale, meta={"seed": seed})


def batched_decode(seed: int = 1001, *, T: int = 64, lo: int = 8192, hi: int = 32768,
                   P: int = 40000, max_lb: int = 512, top_k: int = 512, H: int = 64) -> ScoreWorkload:
    rng = _rng(seed + 7919)
    valid_lens = rng.integers(lo, hi + 1, size=T).astype(np.int32)
    return decode_workload("batched_decode", seed, T=T, H=H, valid_lens=valid_lens,
                           max_lb=max_lb, P=P, top_k=top_k)


def long_decode(seed: int = 1002, *, T: int = 16, S: int = 262144, P: int = 70000,
                top_k: int = 2048, H: int = 64) -> ScoreWorkload:
    max_lb = S // 64
    return decode_workload("long_decode", seed, T=T, H=H, valid_lens=np.full(T, S, np.int32),
                           max_lb=max_lb, P=P, top_k=top_k)


def prefill(seed: int = 1003, *, rows: int = 4096, ratio: int = 4, base: int = 28672,
            n_blocks: int = 128, H: int = 64, top_k: int = 2048) -> ScoreWorkload:
    """One table shared by every row (row stride 0); row r scores
    ``(r + base) // ratio`` keys."""
    rng = _rng(seed)
    epb, D = 64, D_FP4
    perm = rng.permutation(n_blocks).astype(np.int32)
    block_table = perm.reshape(1, n_blocks).copy()
    keys_fp4, key_scale, key_gscale = nvfp4_pool(rng, n_blocks, epb, D)
    q = _to_bf16_values(rng.standard_normal((rows, H, D)).astype(np.float32))
    w = (rng.standard_normal((rows, H)) / 8.0).astype(np.float32)
    valid_lens = ((np.arange(rows) + base) // ratio).astype(np.int32)
    assert valid_lens.max() <= n_blocks * epb
    return ScoreWorkload("prefill", q, w, block_table, 0, valid_lens, epb, top_k,
                         keys_fp4, key_scale, key_gscale, meta={"seed": seed})


@dataclass
class QsaWorkload:
    raw_keys_bits: np.ndarray   # [n_tok, hd] uint16 bf16 encodings
    raw_keys: np.ndarray        # [n_tok, hd] float32 values of those encodings
    k_norm_w: np.ndarray        # [hd] float32
    q: np.ndarray               # [n_heads, hd] float32
    k_cache_bits: np.ndarray    # [pages, block_size, nkv, hd] uint16 (bf16)
    v_cache_bits: np.ndarray
    page_table: np.ndarray      # [1, pages] int32
    q_raw_bits: np.ndarray = None   # [1, n_heads*hd] uint16 (bf16): the decode query's projection row
    q_norm_w: np.ndarray = None     # [hd] float32
    ratio: int = 16
    rot: int = 64
    theta: float = 1.0e6
    eps: float = 1.0e-6
    top_k: int = 64
    block_size: int = 16

    @property
    def n_blocks(self) -> int:
        return self.raw_keys.shape[0] // self.ratio


def qsa(seed: int = 1004, *, n_tok: int = 8192, hd: int = 128, n_heads: int = 32,
        nkv: int = 4, block_size: int = 16, ratio: int = 16, top_k: int = 64) -> QsaWorkload:
    rng = _rng(seed)
    raw = rng.standard_normal((n_tok, hd)).astype(np.float32)
    bits = _to_bf16_bits(raw)
    vals = _to_bf16_values(raw)
    k_norm_w = (rng.standard_normal(hd) * 0.1).astype(np.float32)
    q = rng.standard_normal((n_heads, hd)).astype(np.float32)
    pages = n_tok // block_size
    kc = _to_bf16_bits(rng.standard_normal((pages, block_size, nkv, hd)).astype(np.float32))
    vc = _to_bf16_bits(rng.standard_normal((pages, block_size, nkv, hd)).astype(np.float32))
    table = rng.permutation(pages).astype(np.int32).reshape(1, pages)
    # drawn last, so the fields above keep their values: the raw projection
    # row the decode query is prepared from, and its norm weight
    q_raw_bits = _to_bf16_bits(rng.standard_normal((1, n_heads * hd)).astype(np.float32))
    q_norm_w = (rng.standard_normal(hd) * 0.1).astype(np.float32)
    return QsaWorkload(bits, vals, k_norm_w, q, kc, vc, table, q_raw_bits, q_norm_w, ratio=ratio, top_k=top_k,
                       block_size=block_size)


CONFIGS = {
    "tiny_decode": tiny_decode,
    "batched_decode": batched_decode,
    "long_decode": long_decode,
    "prefill": prefill,
}
