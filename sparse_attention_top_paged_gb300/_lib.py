"""ctypes binding of libidx (include/idx.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels. PyTorch
supplies device memory and the current stream. There is no fallback: when
``libidx.so`` is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libidx.so")

IDX_OK = 0
STATUS_NAMES = {0: "IDX_OK", 1: "IDX_ERR_INVALID_ARG", 2: "IDX_ERR_UNSUPPORTED",
                3: "IDX_ERR_WORKSPACE_TOO_SMALL", 4: "IDX_ERR_CUDA"}
KEYS_NVFP4, KEYS_F32 = 0, 1
PATHS = {"auto": 0, "tensor": 1, "simt": 2}
Q_FORMATS = {"exact": 0, "nvfp4": 1}
Q_F32, Q_BF16 = 0, 1
STATUS_BAD_BLOCK, STATUS_BAD_LEN, STATUS_BAD_SEL, STATUS_TIMEOUT, STATUS_DEBUG_BOUNDS = 1, 2, 4, 8, 16
STATIC_SCRATCH_BYTES = 8 << 20

c_i32, c_i64, c_u32, c_size, c_f32, c_vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                             ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p)


class ScoreTopkArgs(ctypes.Structure):
    """Mirror of ``idx_score_topk_args``."""
    _fields_ = [
        ("T", c_i32), ("H", c_i32), ("D", c_i32),
        ("q", c_vp), ("w", c_vp),
        ("key_format", c_i32),
        ("keys_fp4", c_vp), ("key_scale", c_vp), ("key_gscale", c_vp), ("keys_f32", c_vp),
        ("P", c_i32), ("entries_per_block", c_i32),
        ("block_table", c_vp), ("max_logical_blocks", c_i32), ("bt_stride", c_i64),
        ("valid_lens", c_vp),
        ("top_k", c_i32),
        ("topk_idx", c_vp), ("topk_score", c_vp),
        ("scores_out", c_vp), ("ld_scores", c_i64),
        ("dev_status", c_vp),
        ("workspace", c_vp), ("workspace_bytes", c_size),
        ("path", c_i32), ("num_ctas", c_i32),
        ("timing_events", c_vp * 2),
        ("q_format", c_i32),
        ("q_dtype", c_i32),
    ]


class GatherKvArgs(ctypes.Structure):
    """Mirror of ``idx_gather_kv_args``."""
    _fields_ = [
        ("T", c_i32), ("n_sel", c_i32),
        ("sel", c_vp), ("block_table", c_vp),
        ("max_logical_blocks", c_i32), ("bt_stride", c_i64),
        ("P", c_i32), ("block_size", c_i32),
        ("k_cache", c_vp), ("v_cache", c_vp), ("row_bytes", c_i64),
        ("k_out", c_vp), ("v_out", c_vp),
        ("dev_status", c_vp),
    ]


class GatherSplitArgs(ctypes.Structure):
    """Mirror of ``idx_gather_split_args``."""
    _fields_ = [
        ("T", c_i32), ("n_sel", c_i32),
        ("sel", c_vp), ("block_table", c_vp),
        ("max_logical_blocks", c_i32), ("bt_stride", c_i64),
        ("P", c_i32), ("block_size", c_i32),
        ("nope", c_vp), ("nope_scale", c_vp), ("rope", c_vp),
        ("nope_dim", c_i32), ("rope_dim", c_i32),
        ("out", c_vp), ("dev_status", c_vp),
    ]


class IndexerError(RuntimeError):
    def __init__(self, where: str, code: int):
        super().__init__(f"{where} failed: {STATUS_NAMES.get(code, code)}")
        self.code = code


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libidx.so (built in-tree by ``build.build()``) and declare its
    signatures. Raises OSError when the library is absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise OSError(f"libidx.so not found at {p}: run sparse_attention_top_paged_gb300.build.build()")
        lib = ctypes.CDLL(p)
        P = ctypes.POINTER
        lib.idx_score_topk_workspace_size.argtypes = [P(ScoreTopkArgs), P(c_size)]
        lib.idx_score_topk_workspace_size.restype = c_i32
        lib.idx_score_topk.argtypes = [P(ScoreTopkArgs), c_vp]
        lib.idx_score_topk.restype = c_i32
        lib.idx_score_topk_static.argtypes = [P(ScoreTopkArgs), c_vp]
        lib.idx_score_topk_static.restype = c_i32
        lib.idx_quantize_q_nvfp4.argtypes = [c_vp, c_i64, c_vp, c_vp, c_vp, c_vp]
        lib.idx_quantize_q_nvfp4.restype = c_i32
        lib.idx_gather_kv.argtypes = [P(GatherKvArgs), c_vp]
        lib.idx_gather_kv.restype = c_i32
        lib.idx_gather_split.argtypes = [P(GatherSplitArgs), c_vp]
        lib.idx_gather_split.restype = c_i32
        lib.idx_block_pool.argtypes = [c_vp, c_vp, c_vp, c_u32, c_u32, c_u32, c_u32, c_u32, c_f32, c_f32, c_vp]
        lib.idx_block_pool.restype = c_i32
        lib.idx_qsa_qprep.argtypes = [c_vp, c_vp, c_vp, c_u32, c_u32, c_u32, c_u32, c_u32, c_u32, c_f32, c_f32,
                                      c_vp]
        lib.idx_qsa_qprep.restype = c_i32
        lib.idx_qsa_prefill_attn.argtypes = [c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_u32, c_u32, c_u32,
                                             c_u32, c_u32, c_u32, c_u32, c_u32, c_f32, c_vp, c_vp]
        lib.idx_qsa_prefill_attn.restype = c_i32
        lib.idx_expand_blocks.argtypes = [c_vp, c_i32, c_i32, c_i32, c_vp, c_vp]
        lib.idx_expand_blocks.restype = c_i32
        lib.idx_valid_lens_from_blocks.argtypes = [c_vp, c_i32, c_i32, c_vp, c_vp]
        lib.idx_valid_lens_from_blocks.restype = c_i32
        lib.idx_status_string.argtypes = [c_i32]
        lib.idx_status_string.restype = ctypes.c_char_p
        lib.idx_version.argtypes = []
        lib.idx_version.restype = c_u32
        if path is None:
            _lib = lib
        return lib
