"""The C ABI without a GPU: the library loads, exports every entry point that
include/idx.h declares, the ctypes mirrors match the C struct layout, and the
host-side validation rejects bad arguments before any device work."""

import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from sparse_attention_top_paged_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "idx.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from sparse_attention_top_paged_gb300 import build
        build.build()
    return _lib.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(idx_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("idx_score_topk", "idx_score_topk_workspace_size", "idx_gather_kv", "idx_block_pool",
              "idx_qsa_qprep", "idx_qsa_prefill_attn", "idx_gather_split", "idx_expand_blocks", "idx_valid_lens_from_blocks", "idx_status_string",
              "idx_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert lib.idx_version() >> 16 == 1
    assert lib.idx_status_string(0) == b"IDX_OK"
    assert lib.idx_status_string(3) == b"IDX_ERR_WORKSPACE_TOO_SMALL"


def test_struct_layout_matches_c():
    """Compile a C program against include/idx.h and compare sizeof/offsetof."""
    prog = r"""
#include <stdio.h>
#include <stddef.h>
#include "idx.h"
#define O(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  printf("idx_score_topk_args.size %zu\n", sizeof(idx_score_topk_args));
  printf("idx_gather_kv_args.size %zu\n", sizeof(idx_gather_kv_args));
  %FIELDS%
  return 0;
}
"""
    lines = []
    for struct, cls in (("idx_score_topk_args", _lib.ScoreTopkArgs), ("idx_gather_kv_args", _lib.GatherKvArgs)):
        for f, _ in cls._fields_:
            lines.append(f"O({struct}, {f})")
    prog = prog.replace("%FIELDS%", "\n  ".join(lines))
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write(prog)
        subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    got = dict(line.rsplit(" ", 1) for line in out.strip().splitlines())
    assert int(got["idx_score_topk_args.size"]) == ctypes.sizeof(_lib.ScoreTopkArgs)
    assert int(got["idx_gather_kv_args.size"]) == ctypes.sizeof(_lib.GatherKvArgs)
    for struct, cls in (("idx_score_topk_args", _lib.ScoreTopkArgs), ("idx_gather_kv_args", _lib.GatherKvArgs)):
        for f, _ in cls._fields_:
            assert int(got[f"{struct}.{f}"]) == getattr(cls, f).offset, (struct, f)


def _good_args():
    """Arguments that pass validation (fake, never-dereferenced addresses)."""
    a = _lib.ScoreTopkArgs()
    a.T, a.H, a.D = 4, 8, 128
    a.q, a.w = 0x10000, 0x20000
    a.key_format = _lib.KEYS_NVFP4
    a.keys_fp4, a.key_scale, a.key_gscale = 0x30000, 0x40000, 0x50000
    a.P, a.entries_per_block = 128, 64
    a.block_table, a.max_logical_blocks, a.bt_stride = 0x60000, 32, 32
    a.valid_lens, a.top_k = 0x70000, 64
    a.topk_idx, a.topk_score = 0x80000, 0x90000
    a.path, a.num_ctas = _lib.PATHS["simt"], 4
    return a


def _ws(lib, a):
    n = ctypes.c_size_t(0)
    st = lib.idx_score_topk_workspace_size(ctypes.byref(a), ctypes.byref(n))
    return st, n.value


def test_workspace_size_host_only(lib):
    a = _good_args()
    st, n = _ws(lib, a)
    assert st == 0 and n >= 4 * 32 * 64 * 4      # SIMT path holds the full score rows
    a.scores_out, a.ld_scores = 0xA0000, 32 * 64
    st, n = _ws(lib, a)
    assert st == 0 and n == 0                     # ... unless the caller supplies them


@pytest.mark.parametrize("field,value,code", [
    ("T", -1, 1), ("H", 0, 1), ("H", 257, 1), ("top_k", 0, 1), ("top_k", 4097, 1),
    ("P", 0, 1), ("entries_per_block", 0, 1), ("max_logical_blocks", 0, 1), ("bt_stride", -1, 1),
    ("D", 64, 2), ("entries_per_block", 24, 2), ("key_format", 7, 1), ("path", 9, 1),
    ("q", 0, 1), ("q", 0x10004, 1), ("keys_fp4", 0x30008, 1), ("topk_idx", 0, 1), ("num_ctas", -2, 1),
    ("q_format", 7, 1), ("q_format", 1, 2),   # NVFP4 q has no CUDA-core path
    ("q_dtype", 7, 1), ("q_dtype", 1, 2),     # bf16 q has no CUDA-core path
])
def test_validation_rejects(lib, field, value, code):
    a = _good_args()
    setattr(a, field, value)
    st, _ = _ws(lib, a)
    assert st == code
    assert lib.idx_score_topk(ctypes.byref(a), None) == code


def test_tensor_path_rejects_f32_keys(lib):
    a = _good_args()
    a.key_format, a.keys_f32 = _lib.KEYS_F32, 0x30000
    a.path = _lib.PATHS["tensor"]
    assert _ws(lib, a)[0] == 2


def test_scores_out_ld_checked(lib):
    a = _good_args()
    a.scores_out, a.ld_scores = 0xA0000, 32 * 64 - 1
    assert _ws(lib, a)[0] == 1


def test_workspace_too_small(lib):
    a = _good_args()
    a.workspace, a.workspace_bytes = 0x100000, 16
    assert lib.idx_score_topk(ctypes.byref(a), None) == 3


def test_empty_calls_launch_nothing(lib):
    a = _good_args()
    a.T = 0
    assert lib.idx_score_topk(ctypes.byref(a), None) == 0
    assert lib.idx_block_pool(None, None, None, 0, 0, 16, 128, 64, ctypes.c_float(1e6), ctypes.c_float(1e-6), None) == 0
    assert lib.idx_expand_blocks(None, 0, 4, 16, None, None) == 0
    assert lib.idx_valid_lens_from_blocks(None, 0, 64, None, None) == 0
    f = ctypes.c_float
    assert lib.idx_qsa_qprep(None, None, None, 0, 5, 4096, 32, 128, 64, f(1e6), f(1e-6), None) == 0
    assert lib.idx_qsa_qprep(None, None, None, 3, 5, 4096, 0, 128, 64, f(1e6), f(1e-6), None) == 0
    assert lib.idx_qsa_prefill_attn(None, None, None, None, 4, 4, None, None, 0, 0, 64, 16, 16, 32, 4, 128,
                                    f(0.088), None, None) == 0
    g = _lib.GatherKvArgs()
    g.T, g.n_sel, g.max_logical_blocks, g.P, g.block_size, g.row_bytes = 0, 5, 1, 1, 16, 1024
    assert lib.idx_gather_kv(ctypes.byref(g), None) == 0
    sp = _lib.GatherSplitArgs()
    sp.T, sp.n_sel, sp.max_logical_blocks, sp.P, sp.block_size, sp.nope_dim, sp.rope_dim = 0, 5, 1, 1, 16, 512, 64
    assert lib.idx_gather_split(ctypes.byref(sp), None) == 0


def test_other_entry_points_validate(lib):
    assert lib.idx_block_pool(None, None, None, 0, 1, 16, 100, 64, ctypes.c_float(1e6), ctypes.c_float(1e-6), None) == 1
    assert lib.idx_block_pool(None, None, None, 0, 1, 16, 128, 63, ctypes.c_float(1e6), ctypes.c_float(1e-6), None) == 1
    assert lib.idx_expand_blocks(None, 1, 4097, 16, None, None) == 1
    f = ctypes.c_float
    assert lib.idx_qsa_qprep(None, None, None, 1, 0, 4096, 32, 100, 64, f(1e6), f(1e-6), None) == 1   # hd % 32
    assert lib.idx_qsa_qprep(None, None, None, 1, 0, 4096, 32, 128, 63, f(1e6), f(1e-6), None) == 1   # odd rot
    assert lib.idx_qsa_qprep(None, None, None, 1, 0, 4000, 32, 128, 64, f(1e6), f(1e-6), None) == 1   # qkw too small
    assert lib.idx_qsa_qprep(None, None, None, 1, 0, 4096, 32, 128, 64, f(1e6), f(1e-6), None) == 1   # null pointers
    pa = lambda hd, nq, nkv: lib.idx_qsa_prefill_attn(None, None, None, None, 4, 4, None, None, 1, 0, 64, 16, 16,
                                                      nq, nkv, hd, f(0.088), None, None)
    assert pa(96, 32, 4) == 1 and pa(128, 30, 4) == 1 and pa(128, 32, 0) == 1 and pa(128, 32, 4) == 1
    assert lib.idx_valid_lens_from_blocks(None, 1, 0, None, None) == 1
    g = _lib.GatherKvArgs()
    g.T, g.n_sel, g.max_logical_blocks, g.P, g.block_size, g.row_bytes = 1, 5, 1, 1, 16, 1000
    assert lib.idx_gather_kv(ctypes.byref(g), None) == 1
    sp = _lib.GatherSplitArgs()
    sp.T, sp.n_sel, sp.max_logical_blocks, sp.P, sp.block_size, sp.nope_dim, sp.rope_dim = 1, 5, 1, 1, 16, 510, 64
    assert lib.idx_gather_split(ctypes.byref(sp), None) == 1      # nope_dim not a multiple of 4
    sp.nope_dim, sp.rope_dim = 512, 63
    assert lib.idx_gather_split(ctypes.byref(sp), None) == 1      # odd rope_dim
    sp.rope_dim = 64
    assert lib.idx_gather_split(ctypes.byref(sp), None) == 1      # null pointers
    assert lib.idx_gather_split(None, None) == 1


def test_quantize_q_nvfp4_validation_host_only(lib):
    q = ctypes.c_void_p
    assert lib.idx_quantize_q_nvfp4(q(0x10000), 0, q(0x20000), q(0x30000), q(0x40000), None) == 0   # nothing to do
    assert lib.idx_quantize_q_nvfp4(q(0x10000), -1, q(0x20000), q(0x30000), q(0x40000), None) == 1
    assert lib.idx_quantize_q_nvfp4(None, 4, q(0x20000), q(0x30000), q(0x40000), None) == 1
    assert lib.idx_quantize_q_nvfp4(q(0x10008), 4, q(0x20000), q(0x30000), q(0x40000), None) == 1   # q 16-byte aligned
