"""Float64 CPU oracle for the lightning indexer over a paged NVFP4 key pool.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may call it. It shares no code with the
CUDA path under ``sparse_attention_top_paged_gb300/``; the two meet only in
the seeded input arrays that ``sparse_attention_top_paged_gb300.workloads``
produces.

Every function states the passage of the source pages it follows:

* "indexer_score_topk.cu" (nvfp4-megamoe-kernel, dsv4/kernels/indexer):
  the header comment (CSA lightning indexer, eq. 16), the "FP4
  dequantization (NVFP4 scheme)" section, the "Min-heap for top-k" section,
  the "Main kernel" section and the "PyTorch binding" section.
* "Commit graph, dsv4/kernels/indexer": commits e74c844 (E2M1 lookup table),
  79ef87f (E2M1 decode fix) and c2f705a (score+top-k, gather KV,
  compute_valid_lens).
* "metrale_model_layers/layers/ops/qsa.rs": the doc comments of
  ``qsa_block_pool``, ``qsa_qprep``, ``qsa_qprep_rows``, ``qsa_score``,
  ``qsa_gather``, ``qsa_score_rows`` and ``qsa_prefill_attn``.

The NVFP4-q mode (queries quantised to NVFP4 for the FP4 tensor-core MMA the
header comment of "indexer_score_topk.cu" plans) is ``quantize_q_nvfp4`` /
``dequantize_q_nvfp4`` / ``nvfp4_q`` in ``indexer.py``; scores in that mode are
``score_topk_rows`` applied to ``nvfp4_q(q)``.

Parity status. Every function is pinned by ``tests/test_oracle_pins.py``
except the RoPE pairing convention inside ``block_pool`` and
``qsa_qprep_rows`` (the pages do not say which dimensions are paired): parity
unpinned for that convention; its special cases (identity at position 0, norm
preservation, rot=0) are pinned.
"""

from .indexer import (  # noqa: F401
    E2M1_MAGNITUDES,
    e2m1_decode,
    e4m3_decode,
    unpack_nibbles,
    resolve_slots,
    dequant_rows,
    index_scores,
    topk_sorted,
    score_topk,
    score_topk_rows,
    valid_lens_from_blocks,
    STATUS_BAD_BLOCK,
    STATUS_BAD_LEN,
    STATUS_BAD_SEL,
    NVFP4_Q_RANGE,
    e4m3_encode,
    e2m1_encode,
    quantize_q_nvfp4,
    dequantize_q_nvfp4,
    nvfp4_q,
)
from .qsa import (block_pool, qsa_qprep_rows, qsa_prefill_attn, qsa_score, gather_kv, gather_split,  # noqa: F401
                  bf16_round, expand_blocks)
