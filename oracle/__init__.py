"""CPU oracle for the CSA2 FP4-KV hot path.

TEST INFRASTRUCTURE. Nothing on the product path may import, call, link or
execute this package: only the tests, the smoke check and the benchmark's
CPU-baseline leg use it. It shares no code with the CUDA library (no common
kernels, headers, helpers, tables or constant generators) and never imports
it.

It is a plain, slow, obviously correct restatement of what the pages
describe, in numpy float64, step by step, with no blocking, fusion or
reordering beyond the definitions. Page citations used in this package:

[CSA2]  wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash с
        контекстом в 1 млн токенов, KV-кэшем FP4 и повторным использованием
        внимания между слоями", section "Сжатое разреженное внимание 2
        (CSA2)": the three static layer modes (Full / Reindex / Reuse),
        Top-512, per-layer main Q and SWA KV, the hierarchical pool of up to
        2048 blocks of 8 positions formed by the Full layer.
[FP4]   same page, section "FP4 KV, ограниченное повторное проигрывание и
        другие расширения": main KV in E2M1 with one E4M3 scale per 16
        channels, NVFP4-style but without the global scale.
[CED]   same page, section "Каузальный энкодер-декодер: вдвое меньший
        префилл": 128-token sliding-window attention in every layer.
[TG]    tgviewer.app, "DeepSeek-V4.1-Flash: Frontier Agents on a Smaller
        Memory Budget", CSA2 bullet: sharing Top-K indices removes
        re-scoring the whole history.

Where the pages are silent the oracle takes the plainest reading and says
so in the docstring of the function concerned:
  * indexer score s_t = sum_h w_h * relu(q_h . k_t), one key per position
    shared by all indexer heads, no 1/sqrt(d) factor;
  * FP4 scale = E4M3(amax/6) rounded to nearest even, saturating; a group
    whose scale rounds to zero stores all-zero codes;
  * block mean = E4M3 of the exact mean of the block's present keys;
  * Top-K order: score descending, then position ascending; the output is
    sorted by position and padded with -1;
  * main K = V (one shared vector per position), softmax scale 1/sqrt(512),
    SWA keys are distinct keys (no de-duplication against the sparse set).

Parity unpinned against the real model: the pages print no worked values,
and there are no trained weights; every pin is against format definitions,
closed forms, library routines, invariants and brute force.
"""
from .formats import (
    E2M1_GRID,
    E4M3_MAX,
    bf16_bits_to_f64,
    e4m3_decode,
    e4m3_encode,
    e2m1_encode_mag,
)
from .csa2 import (
    quantize_fp4,
    dequant_fp4,
    indexer_scores,
    block_means,
    topk_select,
    full_topk,
    form_pool,
    form_pool_block_max,
    pool_positions,
    reindex_topk,
    sparse_attention,
    layer_group,
    prefill_visible,
    swa_ring_after,
    prefill_swa_rows,
)

__all__ = [
    "E2M1_GRID", "E4M3_MAX", "bf16_bits_to_f64", "e4m3_decode", "e4m3_encode",
    "e2m1_encode_mag", "quantize_fp4", "dequant_fp4", "indexer_scores",
    "block_means", "topk_select", "full_topk", "form_pool", "form_pool_block_max",
    "pool_positions", "reindex_topk", "sparse_attention", "layer_group", "prefill_visible",
    "prefill_swa_rows", "swa_ring_after",
]
