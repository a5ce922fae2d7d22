"""Workload shapes of the CSA2 decode/prefill configurations.

Symbols: B batch, n main-KV positions (compressed entries), d = 512 main
dim, H main query heads, H_I x d_I indexer heads x dim, k = 512 Top-K,
W = 128 sliding window, P = 2048 pool blocks of 8 positions.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Config:
    name: str
    workload: str
    B: int
    n: int                 # positions visible at the step (after the append)
    H: int = 64
    H_I: int = 8
    d_I: int = 128
    k: int = 512
    W: int = 128
    P: int = 2048
    d: int = 512
    bias_prob: float = 0.0
    groups: tuple = ()     # ((mode, n_reuse, form_pool), ...) with mode "full"/"reindex"
    steps: int = 1         # consecutive decode steps (stack config)
    n_start: int = 0       # positions cached before the first step (stack config)
    prefill_queries: int = 0
    ratio: int = 1         # compression ratio (tokens per main-KV entry)
    tokens: int = 1        # new tokens per sequence and step (multi-token decode)
    group_caches: bool = False   # each Full group keeps its own caches (the encoder's groups)
    extra: dict = field(default_factory=dict)


CONFIGS = {
    1: Config("cfg1", "full_layer_b1_n2048", B=1, n=2048, H=16, H_I=4, d_I=64,
              groups=(("full", 0, False),)),
    2: Config("cfg2", "decoder_group_full3reuse_b32_ctx131072", B=32, n=131072,
              bias_prob=0.05, groups=(("full", 3, False),)),
    3: Config("cfg3", "decoder_group_pool_reindex3reuse_b8_ctx1048576", B=8, n=1048576,
              groups=(("reindex", 3, True),)),
    4: Config("cfg4", "encoder_prefill_chunk4096_full5reuse_ratio2_ctx262144", B=1, n=131072,
              prefill_queries=4096, ratio=2, groups=(("full", 5, False),)),
    5: Config("cfg5", "decoder_stack20_b4_ctx1048576_256steps", B=4, n=1048576,
              n_start=1048320, steps=256,
              groups=(("full", 3, True),) + (("reindex", 3, False),) * 4),
    6: Config("cfg6", "decoder_group_full3reuse_b32x4tok_ctx131072", B=32, n=131072, bias_prob=0.05,
              groups=(("full", 3, False),), tokens=4),
    # the encoder's 18 layers: 3 groups of Full + 5 Reuse at ratio 2, each group
    # with its own main KV and indexer K (n = entries at the end)
    7: Config("cfg7", "encoder_stack18_ratio2_decode_b4_ctx262144_256steps", B=4, n=131072, ratio=2, steps=256,
              groups=(("full", 5, False),) * 3, group_caches=True),
    8: Config("cfg8", "encoder_stack18_prefill_chunk4096_ratio2_ctx262144", B=1, n=131072, prefill_queries=4096,
              ratio=2, groups=(("full", 5, False),) * 3, group_caches=True),
}


def get_config(i: int) -> Config:
    return CONFIGS[int(i)]
