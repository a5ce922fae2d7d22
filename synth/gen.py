"""Seeded draws: N(0,1) bf16, U(0,1) fp32, N(0,1) FP8-E4M3 (torch cast).

The FP8 inputs (indexer queries and keys) are *given* in E4M3 by the
workloads; the cast used to produce them here is torch's own
``float32 -> float8_e4m3fn`` conversion, i.e. part of input generation, not
of the method under test.
"""
from __future__ import annotations

import torch

# Stream ids: one per logical input tensor, so each can be regenerated alone.
STREAMS = {
    "kv": 1,          # main KV rows (bf16, pre-quantisation)
    "kI": 2,          # indexer keys (E4M3)
    "kI_bias": 3,     # Bernoulli mask for the +3 sigma indexer-key bias
    "qI": 4,          # indexer queries (E4M3), per layer
    "w": 5,           # indexer head weights U(0,1), per layer
    "q": 6,           # main queries (bf16), per layer
    "swa": 7,         # sliding-window KV rows (bf16), per layer
    "qI_pool": 8,     # pool-forming indexer query when no Full layer is present
    "w_pool": 9,
    "kv_new": 10,     # per-step appended rows
    "kI_new": 11,
    "swa_new": 12,
}


def gen_for(seed: int, stream: str | int, device="cpu", sub: int = 0) -> torch.Generator:
    sid = STREAMS[stream] if isinstance(stream, str) else int(stream)
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + sid * 10_007 + int(sub)) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def normal_bf16(shape, seed, stream, device="cpu", sub=0) -> torch.Tensor:
    g = gen_for(seed, stream, device, sub)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def uniform_f32(shape, seed, stream, device="cpu", sub=0) -> torch.Tensor:
    g = gen_for(seed, stream, device, sub)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def normal_e4m3(shape, seed, stream, device="cpu", sub=0) -> torch.Tensor:
    """N(0,1) drawn in fp32 and cast to E4M3; returned as raw uint8 bytes."""
    g = gen_for(seed, stream, device, sub)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def indexer_keys_e4m3(shape, seed, device="cpu", bias_prob=0.0, bias=3.0, sub=0) -> torch.Tensor:
    """Indexer keys [..., n, d_I] as E4M3 bytes.

    With ``bias_prob > 0`` a Bernoulli(bias_prob) draw per position adds
    ``bias`` (in units of the N(0,1) sigma) to every channel of that
    position's key before the FP8 cast, giving clear Top-K winners.
    """
    g = gen_for(seed, "kI", device, sub)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if bias_prob > 0:
        gb = gen_for(seed, "kI_bias", device, sub)
        m = torch.rand(shape[:-1], generator=gb, device=device, dtype=torch.float32) < bias_prob
        x += m.unsqueeze(-1).to(torch.float32) * bias
    return x.to(torch.float8_e4m3fn).view(torch.uint8)
