"""Benchmark of the CSA2 FP4-KV decode hot path on one B300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl csa2|reference]

A step is one decode step of the configured CSA2 layer group(s) over a batch
of sequences whose caches are resident in HBM: append the new token (FP4
quantise of its main-KV row, indexer-key append + block mean, each layer's
SWA ring), then every group (Full or Reindex indexer, Top-512, sparse
attention of the first layer and of each Reuse layer). The default workload
(--config 2) is the decoder layer group Full + 3 Reuse at batch 32 and
131,072 positions, 64 heads, indexer 8 x 128. The metric is decode tokens/s
per layer group (one new token per sequence per step), with the Full
indexer scan's achieved HBM bandwidth as the roofline figure.

Inputs are seeded and synthetic (synth/). With --impl reference the CPU
oracle is timed instead, on a bounded sample of the same workload.
Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (sequences are independent; no data-path
collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 decode tokens/s per layer group at 128K/1M ctx; % of B300 HBM roofline"
UNIT = "tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6400.0
L2_FLUSH_BYTES = 256 << 20


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s): the measured cuBLAS burst, else the fallback."""
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (burst)"
    except Exception:
        return 1800.0, "fallback"


FP4_ROW_BYTES = 288          # 256 B of E2M1 codes + 32 B of E4M3 scales per main-KV row
SWA_ROW_BYTES = 1024         # one bf16 row of 512


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """Samples SM clock and clock-event (throttle) reasons of one GPU every
    20 ms with nvidia-smi (read-only queries; no GPU setting is changed).
    Start it before the warm-up; mark() the timed window; summary() reports
    the samples inside the window, or, if the window was too short to hold
    one, those of the whole warm-up + timed span (flagged as such)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""
        self.window = None

    def start(self):
        try:
            import torch
            idx = str(self.gpu)
            env = dict(os.environ)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, env=env)
            time.sleep(1.0)
        except Exception:
            self.proc = None
        return self

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    @staticmethod
    def _epoch(ts):
        import datetime
        try:
            return datetime.datetime.strptime(ts.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        rows, sm_max = [], None
        for ln in self.out.splitlines():
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 7:
                continue
            try:
                rows.append((self._epoch(p[0]), float(p[1]), [v.lower().startswith("active") for v in p[3:7]]))
                sm_max = float(p[2])
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": sm_max, "reasons": ["unavailable"], "samples": 0}
        inside = [r for r in rows if self.window and r[0] is not None and self.window[0] <= r[0] <= self.window[1]]
        use, span = (inside, "timed") if inside else (rows, "warmup+timed")
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = sorted({n for _, _, fl in use for n, f in zip(names, fl) if f})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": sm_max, "reasons": seen,
                "samples": len(use), "span": span}


# ---------------------------------------------------------------------------
# the workload
# ---------------------------------------------------------------------------
class PinnedArena:
    """Host buffers carved from one pinned allocation (at least 64 MiB), each
    view 512-byte aligned."""

    def __init__(self, torch, nbytes):
        self.torch = torch
        self.buf = torch.empty(max(int(nbytes), 64 << 20), dtype=torch.uint8).pin_memory()
        self.off = 0

    def empty_like(self, t):
        n = t.numel() * t.element_size()
        assert self.off + n <= self.buf.numel(), "pinned arena too small"
        v = self.buf[self.off:self.off + n].view(t.dtype).view(t.shape)
        self.off += (n + 511) & ~511
        return v

    def take(self, t):
        v = self.empty_like(t)
        v.copy_(t.cpu())
        return v


class PipelinedE2E:
    """End-to-end steps as a server runs them: while step i computes, the
    pinned host inputs of step i + 1 are copied in on one stream and the
    outputs of step i are copied out on another. Two device sets of the
    per-step inputs (the workload attributes named in `in_keys`) and of the
    outputs alternate; events keep a set from being overwritten while a step
    or a copy still uses it. Every step's input copy and output read-back runs
    inside the caller's timed region: `begin` issues step 0's copy, step i
    issues step i + 1's unless it is the last."""

    def __init__(self, wl, in_keys):
        torch = self.torch = wl.torch
        self.wl, self.keys = wl, in_keys
        clone = lambda v: [t.clone() for t in v] if isinstance(v, list) else v.clone()
        self.sets = [{k: getattr(wl, k) for k in in_keys}, {k: clone(getattr(wl, k)) for k in in_keys}]
        self.outs = [wl.out, [t.clone() for t in wl.out]]
        self.h2d, self.d2h = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
        self.in_ready, self.in_free, self.out_ready, self.out_free = ev(), ev(), ev(), ev()
        self.used = [False, False]                       # set s has run a step (its free events are recorded)
        self.i = 0

    def _copy_in(self, s):
        torch = self.torch
        with torch.cuda.stream(self.h2d):
            if self.used[s]:
                self.h2d.wait_event(self.in_free[s])
            for k in self.keys:
                dst, src = self.sets[s][k], self.wl.h_in[k]
                for d, h in (zip(dst, src) if isinstance(dst, list) else ((dst, src),)):
                    d.copy_(h, non_blocking=True)
            self.in_ready[s].record(self.h2d)

    def begin(self):
        """Start of a run of steps: step 0's inputs (after the caller's start
        event). The caller has joined the previous run (`end`), so no set is
        still in use."""
        self.h2d.wait_stream(self.torch.cuda.current_stream())
        self.d2h.wait_stream(self.torch.cuda.current_stream())
        self.used = [False, False]
        self.i = 0
        self._copy_in(0)

    def step(self, last):
        torch, wl = self.torch, self.wl
        s = self.i % 2
        cur = torch.cuda.current_stream()
        if not last:
            self._copy_in(1 - s)
        cur.wait_event(self.in_ready[s])
        if self.used[s]:
            cur.wait_event(self.out_free[s])             # step i - 2's outputs have been read back
        for k in self.keys:
            setattr(wl, k, self.sets[s][k])
        wl.out = self.outs[s]
        wl.step()
        self.in_free[s].record(cur)
        self.out_ready[s].record(cur)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.out_ready[s])
            for h, d in zip(wl.h_out, self.outs[s]):
                h.copy_(d, non_blocking=True)
            self.out_free[s].record(self.d2h)
        self.used[s] = True
        self.i += 1

    def end(self):
        """Join the copy streams into the caller's stream (before its end event)."""
        cur = self.torch.cuda.current_stream()
        cur.wait_stream(self.d2h)
        cur.wait_stream(self.h2d)

    def restore(self):
        """Bind the workload's original input and output tensors again."""
        for k in self.keys:
            setattr(self.wl, k, self.sets[0][k])
        self.wl.out = self.outs[0]


class DecodeWorkload:
    """Caches, per-layer inputs and the per-step calls of one decode config."""

    def __init__(self, cfg, device, seed=1234, batch=None, pool_rule="mean"):
        import torch
        import synth
        from fp4_kv_cache_06_b300 import csa2
        self.torch, self.csa2 = torch, csa2
        self.cfg = cfg
        self.pool_rule = pool_rule
        self.dev = device
        B = self.B = batch or cfg.B
        d_I, H_I, H, W, k, P = cfg.d_I, cfg.H_I, cfg.H, cfg.W, cfg.k, cfg.P
        self.n_end = cfg.n                               # positions visible after the last step
        self.n_first = cfg.n_start + 1 if cfg.steps > 1 else cfg.n
        self.n_cap = cfg.n
        n_pre = self.n_first - 1                         # positions cached before the first step
        self.layers = sum(1 + g[1] for g in cfg.groups)
        dev = device
        u8, i64, i32 = torch.uint8, torch.int64, torch.int32
        self.codes = torch.empty((B, self.n_cap, 256), dtype=u8, device=dev)
        self.scales = torch.empty((B, self.n_cap, 32), dtype=u8, device=dev)
        self.kI = torch.empty((B, self.n_cap, d_I), dtype=u8, device=dev)
        self.kbar = torch.zeros((B, (self.n_cap + 7) // 8, d_I), dtype=u8, device=dev)
        chunk = 1 << 17
        for b in range(B):                               # main KV: bf16 N(0,1) -> FP4 (resident)
            for c0 in range(0, n_pre, chunk):
                r = min(chunk, n_pre - c0)
                x = synth.normal_bf16((1, r, 512), seed, "kv", dev, sub=b * 4096 + c0 // chunk)
                csa2.csa2_quantize_kv_fp4(x, self.codes[b:b + 1], self.scales[b:b + 1],
                                          pos=torch.tensor([c0], dtype=i64, device=dev))
            self.kI[b, :n_pre] = synth.indexer_keys_e4m3((n_pre, d_I), seed, dev, bias_prob=cfg.bias_prob, sub=b)
        nt = torch.full((B,), n_pre, dtype=i64, device=dev)
        if n_pre > 0:
            csa2.csa2_block_means(self.kI, nt, self.kbar, n_max=n_pre)
        self.swa = [synth.normal_bf16((B, W, 512), seed, "swa", dev, sub=l) for l in range(self.layers)]
        self.q = [synth.normal_bf16((B, H, 512), seed, "q", dev, sub=l) for l in range(self.layers)]
        self.out = [torch.empty((B, H, 512), dtype=torch.bfloat16, device=dev) for _ in range(self.layers)]
        G = len(cfg.groups)
        self.qI = [synth.normal_e4m3((B, H_I, d_I), seed, "qI", dev, sub=g) for g in range(G)]
        self.w = [synth.uniform_f32((B, H_I), seed, "w", dev, sub=g) for g in range(G)]
        self.qI_pool = synth.normal_e4m3((B, H_I, d_I), seed, "qI_pool", dev)
        self.w_pool = synth.uniform_f32((B, H_I), seed, "w_pool", dev)
        self.kv_new = synth.normal_bf16((B, 512), seed, "kv_new", dev)
        self.kI_new = synth.indexer_keys_e4m3((B, d_I), seed + 1, dev, bias_prob=cfg.bias_prob)
        self.swa_new = [synth.normal_bf16((B, 512), seed, "swa_new", dev, sub=l) for l in range(self.layers)]
        self.idx = [torch.empty((B, k), dtype=i32, device=dev) for _ in range(G)]
        self.pool = torch.full((B, P), -1, dtype=i32, device=dev)
        self.pos = torch.full((B,), n_pre, dtype=i64, device=dev)
        self.n = torch.full((B,), n_pre + 1, dtype=i64, device=dev)
        self.swa_len = torch.full((B,), min(n_pre + 1, W), dtype=i32, device=dev)
        self.ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_LAYER_GROUP, B, self.n_cap, k, P, H), dev)
        self.step_i = 0
        torch.cuda.synchronize()

    def _rule(self, mode):
        """Pool rule of a group that forms the pool: a Full group may take the
        block maxima of its own scores; otherwise the blocks' mean keys."""
        if self.pool_rule == "max" and mode == "full":
            return self.csa2.POOL_BLOCK_MAX
        return self.csa2.POOL_MEAN_KEY

    def pool_recall(self):
        """Share of the pool-forming Full group's Top-k positions whose block is
        in the pool it formed (after the last step; None without such a group)."""
        torch = self.torch
        for g, (mode, _, form_pool) in enumerate(self.cfg.groups):
            if mode == "full" and form_pool:
                idx, pool = self.idx[g].long(), self.pool.long()
                hits = total = 0
                for b in range(idx.shape[0]):                # membership per query row
                    sel = idx[b][idx[b] >= 0]
                    hits += int(torch.isin(sel // 8, pool[b][pool[b] >= 0]).sum())
                    total += int(sel.numel())
                return round(hits / max(1, total), 6)
        return None

    def reset_positions(self):
        """Restart the step sequence (positions back to the first step's)."""
        self.step_i = 0
        self.pos.fill_(self.n_first - 1)
        self.n.fill_(self.n_first)

    def step(self, events=None):
        """One decode step; `events` (optional) = per-group lists of CUDA events."""
        csa2, cfg = self.csa2, self.cfg
        if self.step_i > 0 and self.cfg.steps > 1:
            self.pos.add_(1)
            self.n.add_(1)
        csa2.csa2_append_step(self.kv_new, self.kI_new, self.swa_new, self.swa, self.pos, self.codes,
                              self.scales, self.kI, self.kbar)
        n_max = self.n_first + (self.cfg.steps - 1 if self.cfg.steps > 1 else 0)
        n_max = min(n_max, self.n_cap)
        l0 = 0
        for g, (mode, n_reuse, form_pool) in enumerate(cfg.groups):
            L = 1 + n_reuse
            csa2.csa2_layer_group(
                csa2.MODE_FULL if mode == "full" else csa2.MODE_REINDEX, self.n, n_max, self.codes, self.scales,
                self.kI, self.qI[g], self.w[g], self.idx[g], self.q[l0:l0 + L], self.swa[l0:l0 + L], self.swa_len,
                self.out[l0:l0 + L], self.ws, kbar=self.kbar, pool=self.pool,
                form_pool=self._rule(mode) if form_pool else csa2.POOL_NONE,
                qI_pool=self.qI_pool if mode == "reindex" else None,
                w_pool=self.w_pool if mode == "reindex" else None,
                events=None if events is None else events[g])
            l0 += L
        self.step_i += 1

    def alg_bytes(self):
        """Algorithmic bytes of one step by kind (the roofline numerators):
        indexer keys of every Full scan, block means of every pool formed on
        the mean-key rule, the pool slots of every Reindex scan, and, per
        layer, the gathered FP4 rows and the SWA rows."""
        cfg, B = self.cfg, self.B
        n = min(self.n_end, self.n_cap)
        d_I = cfg.d_I
        out = {"indexer_keys": 0, "block_means": 0, "pool_slots": 0}
        for mode, n_reuse, form_pool in cfg.groups:
            if mode == "full":
                out["indexer_keys"] += B * n * d_I
            if form_pool and not (mode == "full" and self.pool_rule == "max"):
                out["block_means"] += B * ((n + 7) // 8) * d_I
            if mode == "reindex":
                out["pool_slots"] += B * cfg.P * 8 * d_I
        out["gather"] = self.layers * B * cfg.k * FP4_ROW_BYTES
        out["swa"] = self.layers * B * cfg.W * SWA_ROW_BYTES
        return out

    def attn_launch_bytes(self, n_layers):
        """Algorithmic bytes of one attention launch over n_layers layers
        (each layer's gathered rows and SWA rows, as in alg_bytes)."""
        return n_layers * self.B * (self.cfg.k * FP4_ROW_BYTES + self.cfg.W * SWA_ROW_BYTES)

    def attn_launch_flops(self, n_layers):
        """4 H (k + W) d flops per row and layer (S and PV)."""
        return 4.0 * n_layers * self.B * self.cfg.H * (self.cfg.k + self.cfg.W) * 512

    def step_layerwise(self, events=None):
        """The same step with one attention launch per layer, each after the
        previous one (the schedule of a model whose next layer's query
        depends on this layer's output): the group call attends its first
        layer, then csa2_sparse_attn attends each Reuse layer. `events` as in
        step(); event 3 + l follows layer l's own launch."""
        csa2, cfg = self.csa2, self.cfg
        if self.step_i > 0 and self.cfg.steps > 1:
            self.pos.add_(1)
            self.n.add_(1)
        csa2.csa2_append_step(self.kv_new, self.kI_new, self.swa_new, self.swa, self.pos, self.codes,
                              self.scales, self.kI, self.kbar)
        n_max = self.n_first + (self.cfg.steps - 1 if self.cfg.steps > 1 else 0)
        n_max = min(n_max, self.n_cap)
        l0 = 0
        for g, (mode, n_reuse, form_pool) in enumerate(cfg.groups):
            ev = None if events is None else events[g]
            csa2.csa2_layer_group(
                csa2.MODE_FULL if mode == "full" else csa2.MODE_REINDEX, self.n, n_max, self.codes, self.scales,
                self.kI, self.qI[g], self.w[g], self.idx[g], self.q[l0:l0 + 1], self.swa[l0:l0 + 1], self.swa_len,
                self.out[l0:l0 + 1], self.ws, kbar=self.kbar, pool=self.pool,
                form_pool=self._rule(mode) if form_pool else csa2.POOL_NONE,
                qI_pool=self.qI_pool if mode == "reindex" else None,
                w_pool=self.w_pool if mode == "reindex" else None,
                events=None if ev is None else ev[:4])
            for r in range(n_reuse):
                l = l0 + 1 + r
                csa2.csa2_sparse_attn(self.q[l], self.codes, self.scales, self.idx[g], self.swa[l], self.swa_len,
                                      self.out[l], self.ws)
                if ev is not None:
                    ev[4 + r].record()
            l0 += 1 + n_reuse
        self.step_i += 1

    def scan_positions(self):
        """Positions the Full scans of one step read (for the roofline)."""
        return sum(self.B * min(self.n_end, self.n_cap) for (m, _, _) in self.cfg.groups if m == "full")

    tokens_per_step = property(lambda self: self.B)

    def scan_bytes(self, d_I):
        """Algorithmic bytes of one Full-scan launch: every indexer key once."""
        return self.B * min(self.n_end, self.n_cap) * d_I

    def scan_score_bytes(self):
        """The fp32 score the scan writes per query row and position."""
        return self.B * min(self.n_end, self.n_cap) * 4

    def pool_scan_bytes(self, d_I):
        """Algorithmic bytes of one block-mean scan (pool formation)."""
        return self.B * ((min(self.n_end, self.n_cap) + 7) // 8) * d_I

    # host-side step for the end-to-end figure: per-step inputs from pinned host memory
    def host_buffers(self):
        """Pinned host copies of the per-step inputs (E2E_INPUTS) and of the
        outputs, carved from one pinned arena: host-to-device copies from
        small, separately pinned buffers ran at about a quarter of the link's
        rate on the B300 hosts, from one large allocation at the full rate."""
        items = lambda v: v if isinstance(v, list) else [v]
        ins = {k: getattr(self, k) for k in self.E2E_INPUTS}
        size = lambda t: t.numel() * t.element_size()
        h2d = sum(size(t) for v in ins.values() for t in items(v))
        d2h = sum(size(t) for t in self.out)
        arena = PinnedArena(self.torch, h2d + d2h + 512 * (sum(len(items(v)) for v in ins.values()) + len(self.out)))
        self.h_in = {k: ([arena.take(t) for t in v] if isinstance(v, list) else arena.take(v)) for k, v in ins.items()}
        self.h_out = [arena.empty_like(t) for t in self.out]
        return h2d, d2h

    E2E_INPUTS = ("kv_new", "kI_new", "swa_new", "q", "qI", "w")


class MultiTokenWorkload(DecodeWorkload):
    """Multi-token decode: R new tokens of each of B sequences per step. The
    R rows are appended to the caches, then each layer group runs with one
    query row per token (rows_per_seq = R); every token sees the cache up to
    itself and attends over its own 128-token window. The windows' bf16 rows
    (W + R - 1 per sequence and layer) are per-step inputs, like the layer
    queries."""

    def __init__(self, cfg, device, seed=1234, batch=None, pool_rule="mean"):
        super().__init__(cfg, device, seed, batch, pool_rule)
        import synth
        torch = self.torch
        B, R = self.B, cfg.tokens
        self.R, self.rows = R, B * R
        rows, d_I, H_I, H, W, k, P = self.rows, cfg.d_I, cfg.H_I, cfg.H, cfg.W, cfg.k, cfg.P
        dev = self.dev
        n_pre = cfg.n - R                                # the step appends positions n_pre .. n_pre + R - 1
        G = len(cfg.groups)
        self.swa = [synth.normal_bf16((B, W + R - 1, 512), seed, "swa", dev, sub=l) for l in range(self.layers)]
        self.q = [synth.normal_bf16((rows, H, 512), seed, "q", dev, sub=l) for l in range(self.layers)]
        self.out = [torch.empty((rows, H, 512), dtype=torch.bfloat16, device=dev) for _ in range(self.layers)]
        self.qI = [synth.normal_e4m3((rows, H_I, d_I), seed, "qI", dev, sub=g) for g in range(G)]
        self.w = [synth.uniform_f32((rows, H_I), seed, "w", dev, sub=g) for g in range(G)]
        self.qI_pool = synth.normal_e4m3((rows, H_I, d_I), seed, "qI_pool", dev)
        self.w_pool = synth.uniform_f32((rows, H_I), seed, "w_pool", dev)
        self.kv_new = synth.normal_bf16((B, R, 512), seed, "kv_new", dev)
        self.kI_new = synth.indexer_keys_e4m3((B, R, d_I), seed + 1, dev, bias_prob=cfg.bias_prob)
        self.idx = [torch.empty((rows, k), dtype=torch.int32, device=dev) for _ in range(G)]
        self.pool = torch.full((rows, P), -1, dtype=torch.int32, device=dev)
        self.pos = torch.full((B,), n_pre, dtype=torch.int64, device=dev)
        n_row = torch.arange(rows, device=dev, dtype=torch.int64) % R + n_pre + 1
        self.n = n_row.contiguous()
        self.swa_len = torch.clamp(n_row, max=W).to(torch.int32).contiguous()
        self.ws = self.csa2.alloc_workspace(
            self.csa2.workspace_size(self.csa2.OP_LAYER_GROUP, rows, self.n_cap, k, P, H), dev)
        torch.cuda.synchronize()

    tokens_per_step = property(lambda self: self.rows)

    def scan_bytes(self, d_I):
        return self.B * self.n_cap * d_I                 # keys read once per sequence for its R rows

    def scan_score_bytes(self):
        return self.rows * self.n_cap * 4

    def alg_bytes(self):
        cfg, rows = self.cfg, self.rows
        out = super().alg_bytes()
        out["gather"] = self.layers * rows * cfg.k * FP4_ROW_BYTES
        out["swa"] = self.layers * rows * cfg.W * SWA_ROW_BYTES
        out["pool_slots"] = sum(rows * cfg.P * 8 * cfg.d_I for m, _, _ in cfg.groups if m == "reindex")
        return out

    def attn_launch_bytes(self, n_layers):
        return n_layers * self.rows * (self.cfg.k * FP4_ROW_BYTES + self.cfg.W * SWA_ROW_BYTES)

    def attn_launch_flops(self, n_layers):
        return 4.0 * n_layers * self.rows * self.cfg.H * (self.cfg.k + self.cfg.W) * 512

    step_layerwise = None

    def reset_positions(self):
        self.step_i = 0

    def step(self, events=None):
        csa2, cfg = self.csa2, self.cfg
        csa2.csa2_quantize_kv_fp4(self.kv_new, self.codes, self.scales, pos=self.pos)
        csa2.csa2_append_indexer_k(self.kI_new, self.kI, self.kbar, pos=self.pos)
        l0 = 0
        for g, (mode, n_reuse, form_pool) in enumerate(cfg.groups):
            L = 1 + n_reuse
            csa2.csa2_layer_group(
                csa2.MODE_FULL if mode == "full" else csa2.MODE_REINDEX, self.n, self.n_cap, self.codes, self.scales,
                self.kI, self.qI[g], self.w[g], self.idx[g], self.q[l0:l0 + L], self.swa[l0:l0 + L], self.swa_len,
                self.out[l0:l0 + L], self.ws, kbar=self.kbar, pool=self.pool,
                form_pool=self._rule(mode) if form_pool else csa2.POOL_NONE,
                qI_pool=self.qI_pool if mode == "reindex" else None,
                w_pool=self.w_pool if mode == "reindex" else None,
                events=None if events is None else events[g], rows_per_seq=self.R)
            l0 += L
        self.step_i += 1

    E2E_INPUTS = ("kv_new", "kI_new", "swa", "q", "qI", "w")


class EncoderDecodeWorkload(DecodeWorkload):
    """Decode through the encoder's layer groups at compression ratio r. Every
    group keeps its own caches (its Full layer's main KV and indexer K). Each
    step appends the token's SWA row to every layer and, when the token
    completes an entry (every r-th token), one compressed entry to every
    group's caches; the append kernel decides that on the device and writes
    the token's visible entry count and SWA length, which the groups then use.
    The entries themselves are inputs (merging r tokens needs weights)."""

    def __init__(self, cfg, device, seed=1234, batch=None, pool_rule="mean"):
        import torch
        import synth
        from fp4_kv_cache_06_b300 import csa2
        self.torch, self.csa2, self.cfg, self.pool_rule, self.dev = torch, csa2, cfg, pool_rule, device
        B = self.B = batch or cfg.B
        r, d_I, H_I, H, W, k, P = cfg.ratio, cfg.d_I, cfg.H_I, cfg.H, cfg.W, cfg.k, cfg.P
        self.n_cap = self.n_end = cfg.n                  # entries per group cache after the last step
        self.t_first = cfg.n * r - cfg.steps             # token of the first step; the last sees all n entries
        e_pre = self.t_first // r                        # entries complete before the first step
        G = len(cfg.groups)
        self.layers = sum(1 + g[1] for g in cfg.groups)
        dev, u8 = device, torch.uint8
        self.codes, self.scales, self.kI, self.kbar = [], [], [], []
        chunk = 1 << 17
        for g in range(G):
            codes = torch.empty((B, self.n_cap, 256), dtype=u8, device=dev)
            scales = torch.empty((B, self.n_cap, 32), dtype=u8, device=dev)
            kI = torch.empty((B, self.n_cap, d_I), dtype=u8, device=dev)
            kbar = torch.zeros((B, (self.n_cap + 7) // 8, d_I), dtype=u8, device=dev)
            for b in range(B):
                for c0 in range(0, e_pre, chunk):
                    rr = min(chunk, e_pre - c0)
                    x = synth.normal_bf16((1, rr, 512), seed, "kv", dev, sub=(g * 64 + b) * 4096 + c0 // chunk)
                    csa2.csa2_quantize_kv_fp4(x, codes[b:b + 1], scales[b:b + 1],
                                              pos=torch.tensor([c0], dtype=torch.int64, device=dev))
                kI[b, :e_pre] = synth.indexer_keys_e4m3((e_pre, d_I), seed, dev, sub=g * 64 + b)
            csa2.csa2_block_means(kI, torch.full((B,), e_pre, dtype=torch.int64, device=dev), kbar, n_max=e_pre)
            self.codes.append(codes); self.scales.append(scales); self.kI.append(kI); self.kbar.append(kbar)
        self.swa = [synth.normal_bf16((B, W, 512), seed, "swa", dev, sub=l) for l in range(self.layers)]
        self.q = [synth.normal_bf16((B, H, 512), seed, "q", dev, sub=l) for l in range(self.layers)]
        self.out = [torch.empty((B, H, 512), dtype=torch.bfloat16, device=dev) for _ in range(self.layers)]
        self.qI = [synth.normal_e4m3((B, H_I, d_I), seed, "qI", dev, sub=g) for g in range(G)]
        self.w = [synth.uniform_f32((B, H_I), seed, "w", dev, sub=g) for g in range(G)]
        self.kv_new = [synth.normal_bf16((B, 512), seed, "kv_new", dev, sub=g) for g in range(G)]
        self.kI_new = [synth.indexer_keys_e4m3((B, d_I), seed + 1, dev, sub=g) for g in range(G)]
        self.swa_new = [synth.normal_bf16((B, 512), seed, "swa_new", dev, sub=l) for l in range(self.layers)]
        self.idx = [torch.empty((B, k), dtype=torch.int32, device=dev) for _ in range(G)]
        self.pos = torch.full((B,), self.t_first, dtype=torch.int64, device=dev)
        self.n = torch.zeros((B,), dtype=torch.int64, device=dev)            # written by the append
        self.swa_len = torch.zeros((B,), dtype=torch.int32, device=dev)      # written by the append
        self.ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_LAYER_GROUP, B, self.n_cap, k, P, H), dev)
        self.step_i = 0
        torch.cuda.synchronize()

    def reset_positions(self):
        self.step_i = 0
        self.pos.fill_(self.t_first)

    step_layerwise = None

    def pool_recall(self):
        return None

    def step(self, events=None):
        csa2, cfg = self.csa2, self.cfg
        if self.step_i > 0:
            self.pos.add_(1)
        l0 = 0
        for g, (mode, n_reuse, _) in enumerate(cfg.groups):
            L = 1 + n_reuse
            csa2.csa2_append_step_ratio(self.kv_new[g], self.kI_new[g], self.swa_new[l0:l0 + L], self.swa[l0:l0 + L],
                                        self.pos, cfg.ratio, self.codes[g], self.scales[g], self.kI[g], self.kbar[g],
                                        n_vis_out=self.n if g == 0 else None,
                                        swa_len_out=self.swa_len if g == 0 else None)
            l0 += L
        l0 = 0
        for g, (mode, n_reuse, _) in enumerate(cfg.groups):
            L = 1 + n_reuse
            csa2.csa2_layer_group(csa2.MODE_FULL, self.n, self.n_cap, self.codes[g], self.scales[g], self.kI[g],
                                  self.qI[g], self.w[g], self.idx[g], self.q[l0:l0 + L], self.swa[l0:l0 + L],
                                  self.swa_len, self.out[l0:l0 + L], self.ws,
                                  events=None if events is None else events[g])
            l0 += L
        self.step_i += 1

    E2E_INPUTS = ("kv_new", "kI_new", "swa_new", "q", "qI", "w")


class PrefillWorkload:
    """One encoder prefill chunk: queries at tokens p0..p0+Q-1 over a cache of n
    compressed entries (ratio 2), one Full + Reuse group per entry of
    cfg.groups. With cfg.group_caches every group has its own caches (its Full
    layer's main KV and indexer K); otherwise they share one."""

    def __init__(self, cfg, device, seed=1234, queries=None):
        import torch
        import synth
        from fp4_kv_cache_06_b300 import csa2
        self.torch, self.csa2, self.cfg, self.dev = torch, csa2, cfg, device
        Q = self.Q = queries or cfg.prefill_queries
        n, H, W, k = cfg.n, cfg.H, cfg.W, cfg.k
        self.n_keys = n
        tokens = n * cfg.ratio                               # context incl. the chunk
        self.p0 = tokens - Q
        dev = device
        G = self.G = len(cfg.groups)
        n_caches = G if cfg.group_caches else 1
        self.codes, self.scales, self.kI = [], [], []
        chunk = 1 << 16
        for c in range(n_caches):
            codes = torch.empty((n, 256), dtype=torch.uint8, device=dev)
            scales = torch.empty((n, 32), dtype=torch.uint8, device=dev)
            for c0 in range(0, n, chunk):
                r = min(chunk, n - c0)
                x = synth.normal_bf16((1, r, 512), seed, "kv", dev, sub=c * 4096 + c0 // chunk)
                csa2.csa2_quantize_kv_fp4(x, codes[None], scales[None],
                                          pos=torch.tensor([c0], dtype=torch.int64, device=dev))
            self.codes.append(codes)
            self.scales.append(scales)
            self.kI.append(synth.indexer_keys_e4m3((n, cfg.d_I), seed, dev, sub=c))
        self.qI = [synth.normal_e4m3((Q, cfg.H_I, cfg.d_I), seed, "qI", dev, sub=g) for g in range(G)]
        self.w = [synth.uniform_f32((Q, cfg.H_I), seed, "w", dev, sub=g) for g in range(G)]
        self.group_layers = [1 + g[1] for g in cfg.groups]
        self.layers = sum(self.group_layers)
        self.q = [synth.normal_bf16((Q, H, 512), seed, "q", dev, sub=l) for l in range(self.layers)]
        self.swa = [synth.normal_bf16((Q + W - 1, 512), seed, "swa", dev, sub=l) for l in range(self.layers)]
        self.out = [torch.empty((Q, H, 512), dtype=torch.bfloat16, device=dev) for _ in range(self.layers)]
        pos = torch.arange(self.p0, self.p0 + Q, device=dev, dtype=torch.int64)
        self.n_vis = torch.clamp((pos + 1) // cfg.ratio, max=n).contiguous()
        self.swa_len = torch.clamp(pos + 1, max=W).to(torch.int32).contiguous()
        self.idx = torch.empty((Q, k), dtype=torch.int32, device=dev)
        self.ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_PREFILL_GROUP, Q, n, k, 0, H), dev)
        self.B = Q
        torch.cuda.synchronize()

    def step(self, events=None):
        l0 = 0
        for g in range(self.G):
            c, L = (g if self.cfg.group_caches else 0), self.group_layers[g]
            self.csa2.csa2_prefill_group(self.n_vis, self.codes[c], self.scales[c], self.kI[c], self.qI[g], self.w[g],
                                         self.idx, self.q[l0:l0 + L], self.swa[l0:l0 + L], self.swa_len,
                                         self.out[l0:l0 + L], self.ws, events=None if events is None else events[g])
            l0 += L

    E2E_INPUTS = ("q", "swa", "qI", "w")

    def host_buffers(self):
        """Pinned host copies of the chunk's inputs (every layer's queries and
        window rows, the indexer queries and head weights) and of the outputs."""
        items = lambda v: v if isinstance(v, list) else [v]
        ins = {k: getattr(self, k) for k in self.E2E_INPUTS}
        size = lambda t: t.numel() * t.element_size()
        h2d = sum(size(t) for v in ins.values() for t in items(v))
        d2h = sum(size(t) for t in self.out)
        arena = PinnedArena(self.torch, h2d + d2h + 512 * (sum(len(items(v)) for v in ins.values()) + len(self.out)))
        self.h_in = {k: ([arena.take(t) for t in v] if isinstance(v, list) else arena.take(v)) for k, v in ins.items()}
        self.h_out = [arena.empty_like(t) for t in self.out]
        return h2d, d2h

    def gemm_flops(self):
        return 2.0 * self.Q * self.cfg.H_I * self.n_keys * self.cfg.d_I

    def attn_flops_per_layer(self):
        return 4.0 * self.Q * self.cfg.H * (self.cfg.k + self.cfg.W) * 512


def run_prefill(args, world, rank, local):
    import torch
    import synth
    from fp4_kv_cache_06_b300 import csa2
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = synth.get_config(args.config)
    wl = PrefillWorkload(cfg, dev, seed=1234 + 7919 * rank, queries=args.batch)
    clk = ClockSampler(local).start()
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()

    def mk():
        e = torch.cuda.Event(enable_timing=True, external=True)
        e.record()
        return e
    evs = [[[mk() for _ in range(3 + L)] for L in wl.group_layers] for _ in range(args.steps)]
    step_ev = [(mk(), mk()) for _ in range(args.steps)]
    torch.cuda.synchronize()
    # the timed graph has only the step events (an event between two launches
    # would cancel their programmatic overlap); the phase graph, replayed after
    # it, has the per-group events
    launches0 = csa2.launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(args.steps):
            step_ev[i][0].record()
            wl.step()
            step_ev[i][1].record()
    launches = csa2.launch_count() - launches0
    pgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pgraph):
        for i in range(args.steps):
            wl.step(events=evs[i])
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    tw0 = time.time()
    graph.replay()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clk.mark(tw0, time.time())
    clk.stop()
    barrier(world)
    ms = statistics.mean(a.elapsed_time(b) for a, b in step_ev)
    ms_max = max_over_ranks(ms, world, dev)
    pgraph.replay()
    torch.cuda.synchronize()
    gemm_ms = statistics.mean(e[0].elapsed_time(e[1]) for es in evs for e in es)
    topk_ms = statistics.mean(e[1].elapsed_time(e[2]) for es in evs for e in es)
    attn_ms = statistics.mean(e[2 + j].elapsed_time(e[3 + j]) for es in evs for g, e in enumerate(es)
                              for j in range(wl.group_layers[g]))
    e2e = None
    if not args.no_e2e:
        # the chunk's inputs in from pinned host memory and its outputs back,
        # neighbouring chunks' copies overlapping the compute (PipelinedE2E)
        h2d, d2h = wl.host_buffers()
        pipe = PipelinedE2E(wl, wl.E2E_INPUTS)
        pipe.begin()
        for i in range(2):
            pipe.step(last=i == 1)
        pipe.end()
        torch.cuda.synchronize()
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph):
            pipe.begin()
            for i in range(args.steps):
                pipe.step(last=i == args.steps - 1)
            pipe.end()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record()
        e2e_graph.replay()
        e1.record()
        pipe.restore()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
        e2e = {"value": world * wl.Q / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
               "schedule": "chunk i+1's inputs in and chunk i's outputs out on two copy streams during chunk i; "
                           "K chunks as one CUDA graph"}
    bf16, bf16_kind = bf16_peak()
    kind = f"{bf16_kind} bf16 x 2 (nominal fp8/bf16 ratio)"
    fp8_peak = 2 * bf16
    ach = wl.gemm_flops() / (gemm_ms / 1e3) / 1e12
    res = {
        "metric": ("CSA2 prefill query tokens/s per encoder group (ratio 2); % of B300 FP8 tensor roofline"
                   if wl.G == 1 else
                   f"CSA2 prefill query tokens/s through the {wl.G}-group encoder stack (ratio 2); "
                   "% of B300 FP8 tensor roofline"),
        "value": world * wl.Q / (ms_max / 1e3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3+bf16", "data": "synthetic",
        "config": {"workload": cfg.workload, "config_index": args.config, "queries": wl.Q, "entries": wl.n_keys,
                   "first_query_token": wl.p0, "heads": cfg.H, "indexer": f"{cfg.H_I}x{cfg.d_I}",
                   "topk": cfg.k, "swa": cfg.W, "layers": wl.layers, "groups": [list(g) for g in cfg.groups],
                   "separate_group_caches": cfg.group_caches, "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2: every layer's queries, Q x 64 x 512 bf16 (268 MB at 4096 queries)"},
        "roofline": {"bound": "tensor", "kernel": "k_prefill_index (tcgen05 FP8 indexer GEMM)",
                     "achieved": round(ach, 1), "peak": fp8_peak, "peak_kind": kind, "unit": "TFLOP/s",
                     "frac": round(ach / fp8_peak, 4), "traffic": None, "gemm_ms": round(gemm_ms, 4),
                     "algorithmic_flops_per_launch": wl.gemm_flops()},
        "e2e": e2e, "gpu_launches": int(launches), "clocks": clk.summary(),
        "phases_ms": {"indexer_gemm_ms": gemm_ms, "topk_ms": topk_ms, "attn_ms_per_layer": attn_ms,
                      "attn_tflops": wl.attn_flops_per_layer() / (attn_ms / 1e3) / 1e12},
        "wall_s": wall,
    }
    return res


class L2Flush:
    """Evicts L2 between timed steps, outside the step's events: writes a
    256 MiB buffer (larger than the 126 MB L2), then reads another 256 MiB
    one so that the dirty lines of the write are written back during the
    flush rather than during the next step."""

    def __init__(self, dev):
        import torch
        self.a = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.b = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.a.zero_()
        torch.sum(self.b, dim=0, out=self.sink)


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def scan_traffic(d_I, positions_per_launch):
    """DRAM bytes per Full-scan launch from the committed ncu summary, if the
    scan kernel's source is unchanged since it was captured; else None."""
    path = os.path.join(ROOT, "profiles", "index_scan_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        src = os.path.join(ROOT, "fp4_kv_cache_06_b300", "csrc", "index_scan.cu")
        if rec.get("source_sha256_16") != source_hash(src):
            return None
        return rec["dram_bytes_per_position"] * positions_per_launch
    except Exception:
        return None


def decode_config(cfg, config_index, batch, world, pool_rule="mean"):
    """The `config` object of a decode bench line (both arms print the same one)."""
    extra = {"pool_rule": "block max of the Full scores"} if pool_rule == "max" else {}
    if cfg.tokens > 1:
        extra["tokens_per_sequence"] = cfg.tokens
    return {**extra, "workload": cfg.workload, "config_index": config_index, "batch": batch,
            "context": cfg.n, "heads": cfg.H, "indexer": f"{cfg.H_I}x{cfg.d_I}", "topk": cfg.k,
            "swa": cfg.W, "groups": [list(g) for g in cfg.groups], "parallelism": f"replicas{world}",
            "l2": "flushed before every step outside the per-step events (256 MiB write, then a 256 MiB read "
                  "so the write-backs land in the flush)"}


def run_csa2(args, world, rank, local):
    import torch
    import synth
    from fp4_kv_cache_06_b300 import csa2

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = synth.get_config(args.config)
    if cfg.prefill_queries:
        raise SystemExit("the prefill configuration is not a decode bench workload")
    wl_cls = (MultiTokenWorkload if cfg.tokens > 1 else EncoderDecodeWorkload if cfg.group_caches
              else DecodeWorkload)
    wl = wl_cls(cfg, dev, seed=1234 + 7919 * rank, batch=args.batch, pool_rule=args.pool_rule)
    G = len(cfg.groups)
    flush = L2Flush(dev)
    total_steps = args.warmup + args.steps
    if cfg.steps > 1 and total_steps > cfg.steps:
        pass  # positions wrap below so the cache never exceeds its capacity

    def maybe_wrap():
        if cfg.steps > 1 and wl.step_i >= cfg.steps:
            wl.reset_positions()

    clk = ClockSampler(local).start()
    for _ in range(args.warmup):
        maybe_wrap()
        wl.step()
    torch.cuda.synchronize()
    if cfg.steps > 1:
        wl.reset_positions()

    # The timed region is ONE CUDA graph holding all K steps (host launch
    # overhead removed): per step an L2 flush, then [start event, step with
    # its phase events, end event]. Events are external graph nodes.
    # per-group events: [0] scan start, [1] scan end, [2] after Top-K/pool, then one per layer
    def mk():
        e = torch.cuda.Event(enable_timing=True, external=True)
        e.record()
        return e
    step_ev = [(mk(), mk()) for _ in range(args.steps)]
    grp_ev = [[[mk() for _ in range(3 + 1 + cfg.groups[g][1])] for g in range(G)] for _ in range(args.steps)]
    torch.cuda.synchronize()

    def capture(phases, step_fn=None, sev=None):
        """K steps as one graph: the timed one has only the step events (an
        event between two launches would cancel their programmatic overlap);
        the phase one (replayed separately) has the per-group events."""
        step_fn = step_fn or wl.step
        sev = sev or step_ev
        if cfg.steps > 1:
            wl.reset_positions()
            wl.step_i = 1                               # captured steps advance the positions
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(args.steps):
                flush()                                # evict L2 between steps (outside the step events)
                if not phases:
                    sev[i][0].record()
                step_fn(events=grp_ev[i] if phases else None)
                if not phases:
                    sev[i][1].record()
        return g

    def rewind():
        if cfg.steps > 1:
            wl.reset_positions()
            wl.pos.sub_(1)                             # the first captured step adds 1
            wl.n.sub_(1)

    launches0 = csa2.launch_count()
    graph = capture(False)
    launches = csa2.launch_count() - launches0        # kernels launched per replay of the timed graph
    rewind()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    tw0 = time.time()
    graph.replay()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clk.mark(tw0, time.time())
    clk.stop()
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, world, dev)
    # the phase breakdown (and the scan's duration for the roofline) from a
    # second replay with the per-group events
    pgraph = capture(True)
    rewind()
    torch.cuda.synchronize()
    pgraph.replay()
    torch.cuda.synchronize()
    # events 0 -> 1 of a group bracket its largest indexer kernel: the Full
    # scan, or the block-mean scan of a Reindex group that forms the pool
    def group_phase():
        out = {}
        for g, (mode, nr, fp) in enumerate(cfg.groups):
            ev = [[grp_ev[i][g][j] for j in range(3 + 1 + nr)] for i in range(args.steps)]
            launch = statistics.mean(e[2].elapsed_time(e[3 + nr]) for e in ev)
            out[f"group{g}_{mode}"] = {
                "indexer_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in ev),
                "topk_pool_ms": statistics.mean(e[1].elapsed_time(e[2]) for e in ev),
                "attn_launch_ms": launch,
                "attn_ms_per_layer": launch / (1 + nr),
            }
        return out
    phase = group_phase()

    # the layer-at-a-time schedule: one attention launch per layer, each after
    # the previous (a model whose next query depends on this layer's output)
    layerwise = None
    if getattr(wl, "step_layerwise", None) is not None:
        lw_step_ev = [(mk(), mk()) for _ in range(args.steps)]
        torch.cuda.synchronize()
        lgraph = capture(False, wl.step_layerwise, lw_step_ev)
        rewind()
        torch.cuda.synchronize()
        lgraph.replay()
        torch.cuda.synchronize()
        lw_ms = statistics.mean(a.elapsed_time(b) for a, b in lw_step_ev)
        lpgraph = capture(True, wl.step_layerwise)
        rewind()
        torch.cuda.synchronize()
        lpgraph.replay()
        torch.cuda.synchronize()
        per_layer = [statistics.mean(grp_ev[i][g][2 + j].elapsed_time(grp_ev[i][g][3 + j]) for i in range(args.steps))
                     for g, (_, nr, _) in enumerate(cfg.groups) for j in range(1 + nr)]
        layerwise = {"ms_per_step": lw_ms, "tokens_per_s": wl.tokens_per_step / (lw_ms / 1e3),
                     "attn_ms_per_layer": statistics.mean(per_layer),
                     "attn_ms_first_layer_of_group": statistics.mean(
                         per_layer[sum(1 + g[1] for g in cfg.groups[:k]) ] for k in range(G)),
                     "schedule": "each layer's attention is its own launch, after the previous layer's; the "
                                 "first layer's runs inside the group call"}

    hbm, hbm_kind = peaks()
    bf16, bf16_kind = bf16_peak()
    full = [g for g, (m, _, _) in enumerate(cfg.groups) if m == "full"]
    pool_re = [g for g, (m, _, fp) in enumerate(cfg.groups) if m == "reindex" and fp]
    ms_ev = lambda g: statistics.mean(grp_ev[i][g][0].elapsed_time(grp_ev[i][g][1]) for i in range(args.steps))
    roof = None
    if full:
        scan_avg = statistics.mean(ms_ev(g) for g in full)
        alg = wl.scan_bytes(cfg.d_I)
        per_launch_pos = wl.B * min(wl.n_end, wl.n_cap)
        ach = alg / (scan_avg / 1e3) / 1e9
        incl = (alg + wl.scan_score_bytes()) / (scan_avg / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": "k_index_scan_tma (Full indexer scan)", "achieved": round(ach, 1),
                "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s", "frac": round(ach / hbm, 4),
                "traffic": scan_traffic(cfg.d_I, per_launch_pos) if cfg.tokens == 1 else None,
                "algorithmic_bytes_per_launch": alg,
                "bytes_basis": "indexer keys read once per sequence (the fp32 score writes are not counted)",
                "frac_incl_score_writes": round(incl / hbm, 4), "scan_ms": round(scan_avg, 4)}
    elif pool_re:
        scan_avg = statistics.mean(ms_ev(g) for g in pool_re)
        alg = wl.pool_scan_bytes(cfg.d_I)
        ach = alg / (scan_avg / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": "k_index_scan_tma (block-mean scan of the pool formation)",
                "achieved": round(ach, 1), "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "traffic": None, "algorithmic_bytes_per_launch": alg,
                "bytes_basis": "block-mean keys read once", "scan_ms": round(scan_avg, 4)}

    # per-phase rooflines: the scan (above), each group's attention launch
    # (gathered FP4 rows and SWA rows per layer, and the tensor work), the step
    alg_step = wl.alg_bytes()
    alg_total = sum(alg_step.values())
    attn = []
    for g, (mode, nr, _) in enumerate(cfg.groups):
        t = phase[f"group{g}_{mode}"]["attn_launch_ms"] / 1e3
        by, fl = wl.attn_launch_bytes(1 + nr), wl.attn_launch_flops(1 + nr)
        attn.append({"group": g, "layers": 1 + nr, "launch_ms": round(t * 1e3, 5),
                     "hbm_gbs": round(by / t / 1e9, 1), "frac_hbm": round(by / t / 1e9 / hbm, 4),
                     "tflops": round(fl / t / 1e12, 1), "frac_tensor": round(fl / t / 1e12 / bf16, 4)})
    attn_s = sum(phase[f"group{g}_{m}"]["attn_launch_ms"] for g, (m, _, _) in enumerate(cfg.groups)) / 1e3
    gather = {"bytes_per_step": alg_step["gather"],
              "achieved_gbs": round(alg_step["gather"] / attn_s / 1e9, 1),
              "frac_hbm": round(alg_step["gather"] / attn_s / 1e9 / hbm, 4),
              "basis": "the FP4 rows (288 B each) that the step's attention launches gather, over the time "
                       "of those launches; the launches also read SWA rows and queries and run the MMAs"}
    phases_roofline = {
        "scan": roof,
        "attention_launches": attn,
        "attention_peaks": {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_kind": bf16_kind},
        "step": {"algorithmic_bytes": alg_total, "by_kind": alg_step,
                 "achieved_gbs": round(alg_total / (ms_max / 1e3) / 1e9, 1),
                 "frac_hbm": round(alg_total / (ms_max / 1e3) / 1e9 / hbm, 4)},
    }

    # end-to-end: per-step inputs from pinned host memory, outputs back to host,
    # the copies of neighbouring steps overlapping the compute (PipelinedE2E).
    # Like the timed region, the K steps are one CUDA graph: every step's input
    # copy, launches and read-back are nodes of it, replayed once.
    e2e = None
    if not args.no_e2e:
        h2d, d2h = wl.host_buffers()
        pipe = PipelinedE2E(wl, wl.E2E_INPUTS)
        if cfg.steps > 1:
            wl.reset_positions()
        pipe.begin()
        for i in range(2):
            maybe_wrap()
            pipe.step(last=i == 1)
        pipe.end()
        torch.cuda.synchronize()
        if cfg.steps > 1:
            wl.reset_positions()
            wl.step_i = 1                               # captured steps advance the positions
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph):
            pipe.begin()
            for i in range(args.steps):
                pipe.step(last=i == args.steps - 1)
            pipe.end()
        if cfg.steps > 1:
            wl.reset_positions()
            wl.pos.sub_(1)                             # the first captured step adds 1
            wl.n.sub_(1)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record()
        e2e_graph.replay()
        e1.record()
        pipe.restore()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
        e2e = {"value": world * wl.tokens_per_step / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
               "schedule": "step i+1's inputs in and step i's outputs out on two copy streams during step i; "
                           "K steps as one CUDA graph"}

    res = {
        "metric": METRIC, "value": world * wl.tokens_per_step / (ms_max / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+bf16", "data": "synthetic",
        "config": decode_config(cfg, args.config, wl.B, world, args.pool_rule),
        "roofline": roof, "e2e": e2e, "gpu_launches": int(launches), "clocks": clk.summary(),
        "phases_ms": phase, "phases_roofline": phases_roofline, "fp4_gather": gather,
        "wall_s": wall, "step_ms_min": min(step_ms), "step_ms_max": max(step_ms),
    }
    if layerwise is not None:
        res["layer_at_a_time"] = layerwise
    recall = wl.pool_recall()
    if recall is not None:
        res["pool_recall"] = recall
    return res


# ---------------------------------------------------------------------------
# the oracle, timed on the host cores
# ---------------------------------------------------------------------------
class OracleSample:
    """One decode step of ONE sequence of the config, run by the oracle.

    Inputs are generated once (untimed). step() is the timed part: the new
    entry's FP4 append, then every layer group of the config in order:
    - the indexer over every position (Full) or block means + pool + Reindex;
    - Top-512;
    - each of the group's layers' attention.
    Groups share one cache, or each Full group has its own when the config
    says so. The FP4 rows a step reads are quantised by the oracle inside the
    step from their bf16 source rows (the oracle keeps no FP4 cache of its
    own)."""

    def __init__(self, cfg, seed=99):
        import numpy as np
        import torch
        import synth
        self.cfg = cfg
        n, d_I, H_I, H = cfg.n, cfg.d_I, cfg.H_I, cfg.H
        G = len(cfg.groups)
        n_caches = G if cfg.group_caches else 1
        bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
        self.kI, self.kv = [], []
        chunk = 1 << 16
        for c in range(n_caches):
            self.kI.append(synth.indexer_keys_e4m3((n, d_I), seed, bias_prob=cfg.bias_prob, sub=c).numpy())
            kv = np.empty((n, 512), dtype=np.uint16)
            for c0 in range(0, n, chunk):
                r = min(chunk, n - c0)
                kv[c0:c0 + r] = bits(synth.normal_bf16((r, 512), seed, "kv", sub=c * 4096 + c0 // chunk))
            self.kv.append(kv)
        self.layers = sum(1 + g[1] for g in cfg.groups)
        self.q = [bits(synth.normal_bf16((H, 512), seed, "q", sub=l)) for l in range(self.layers)]
        self.swa = [bits(synth.normal_bf16((cfg.W, 512), seed, "swa", sub=l)) for l in range(self.layers)]
        self.qI = [synth.normal_e4m3((H_I, d_I), seed, "qI", sub=g).numpy() for g in range(G)]
        self.w = [synth.uniform_f32((H_I,), seed, "w", sub=g).numpy() for g in range(G)]
        self.qI_pool = synth.normal_e4m3((H_I, d_I), seed, "qI_pool").numpy()
        self.w_pool = synth.uniform_f32((H_I,), seed, "w_pool").numpy()
        self.codes = [np.zeros((n, 256), dtype=np.uint8) for _ in range(n_caches)]
        self.scales = [np.zeros((n, 32), dtype=np.uint8) for _ in range(n_caches)]
        parts = []
        for mode, n_reuse, form_pool in cfg.groups:
            first = f"Full scan of all {n} positions" if mode == "full" else "Reindex over the pool"
            parts.append(first + (" + pool" if form_pool else "") + f", Top-{cfg.k}, {1 + n_reuse} attention layers")
        self.desc = (f"one sequence (batch 1) of the {cfg.workload} step: FP4 append, then "
                     + "; ".join(parts)
                     + ("; separate caches per group" if cfg.group_caches else "")
                     + "; gathered rows quantised inside the step"
                     + (f"; one of the {cfg.tokens} new tokens of a multi-token step (each costs the same)"
                        if cfg.tokens > 1 else ""))

    def step(self):
        import oracle
        cfg, n = self.cfg, self.cfg.n
        t0 = time.perf_counter()
        for kv in self.kv:
            oracle.quantize_fp4(kv[n - 1:n])
        pool, l0 = None, 0
        for g, (mode, n_reuse, form_pool) in enumerate(cfg.groups):
            c = g if cfg.group_caches else 0
            kI = self.kI[c]
            if mode == "full":
                idx, _ = oracle.full_topk(self.qI[g], self.w[g], kI, n, cfg.k)
                if form_pool:
                    pool, _ = oracle.form_pool(self.qI[g], self.w[g], oracle.block_means(kI, n), cfg.P)
            else:
                if form_pool or pool is None:
                    pool, _ = oracle.form_pool(self.qI_pool, self.w_pool, oracle.block_means(kI, n), cfg.P)
                idx, _, _ = oracle.reindex_topk(self.qI[g], self.w[g], kI, pool, n, cfg.k)
            rows = idx[idx >= 0]
            self.codes[c][rows], self.scales[c][rows] = oracle.quantize_fp4(self.kv[c][rows])
            for l in range(l0, l0 + 1 + n_reuse):
                oracle.sparse_attention(self.q[l], self.codes[c], self.scales[c], idx, self.swa[l], cfg.W)
            l0 += 1 + n_reuse
        return time.perf_counter() - t0


class OraclePrefillSample:
    """The oracle on sampled queries of one prefill chunk: for each query its
    Full-layer Top-k over the entries it sees, then every layer of its
    group(s). Spread over the chunk and including its last (causal tail)
    queries; the chunk's time is extrapolated as queries x mean per query."""

    def __init__(self, cfg, n_sample=32, seed=99):
        import numpy as np
        import torch
        import synth
        self.cfg = cfg
        n, Q = cfg.n, cfg.prefill_queries
        self.p0 = n * cfg.ratio - Q
        G = len(cfg.groups)
        n_caches = G if cfg.group_caches else 1
        bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
        chunk = 1 << 16
        self.kI, self.kv = [], []
        for c in range(n_caches):
            self.kI.append(synth.indexer_keys_e4m3((n, cfg.d_I), seed, sub=c).numpy())
            kv = np.empty((n, 512), dtype=np.uint16)
            for c0 in range(0, n, chunk):
                r = min(chunk, n - c0)
                kv[c0:c0 + r] = bits(synth.normal_bf16((r, 512), seed, "kv", sub=c * 4096 + c0 // chunk))
            self.kv.append(kv)
        self.layers = sum(1 + g[1] for g in cfg.groups)
        self.q = [bits(synth.normal_bf16((cfg.H, 512), seed, "q", sub=l)) for l in range(self.layers)]
        self.swa = [bits(synth.normal_bf16((cfg.W, 512), seed, "swa", sub=l)) for l in range(self.layers)]
        self.qI = [synth.normal_e4m3((cfg.H_I, cfg.d_I), seed, "qI", sub=g).numpy() for g in range(G)]
        self.w = [synth.uniform_f32((cfg.H_I,), seed, "w", sub=g).numpy() for g in range(G)]
        tail = 8
        spread = np.linspace(0, Q - tail - 1, n_sample - tail).astype(np.int64)
        self.queries = sorted(set(spread.tolist()) | set(range(Q - tail, Q)))
        self.desc = (f"{len(self.queries)} sampled queries of the {cfg.workload} chunk (spread over it, with its last "
                     f"{tail}): per query the Full Top-{cfg.k} over the entries it sees and its {self.layers} layers' "
                     f"attention; chunk time extrapolated as {Q} x the mean per query")

    def run(self):
        import numpy as np
        import oracle
        cfg = self.cfg
        times = []
        for qi in self.queries:
            p = self.p0 + qi
            n_vis = int(oracle.prefill_visible(p, cfg.ratio))
            t0 = time.perf_counter()
            l0 = 0
            for g, (mode, n_reuse, _) in enumerate(cfg.groups):
                c = g if cfg.group_caches else 0
                idx, _ = oracle.full_topk(self.qI[g], self.w[g], self.kI[c], n_vis, cfg.k)
                rows = idx[idx >= 0]
                # the gathered rows, quantised by the oracle; the attention
                # reads them through indices into this compact block
                cq, sq = oracle.quantize_fp4(self.kv[c][rows])
                local = np.full(cfg.k, -1, dtype=np.int64)
                local[:rows.size] = np.arange(rows.size)
                swa_len = min(p + 1, cfg.W)
                for l in range(l0, l0 + 1 + n_reuse):
                    oracle.sparse_attention(self.q[l], cq, sq, local, self.swa[l], swa_len)
                l0 += 1 + n_reuse
            times.append(time.perf_counter() - t0)
        return statistics.mean(times)


def oracle_baseline(cfg, min_s=10.0, max_steps=30):
    """Time the oracle's sample step repeatedly for about min_s seconds."""
    smp = OracleSample(cfg)
    times = []
    while sum(times) < min_s and len(times) < max_steps:
        times.append(smp.step())
    t = statistics.mean(times)
    return t, smp.desc + f"; mean of {len(times)} steps"


def oracle_cores():
    try:
        from threadpoolctl import threadpool_info
        return max([int(i.get("num_threads", 1)) for i in threadpool_info()] + [1])
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, world, rank):
    import synth
    cfg = synth.get_config(args.config)
    smp = OracleSample(cfg)
    for _ in range(args.warmup):
        smp.step()
    times = [smp.step() for _ in range(args.steps)]
    desc = smp.desc + f"; mean of {len(times)} steps"
    t = statistics.mean(times)
    value = 1.0 / t
    cores = oracle_cores()
    return {
        "metric": METRIC, "impl": "reference", "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(cfg, args.config, args.batch or cfg.B, world, args.pool_rule),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--batch", type=int, default=None, help="override the batch (profiling runs)")
    ap.add_argument("--impl", default="csa2", choices=["csa2", "reference"])
    ap.add_argument("--pool-rule", default="mean", choices=["mean", "max"],
                    help="how a Full group that forms the pool scores blocks: mean key (default) or block max")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "csa2":
        args.warmup = 3
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(run_reference(args, world, 0)), flush=True)
        return
    world, rank, local = dist_setup(args.gpus)
    import synth
    if synth.get_config(args.config).prefill_queries:
        res = run_prefill(args, world, rank, local)
    else:
        res = run_csa2(args, world, rank, local)
    if rank == 0 and not args.no_cpu_baseline:
        cfg = synth.get_config(args.config)
        if cfg.prefill_queries:
            smp = OraclePrefillSample(cfg)
            per_q = smp.run()
            res["cpu_baseline"] = {"value": 1.0 / per_q, "unit": "tokens/s", "cores": oracle_cores(),
                                   "kind": "oracle", "sample": smp.desc, "extrapolated": True,
                                   "chunk_s_extrapolated": per_q * cfg.prefill_queries}
        else:
            dt, desc = oracle_baseline(cfg)
            res["cpu_baseline"] = {"value": 1.0 / dt, "unit": UNIT, "cores": oracle_cores(), "kind": "oracle",
                                   "sample": desc}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
