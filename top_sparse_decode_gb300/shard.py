"""One decode step of a sequence split by tokens across the ranks of a process group
(HashAttention: Semantic Sparsity for Faster Inference, 2.5: a context held by
several devices needs one exchange of top-k candidates and one of attention
partials).

Rank s holds tokens [a_s, a_s + n_s) of the sequence -- its own K, V and bit-plane
index, cut at whole 64-token scale blocks so that its scores are the unsharded
ones.  A step is SPMD over the ranks:

    phase 1  the shard's plan, scan and top-k (sd_plan_score, sd_topk_wmax) with the
             sequence's budget k and the forced windows the shard holds, then its
             competing candidates (sd_shard_candidates);
             -> all-gather of (score, global index, count)
    phase 2  the sequence's top-k (sd_topk_merge, the same on every rank), the
             shard's attention set (sd_shard_select) and its attention over it
             (sd_gather_attend);
             -> all-gather of (out, lse)
    phase 3  the split-softmax combine (sd_attend_combine).

This module orders the calls and owns the buffers; every value is computed by
libsd's kernels.  The exchanges are torch.distributed all-gathers (any backend);
run_sharded_step drives one rank, and the phases can also be driven for every
shard from one process (the single-GPU tests do that).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import torch

from . import (SD_IDX_PLANES, sd_attend_combine, sd_gather_attend, sd_gather_attend_workspace_size,
               sd_shard_candidates, sd_shard_select, sd_topk_merge)
from .pipeline import DecodeStep, StepConfig


def shard_bounds(n: int, shards: int) -> list:
    """Token boundaries 0 = a_0 < a_1 < ... < a_S = n of S contiguous shards, cut at
    multiples of 64 tokens: a_s = 64 * floor(ceil(n / 64) * s / S)."""
    blocks = (n + 63) // 64
    return [min(n, 64 * ((blocks * s) // shards)) for s in range(shards + 1)]


def shard_windows(n: int, a: int, b: int, sink: int, local: int) -> tuple:
    """(sink_s, local_s): the parts of the sequence's forced windows [0, lead) and
    [tail, n) that shard [a, b) holds, in its own indices (lead = min(sink, n),
    tail = max(n - local, lead), the unsharded top-k's windows)."""
    lead = min(sink, n)
    tail = max(n - local, lead)
    ns = b - a
    return min(max(lead - a, 0), ns), min(max(b - max(a, tail), 0), ns)


class ShardStep:
    """Rank `shard`'s buffers and calls for one step of the sequence described by
    cfg (its n, k, sink, local, plan mode and budget are the whole sequence's).
    K_s, V_s: bf16 [B][Hkv][n_cap_s][d] with the shard's n_s tokens first; index_s:
    its bit-plane index ({"planes", "scales"}, built from K_s)."""

    def __init__(self, cfg: StepConfig, shard: int, shards: int, K_s: torch.Tensor,
                 V_s: torch.Tensor, index_s: dict, sigma2: torch.Tensor,
                 n_cap_s: int = 0, scale: Optional[float] = None):
        if cfg.kind != SD_IDX_PLANES:
            raise ValueError("sequence shards are built on the bit-plane step")
        self.cfg, self.shard, self.shards = cfg, shard, shards
        cut = shard_bounds(cfg.n, shards)
        self.a, b = cut[shard], cut[shard + 1]
        self.n_s = b - self.a
        self.sink_s, self.local_s = shard_windows(cfg.n, self.a, b, cfg.sink, cfg.local)
        self.local = StepConfig(SD_IDX_PLANES, cfg.B, cfg.Hq, cfg.Hkv, self.n_s, cfg.d, k=cfg.k,
                                sink=self.sink_s, local=self.local_s, plan_mode=cfg.plan_mode,
                                budget=cfg.budget, n_cap=n_cap_s)
        self.step = DecodeStep(self.local, K_s, V_s, index_s, sigma2=sigma2, scale=scale)
        self.scale = self.step.scale
        dev = K_s.device
        rows, k = cfg.B * cfg.Hkv, cfg.k
        self.rows = rows
        self.cand_score = torch.empty((rows, k), dtype=torch.float32, device=dev)
        self.cand_idx = torch.empty((rows, k), dtype=torch.int32, device=dev)
        self.cand_count = torch.empty((rows,), dtype=torch.int32, device=dev)
        self.sel_idx = torch.empty((rows, k), dtype=torch.int32, device=dev)
        self.sel_count = torch.empty((rows,), dtype=torch.int32, device=dev)
        self.set_stride = self.sink_s + self.local_s + k
        self.my_idx = torch.empty((rows, self.set_stride), dtype=torch.int32, device=dev)
        self.my_count = torch.empty((rows,), dtype=torch.int32, device=dev)
        ws = sd_gather_attend_workspace_size(self.step.shape, self.set_stride)
        self.att_ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.part_out = torch.empty((cfg.B, cfg.Hq, cfg.d), dtype=torch.float32, device=dev)
        self.part_lse = torch.empty((cfg.B, cfg.Hq), dtype=torch.float32, device=dev)
        self.out = torch.empty((cfg.B, cfg.Hq, cfg.d), dtype=torch.float32, device=dev)
        self.lse = torch.empty((cfg.B, cfg.Hq), dtype=torch.float32, device=dev)

    def phase1(self, q, stream=None):
        """The shard's plan, scan and top-k; returns its candidates (score, global
        index, count) for the first exchange."""
        st = self.step
        st.stage_plan_score(q, stream)
        st.stage_topk(stream)
        sd_shard_candidates(st.scores, self.rows, self.n_s, st.idx, self.local.max_count,
                            st.count, self.sink_s, self.local_s, self.a, self.cfg.k,
                            self.cand_score, self.cand_idx, self.cand_count, stream)
        return self.cand_score, self.cand_idx, self.cand_count

    def phase2(self, q, all_score, all_idx, all_count, stream=None):
        """all_*: every shard's candidates stacked [S][rows][k] / [S][rows]; returns
        the shard's attention (out, lse) over its part of the merged set and its
        forced windows, for the second exchange."""
        S, k = all_score.shape[0], self.cfg.k
        sd_topk_merge(self.rows, S, k, all_score, all_idx, all_count, self.sel_idx, k,
                      self.sel_count, stream)
        sd_shard_select(self.rows, self.sel_idx, k, self.sel_count, self.a, self.n_s,
                        self.sink_s, self.local_s, k, self.my_idx, self.set_stride,
                        self.my_count, stream)
        sd_gather_attend(self.step.shape, q, self.step.K, self.step.V, self.my_idx,
                         self.set_stride, self.my_count, self.set_stride, self.scale,
                         self.part_out, self.part_lse, self.att_ws, stream)
        return self.part_out, self.part_lse

    def phase3(self, all_out, all_lse, stream=None):
        """all_out [S][B][Hq][d], all_lse [S][B][Hq]: the sequence's attention."""
        cfg = self.cfg
        sd_attend_combine(all_out.shape[0], cfg.B, cfg.Hq, all_out, all_lse, self.out, self.lse,
                          stream)
        return self.out, self.lse


def all_gather_stacked(t: torch.Tensor, group=None) -> torch.Tensor:
    """[world, *t.shape]: every rank's t, in rank order."""
    import torch.distributed as dist
    parts = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


def run_sharded_step(step, q, group=None, gather=all_gather_stacked):
    """One step on this rank: phase 1, the candidate exchange, phase 2, the partial
    exchange, phase 3.  `step` is a ShardStep (or any object with the same phases)."""
    c = step.phase1(q)
    g1 = [gather(x, group) for x in c]
    p = step.phase2(q, *g1)
    g2 = [gather(x, group) for x in p]
    return step.phase3(*g2)


def run_shards_locally(steps: Sequence, q):
    """Every shard's phases from one process (no process group): the exchanges are
    stacks of the shards' tensors in shard order."""
    c = [s.phase1(q) for s in steps]
    g1 = [torch.stack([x[i] for x in c]) for i in range(3)]
    p = [s.phase2(q, *g1) for s in steps]
    g2 = [torch.stack([x[i] for x in p]) for i in range(2)]
    return [s.phase3(*g2) for s in steps]
