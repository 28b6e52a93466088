"""One decode step of the sparse-decode hot path, composed from the C-ABI calls.

This module owns buffers and call order only; every value is computed by
libsd's kernels.  A step for one layer, all heads and the whole batch is

    query map (Hamming) or read plan (bit planes)  ->  sd_score  ->  sd_topk
        ->  sd_gather_attend

and the per-stage split T = T_qmap + T_scan + T_topk + T_att follows
HashAttention: Semantic Sparsity for Faster Inference, 2.5.  For bit planes the
read plan is computed inside the scan (sd_plan_score, same results) unless
StepConfig.plan_in_scan is False, and the scan also writes each 32-token word's
maximum score, from which sd_topk_wmax draws the same top-k as sd_topk unless
StepConfig.wmax is False (with StepConfig.select_attend the top-k and the
gather-attend then run as one call, sd_select_attend, same results); with
StepConfig.fused the scan and the top-k run as one call instead (sd_score_topk,
same results).  For signatures the scan
and the top-k run as one call (sd_hamming_topk, same idx and count, no scores)
unless StepConfig.hamming_fused is False.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

from . import (SD_IDX_LANDMARK, SD_IDX_MINMAX, SD_IDX_PLANES, SD_IDX_SIG, SD_PLAN_WATERFILL,
               SD_SCORE_F32, SD_SCORE_I32, make_select, make_shape, sd_build_index, sd_encode_query,
               sd_gather_attend, sd_gather_attend_workspace_size, sd_plan, sd_plan_score,
               sd_score, sd_score_topk, sd_score_topk_workspace_size, sd_topk,
               sd_hamming_topk, sd_hamming_topk_workspace_size, sd_select_attend,
               sd_select_attend_workspace_size, sd_topk_wmax,
               sd_topk_workspace_size)

KIND_NAMES = {SD_IDX_SIG: "hamming", SD_IDX_PLANES: "planes", SD_IDX_MINMAX: "quest",
              SD_IDX_LANDMARK: "landmark"}
BLOCK_OF = {SD_IDX_MINMAX: 16, SD_IDX_LANDMARK: 8}  # tokens per scored unit (else 1)


@dataclasses.dataclass
class StepConfig:
    kind: int                 # SD_IDX_SIG, SD_IDX_PLANES, SD_IDX_MINMAX or SD_IDX_LANDMARK
    B: int
    Hq: int
    Hkv: int
    n: int
    d: int = 128
    k: int = 512              # tokens (token mode) or blocks (MINMAX, LANDMARK)
    sink: int = 0             # forced leading units
    local: int = 0            # forced trailing units
    plan_mode: int = SD_PLAN_WATERFILL
    budget: int = 56          # bits per token per KV head (water-filling) or r (fixed)
    fused: bool = False       # bit planes: scan and top-k in one call (sd_score_topk)
    plan_in_scan: bool = True  # bit planes: the plan computed by the scan (sd_plan_score)
    wmax: bool = True         # bit planes with plan_in_scan: word maxima -> sd_topk_wmax
    select_attend: bool = False  # with wmax: top-k and gather-attend in one call
    hamming_fused: bool = True  # signatures: scan and top-k in one call (sd_hamming_topk)
    n_cap: int = 0            # allocated tokens per (sequence, KV head), >= n (0: n); the
                              # stride of K, V and the index; a multiple of 64 for planes

    @property
    def cap(self) -> int:
        return self.n_cap or self.n

    @property
    def block(self) -> int:
        return BLOCK_OF.get(self.kind, 1)

    @property
    def n_units(self) -> int:
        return (self.n + self.block - 1) // self.block

    @property
    def max_count(self) -> int:
        return min(self.n_units, self.sink + self.local + self.k) * self.block


def index_buffers(cfg: StepConfig, device="cuda") -> dict:
    """Allocates the key-side index of cfg.kind (uninitialised)."""
    B, H, n, d = cfg.B, cfg.Hkv, cfg.cap, cfg.d
    if cfg.kind == SD_IDX_SIG:
        return {"sig": torch.empty((B, H, n), dtype=torch.int32, device=device)}
    if cfg.kind == SD_IDX_PLANES:
        return {"planes": torch.empty((B, H, d, 4, n // 32), dtype=torch.int32, device=device),
                "scales": torch.empty((B, H, d, n // 64), dtype=torch.int16, device=device)}
    if cfg.kind == SD_IDX_LANDMARK:
        return {"landmarks": torch.empty((B, H, (n + 7) // 8, d), dtype=torch.int16,
                                         device=device)}
    nblk = (n + 15) // 16
    return {"summ": torch.empty((B, H, nblk, 2, d), dtype=torch.int16, device=device)}


def build_index(cfg: StepConfig, K: torch.Tensor, enc=None, stream=None) -> dict:
    """Runs sd_build_index for cfg.kind (the KV-write path) and returns the index."""
    shp = make_shape(cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.d, cfg.n_cap)
    idx = index_buffers(cfg, K.device)
    if cfg.kind == SD_IDX_SIG:
        sd_build_index(SD_IDX_SIG, shp, K, enc, idx["sig"], None, stream)
    elif cfg.kind == SD_IDX_PLANES:
        sd_build_index(SD_IDX_PLANES, shp, K, None, idx["planes"], idx["scales"], stream)
    elif cfg.kind == SD_IDX_LANDMARK:
        sd_build_index(SD_IDX_LANDMARK, shp, K, None, idx["landmarks"], None, stream)
    else:
        sd_build_index(SD_IDX_MINMAX, shp, K, None, idx["summ"], None, stream)
    return idx


class DecodeStep:
    """Preallocated buffers and the call sequence of one decode step."""

    def __init__(self, cfg: StepConfig, K: torch.Tensor, V: torch.Tensor, index: dict,
                 enc=None, sigma2: Optional[torch.Tensor] = None,
                 scale: Optional[float] = None):
        self.cfg = cfg
        self.K, self.V, self.index, self.enc, self.sigma2 = K, V, index, enc, sigma2
        self.scale = 1.0 / math.sqrt(cfg.d) if scale is None else scale
        dev = K.device
        c = cfg
        self.shape = make_shape(c.B, c.Hq, c.Hkv, c.n, c.d, c.n_cap)
        self.rows = c.B * c.Hkv
        self.sel = make_select(c.k, c.sink, c.local, c.block)
        sdt = torch.int32 if c.kind == SD_IDX_SIG else torch.float32
        self.scores = torch.empty((self.rows, c.n_units), dtype=sdt, device=dev)
        self.qsig = torch.empty((c.B, c.Hq), dtype=torch.int32, device=dev)
        self.plan = torch.empty((c.B, c.Hkv, c.d), dtype=torch.uint8, device=dev)
        self.idx = torch.empty((self.rows, c.max_count), dtype=torch.int32, device=dev)
        self.count = torch.empty((self.rows,), dtype=torch.int32, device=dev)
        tws = sd_topk_workspace_size(self.rows, c.n_units, self.sel)
        self.topk_ws = torch.empty(tws, dtype=torch.uint8, device=dev) if tws else None
        self.fused = c.fused and c.kind == SD_IDX_PLANES
        self.use_wmax = (c.kind == SD_IDX_PLANES and c.plan_in_scan and c.wmax and not self.fused)
        self.wmax = (torch.empty((self.rows, (c.n + 31) // 32), dtype=torch.float32, device=dev)
                     if self.use_wmax else None)
        self.wmax_fresh = False  # the last scan wrote the word maxima of self.scores
        if self.fused:
            fws = sd_score_topk_workspace_size(self.shape, self.sel)
            self.fused_ws = torch.empty(max(fws, 256), dtype=torch.uint8, device=dev)
        aws = sd_gather_attend_workspace_size(self.shape, c.max_count)
        self.att_ws = torch.empty(max(aws, 256), dtype=torch.uint8, device=dev)
        self.use_sa = self.use_wmax and c.select_attend
        self.use_ht = c.kind == SD_IDX_SIG and c.hamming_fused and c.block == 1
        if self.use_ht:
            hws = sd_hamming_topk_workspace_size(self.shape, self.sel)
            self.ht_ws = torch.empty(max(hws, 256), dtype=torch.uint8, device=dev)
        if self.use_sa:
            sws = sd_select_attend_workspace_size(self.shape, self.sel, c.max_count)
            self.sa_ws = torch.empty(max(sws, 256), dtype=torch.uint8, device=dev)
        # out and lse in one buffer (out first), so that one copy moves the result
        nout = c.B * c.Hq * c.d
        self.result = torch.empty(nout + c.B * c.Hq, dtype=torch.float32, device=dev)
        self.out = self.result[:nout].view(c.B, c.Hq, c.d)
        self.lse = self.result[nout:].view(c.B, c.Hq)

    # the four stages, separately callable for per-stage timing
    def stage_prep(self, q, stream=None):
        c = self.cfg
        if c.kind == SD_IDX_SIG:
            sd_encode_query(self.shape, q, self.enc, self.qsig, stream)
        elif c.kind == SD_IDX_PLANES:
            sd_plan(self.shape, q, self.sigma2, c.plan_mode, c.budget, self.plan, stream)

    def stage_score(self, q, stream=None):
        c, ix = self.cfg, self.index
        self.wmax_fresh = False  # sd_score writes no word maxima
        if c.kind == SD_IDX_SIG:
            sd_score(SD_IDX_SIG, self.shape, ix["sig"], None, self.qsig, None, self.scores, stream)
        elif c.kind == SD_IDX_PLANES:
            sd_score(SD_IDX_PLANES, self.shape, ix["planes"], ix["scales"], q, self.plan,
                     self.scores, stream)
        elif c.kind == SD_IDX_LANDMARK:
            sd_score(SD_IDX_LANDMARK, self.shape, ix["landmarks"], None, q, None, self.scores,
                     stream)
        else:
            sd_score(SD_IDX_MINMAX, self.shape, ix["summ"], None, q, None, self.scores, stream)

    def stage_topk(self, stream=None):
        c = self.cfg
        if self.use_wmax and self.wmax_fresh:
            sd_topk_wmax(self.scores, self.wmax, self.rows, c.n, self.sel, self.idx, c.max_count,
                         self.count, self.topk_ws, stream)
            return
        st = SD_SCORE_I32 if c.kind == SD_IDX_SIG else SD_SCORE_F32
        sd_topk(st, self.scores, self.rows, c.n_units, c.n, self.sel, self.idx, c.max_count,
                self.count, self.topk_ws, stream)

    def stage_plan_score(self, q, stream=None):
        """Bit planes: the read plan computed inside the scan (same plan and scores
        as stage_prep followed by stage_score)."""
        c, ix = self.cfg, self.index
        sd_plan_score(self.shape, ix["planes"], ix["scales"], q, self.sigma2, c.plan_mode,
                      c.budget, self.plan, self.scores, self.wmax, stream)
        self.wmax_fresh = self.wmax is not None

    def stage_score_topk(self, q, stream=None):
        """Bit planes: the scan and the top-k in one call (same results as
        stage_score followed by stage_topk)."""
        ix = self.index
        self.wmax_fresh = False
        sd_score_topk(self.shape, ix["planes"], ix["scales"], q, self.plan, self.sel,
                      self.scores, self.idx, self.cfg.max_count, self.count, self.fused_ws,
                      stream)

    def stage_attend(self, q, stream=None):
        c = self.cfg
        sd_gather_attend(self.shape, q, self.K, self.V, self.idx, c.max_count, self.count,
                         c.max_count, self.scale, self.out, self.lse, self.att_ws, stream)

    def stage_hamming_topk(self, q, stream=None):
        """Signatures: the scan and the top-k in one call, without scores (same idx
        and count as stage_score followed by stage_topk)."""
        c = self.cfg
        sd_hamming_topk(self.shape, self.index["sig"], self.qsig, self.sel, self.idx,
                        c.max_count, self.count, self.ht_ws, stream)

    def stage_select_attend(self, q, stream=None):
        """Bit planes with word maxima: the top-k and gather-attend in one call (same
        idx, count, out and lse as stage_topk followed by stage_attend)."""
        c = self.cfg
        if not self.wmax_fresh:
            self.stage_topk(stream)
            self.stage_attend(q, stream)
            return
        sd_select_attend(self.shape, self.scores, self.wmax, self.sel, q, self.K, self.V,
                         self.scale, self.idx, c.max_count, self.count, c.max_count, self.out,
                         self.lse, self.sa_ws, stream)

    def stages(self):
        """(name, fn(q, stream)) of the step's stages in call order."""
        topk = ("topk", lambda q, stream=None: self.stage_topk(stream))
        if self.fused:
            return [("plan", self.stage_prep), ("scan_topk", self.stage_score_topk),
                    ("gather_attend", self.stage_attend)]
        if self.use_ht:
            return [("prep", self.stage_prep), ("scan_topk", self.stage_hamming_topk),
                    ("gather_attend", self.stage_attend)]
        if self.use_sa:
            return [("plan_scan", self.stage_plan_score),
                    ("select_attend", self.stage_select_attend)]
        if self.cfg.kind == SD_IDX_PLANES and self.cfg.plan_in_scan:
            return [("plan_scan", self.stage_plan_score), topk,
                    ("gather_attend", self.stage_attend)]
        first = "plan" if self.cfg.kind == SD_IDX_PLANES else "prep"
        return [(first, self.stage_prep), ("scan", self.stage_score), topk,
                ("gather_attend", self.stage_attend)]

    def run(self, q, stream=None, trace: bool = False):
        """One step.  With trace, each stage is an NVTX range named after it (for a
        profiler's timeline; the ranges cost nothing when no tool is attached)."""
        run_stages(self.stages(), q, stream, trace)
        return self.out


def run_stages(stages, q, stream=None, trace: bool = False, push=None, pop=None):
    """Calls each (name, fn) of `stages` as fn(q, stream), in order; with trace,
    inside an NVTX range of that name (push/pop default to torch.cuda.nvtx)."""
    if trace:
        push = push or torch.cuda.nvtx.range_push
        pop = pop or torch.cuda.nvtx.range_pop
    for name, fn in stages:
        if trace:
            push(f"sd.{name}")
        try:
            fn(q, stream)
        finally:
            if trace:
                pop()
