"""Seeded synthetic inputs for the sparse-decode workloads.

This module produces inputs only: bf16 keys, values and queries, per-channel
calibration variances, encoder weights, planted positions, and free-standing
score arrays and index lists for testing one stage in isolation.  It holds none
of the method's arithmetic (no signature, quantiser, score, selection or
attention step), so that the CUDA library and the CPU oracle can both consume
it without sharing any of the computation they are compared on.

Recipe (all configs):
  * counter-based SplitMix64 stream per (seed, tensor id); Box-Muller normals;
    bf16 by round-to-nearest-even (see synth_gen.c);
  * seed = 20260000 + config id;
  * sigma_j = exp(U[ln 0.1, ln 4]) per (KV head, channel); k_ij ~ N(0, sigma_j^2),
    v ~ N(0, 1), q ~ N(0, 1);
  * planted keys: ||sigma||_2 * q~ / ||q~|| with q~ = sum of the GQA group's
    queries, at distinct uniform positions outside the forced windows;
  * block mode plants whole 16-token blocks: aligned vector + N(0, (sigma_j/4)^2).
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gen.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# tensor ids of the counter streams
TID_Q, TID_K, TID_V, TID_SIGMA, TID_W1, TID_W2, TID_PLANT, TID_BLOCKNOISE = 1, 2, 3, 4, 5, 6, 7, 8
TID_SCORES, TID_IDX = 20, 21


def build(force: bool = False) -> str:
    """Compile libsynth.so next to its source (plain gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _l():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
            lib.synth_uniform.argtypes = [u64, u64, i64, i64, p]
            lib.synth_normal_f64.argtypes = [u64, u64, i64, i64, p]
            lib.synth_normal_f32.argtypes = [u64, u64, i64, ctypes.c_double, p]
            lib.synth_fill_normal_bf16.argtypes = [u64, u64, i64, i64, p, i64, i64, p]
            lib.synth_f64_to_bf16.argtypes = [p, i64, p]
            for f in ("synth_uniform", "synth_normal_f64", "synth_normal_f32",
                      "synth_fill_normal_bf16", "synth_f64_to_bf16"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def uniform(seed: int, tid: int, count: int, start: int = 0) -> np.ndarray:
    out = np.empty(count, np.float64)
    _l().synth_uniform(seed, tid, start, count, _ptr(out))
    return out


def normal(seed: int, tid: int, count: int, start: int = 0) -> np.ndarray:
    out = np.empty(count, np.float64)
    _l().synth_normal_f64(seed, tid, start, count, _ptr(out))
    return out


def normal_f32(seed: int, tid: int, shape, std: float) -> np.ndarray:
    out = np.empty(int(np.prod(shape)), np.float32)
    _l().synth_normal_f32(seed, tid, out.size, float(std), _ptr(out))
    return out.reshape(shape)


def normal_bf16(seed: int, tid: int, nrows: int, ncols: int,
                sigma: Optional[np.ndarray] = None, rows_per_sigma: int = 1) -> np.ndarray:
    """bf16 bit patterns (uint16) of an nrows x ncols normal matrix."""
    out = np.empty((nrows, ncols), np.uint16)
    if sigma is None:
        _l().synth_fill_normal_bf16(seed, tid, nrows, ncols, None, 1, 1, _ptr(out))
    else:
        s = np.ascontiguousarray(sigma, np.float64)
        _l().synth_fill_normal_bf16(seed, tid, nrows, ncols, _ptr(s), rows_per_sigma,
                                    s.shape[0], _ptr(out))
    return out


def to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _l().synth_f64_to_bf16(_ptr(x), x.size, _ptr(out))
    return out


def bf16_to_f64(x: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------------------
# Workload configurations (Qwen3-8B-layer-shaped unless stated)
# --------------------------------------------------------------------------------------
@dataclasses.dataclass
class Config:
    cid: int
    name: str
    B: int
    Hq: int
    Hkv: int
    n: int
    d: int = 128
    planted: int = 8              # planted keys (token mode) or blocks (block mode) per (b, KV head)
    block_mode: bool = False      # plant 16-token blocks instead of single keys
    sink: int = 0                 # forced leading tokens
    local: int = 0                # forced trailing tokens
    k: int = 512                  # retrieval budget (tokens)
    hidden: int = 0               # 0: single 128->32 projection, else 2-layer MLP width
    budgets: tuple = (56,)        # water-filling budgets (bits per token per KV head)
    fixed_r: int = 0              # FIXED(r) plan width (0: not used)
    blk_k: int = 0                # block mode: top blocks
    blk_local: int = 1            # block mode: forced trailing blocks

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def seed(self) -> int:
        return 20260000 + self.cid


CONFIGS: Dict[int, Config] = {
    0: Config(0, "tiny", B=1, Hq=4, Hkv=1, n=4096, sink=4, local=64, k=64, hidden=0,
              budgets=(56,), blk_k=4, blk_local=1),
    1: Config(1, "hash-32k", B=1, Hq=32, Hkv=8, n=32768, sink=128, local=512, k=512,
              hidden=128),
    2: Config(2, "fathom-128k", B=4, Hq=32, Hkv=8, n=131072, k=512,
              budgets=(47, 56, 92)),
    3: Config(3, "quest-b64-16k", B=64, Hq=32, Hkv=8, n=16384, planted=16, block_mode=True,
              blk_k=128, blk_local=1),
    4: Config(4, "longctx-1m", B=1, Hq=32, Hkv=8, n=1 << 20, k=512, budgets=(56,),
              fixed_r=32, hidden=0),
}


def config(cid: int, **over) -> Config:
    return dataclasses.replace(CONFIGS[cid], **over)


@dataclasses.dataclass
class Inputs:
    cfg: Config
    q: np.ndarray          # uint16 bf16 [B][Hq][d]
    K: np.ndarray          # uint16 bf16 [B][Hkv][n][d]
    V: np.ndarray          # uint16 bf16 [B][Hkv][n][d]
    sigma2: np.ndarray     # float32 [Hkv][d]
    W1: np.ndarray         # float32 [hidden or 32][d]
    b1: np.ndarray         # float32 [hidden or 32]
    W2: Optional[np.ndarray]   # float32 [32][hidden] (None for a single projection)
    b2: Optional[np.ndarray]   # float32 [32]
    planted: np.ndarray    # int64 [B][Hkv][P]: token positions, or block ids in block mode


def _distinct_positions(seed: int, stream: int, lo: int, hi: int, count: int) -> np.ndarray:
    """count distinct uniform integers in [lo, hi), drawn in counter order."""
    span = hi - lo
    if span <= 0 or count <= 0:
        return np.zeros(0, np.int64)
    count = min(count, span)
    got, seen, ctr = [], set(), 0
    while len(got) < count:
        u = uniform(seed, TID_PLANT, 64, start=stream * (1 << 20) + ctr)
        ctr += 64
        for x in u:
            p = lo + min(int(x * span), span - 1)
            if p not in seen:
                seen.add(p)
                got.append(p)
                if len(got) == count:
                    break
    return np.array(sorted(got), np.int64)


def make_inputs(cfg: Config, with_v: bool = True) -> Inputs:
    B, Hq, Hkv, n, d, G = cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.d, cfg.G
    seed = cfg.seed
    # calibration: sigma_j log-uniform in [0.1, 4] per (KV head, channel)
    u = uniform(seed, TID_SIGMA, Hkv * d).reshape(Hkv, d)
    sigma = np.exp(math.log(0.1) + u * (math.log(4.0) - math.log(0.1)))
    sigma2 = (sigma * sigma).astype(np.float32)
    q = normal_bf16(seed, TID_Q, B * Hq, d).reshape(B, Hq, d)
    K = normal_bf16(seed, TID_K, B * Hkv * n, d, sigma=sigma, rows_per_sigma=n).reshape(B, Hkv, n, d)
    V = (normal_bf16(seed, TID_V, B * Hkv * n, d).reshape(B, Hkv, n, d) if with_v
         else np.zeros((0,), np.uint16))
    # encoder weights (seeded, untrained): SimHash projection or 2-layer MLP
    if cfg.hidden == 0:
        W1 = normal_f32(seed, TID_W1, (32, d), 1.0)
        b1 = np.zeros(32, np.float32)
        W2 = b2 = None
    else:
        W1 = normal_f32(seed, TID_W1, (cfg.hidden, d), math.sqrt(1.0 / d))
        b1 = np.zeros(cfg.hidden, np.float32)
        W2 = normal_f32(seed, TID_W2, (32, cfg.hidden), math.sqrt(1.0 / cfg.hidden))
        b2 = np.zeros(32, np.float32)
    # planted keys aligned with the group-summed query
    qf = bf16_to_f64(q)
    P = cfg.planted
    if cfg.block_mode:
        nblk = (n + 15) // 16
        planted = np.zeros((B, Hkv, P), np.int64)
        for b in range(B):
            for h in range(Hkv):
                pos = _distinct_positions(seed, b * Hkv + h, 0, nblk - cfg.blk_local, P)
                planted[b, h, :len(pos)] = pos
                qt = qf[b, h * G:(h + 1) * G].sum(axis=0)
                a = np.linalg.norm(sigma[h]) * qt / max(np.linalg.norm(qt), 1e-30)
                rows = (pos[:, None] * 16 + np.arange(16)[None, :]).reshape(-1)
                rows = rows[rows < n]
                noise = normal(seed, TID_BLOCKNOISE, rows.size * d,
                               start=(b * Hkv + h) * (1 << 24)).reshape(rows.size, d)
                K[b, h, rows] = to_bf16(a[None, :] + noise * (sigma[h][None, :] / 4.0))
    else:
        planted = np.zeros((B, Hkv, P), np.int64)
        for b in range(B):
            for h in range(Hkv):
                pos = _distinct_positions(seed, b * Hkv + h, cfg.sink, n - cfg.local, P)
                planted[b, h, :len(pos)] = pos
                qt = qf[b, h * G:(h + 1) * G].sum(axis=0)
                a = np.linalg.norm(sigma[h]) * qt / max(np.linalg.norm(qt), 1e-30)
                K[b, h, pos] = to_bf16(a)[None, :]
    return Inputs(cfg, q, K, V, sigma2, W1, b1, W2, b2, planted)


# --------------------------------------------------------------------------------------
# Free-standing stage inputs (to test one stage on identical inputs on both sides)
# --------------------------------------------------------------------------------------
def make_scores(seed: int, rows: int, n: int, kind: str, levels: int = 0) -> np.ndarray:
    """Synthetic score rows.  kind: 'f32' (normal), 'f32ties' (normal rounded to
    `levels` distinct values, with some +-0.0), 'int' (integers in [-levels, 0]),
    'const' (all equal)."""
    z = normal(seed, TID_SCORES, rows * n).reshape(rows, n)
    if kind == "f32":
        return z.astype(np.float32)
    if kind == "f32ties":
        lv = max(levels, 2)
        x = np.round(z * lv / 4.0) / lv
        s = x.astype(np.float32)
        neg0 = uniform(seed, TID_SCORES + 1, rows * n).reshape(rows, n) < 0.02
        s[neg0 & (s == 0)] = np.float32(-0.0)
        return s
    if kind == "int":
        u = uniform(seed, TID_SCORES + 2, rows * n).reshape(rows, n)
        return (-np.floor(u * (levels + 1))).astype(np.int32)
    if kind == "const":
        return np.zeros((rows, n), np.float32)
    raise ValueError(kind)


def make_index_lists(seed: int, rows: int, n: int, max_count: int,
                     counts: Optional[np.ndarray] = None) -> tuple:
    """Sorted distinct token indices per row, padded with -1 to max_count."""
    idx = np.full((rows, max_count), -1, np.int32)
    if counts is None:
        cu = uniform(seed, TID_IDX, rows)
        counts = np.maximum(1, (cu * max_count).astype(np.int64))
    counts = np.minimum(np.asarray(counts, np.int64), min(max_count, n))
    for r in range(rows):
        u = uniform(seed, TID_IDX + 1, n, start=r * n)
        pick = np.sort(np.argsort(u, kind="stable")[: counts[r]])
        idx[r, : counts[r]] = pick
    return idx, counts.astype(np.int32)
