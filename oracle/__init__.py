"""CPU oracle for the sparse-decode hot path.  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  It wraps ``sd_oracle.c`` (plain C, double accumulation,
built with ``-ffp-contract=off``), which shares no code with the CUDA library.
Every function takes and returns numpy arrays; bf16 tensors travel as their
uint16 bit patterns.

Pins (tests/test_oracle_pins.py) tie each function to something other than
itself: the HashAttention worked example, the bit-plane prefix invariant, brute
force over all bf16 values, brute-force water-filling, the Quest bound,
brute-force top-k, dense softmax attention at k = n.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sd_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PLAN_WATERFILL, PLAN_FIXED, PLAN_FULL = 0, 1, 2
PLAN_TOPQ = 3  # SparQ-style: the r channels of largest sum_g q_gj^2, 4 bits each
PLAN_SPLIT = 4  # water-filling of a sequence's Hkv * budget bits across its KV heads


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _l():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
            lib.orc_f32_to_f16.restype = ctypes.c_uint16
            lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_f32.restype = ctypes.c_float
            lib.orc_threads.argtypes = []
            lib.orc_threads.restype = i32
            lib.orc_set_threads.argtypes = [i32]
            lib.orc_set_threads.restype = i32
            lib.orc_reconstruct.argtypes = [i32, i32, d]
            lib.orc_reconstruct.restype = d
            lib.orc_sig_encode.argtypes = [p, i64, i32, p, p, i32, p, p, p]
            lib.orc_sig_encode.restype = i32
            lib.orc_hamming_score.argtypes = [p, i64, i32, i32, i64, p, p]
            lib.orc_hamming_score.restype = None
            lib.orc_plane_build.argtypes = [p, i64, i32, i64, i32, p, p]
            lib.orc_plane_build.restype = i32
            lib.orc_plan.argtypes = [p, p, i64, i32, i32, i32, i32, i32, p]
            lib.orc_plan.restype = i32
            lib.orc_plane_score.argtypes = [p, p, p, p, i64, i32, i32, i64, i32, p]
            lib.orc_plane_score.restype = None
            lib.orc_plane_score_l1.argtypes = [p, p, p, p, i64, i32, i32, i64, i32, p]
            lib.orc_plane_score_l1.restype = None
            lib.orc_minmax_build.argtypes = [p, i64, i32, i64, i32, p]
            lib.orc_minmax_build.restype = None
            lib.orc_quest_score.argtypes = [p, p, i64, i32, i32, i64, i32, p, p]
            lib.orc_quest_score.restype = None
            lib.orc_topk.argtypes = [p, i32, i64, i64, i32, i32, i32, i32, i64, p, i64, p]
            lib.orc_topk.restype = None
            lib.orc_gather_attend.argtypes = [p, p, p, i64, i32, i32, i64, i32, p, i64, p, d,
                                              p, p]
            lib.orc_gather_attend.restype = None
            lib.orc_prefix_copy.argtypes = [p, p, p, i64, i32, i64, i32, p, p]
            lib.orc_prefix_copy.restype = None
            lib.orc_delta_select.argtypes = [i64, i64, i64, i32, i32, i32, p, p, i64, p, i32,
                                             i64, i32, p, p, p, p, p, p, p, p, i64, p]
            lib.orc_delta_select.restype = i32
            lib.orc_landmark_build.argtypes = [p, i64, i32, i64, i32, i32, p]
            lib.orc_landmark_build.restype = None
            lib.orc_landmark_score.argtypes = [p, p, i64, i32, i32, i64, i32, p, p]
            lib.orc_landmark_score.restype = None
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def threads() -> int:
    return int(_l().orc_threads())


def set_threads(t: int) -> int:
    """Threads of the oracle's parallel loops from now on; returns the previous count."""
    return int(_l().orc_set_threads(int(t)))


def f32_to_f16(x: float) -> int:
    return int(_l().orc_f32_to_f16(float(x)))


def f16_to_f32(h: int) -> float:
    return float(_l().orc_f16_to_f32(int(h)))


def reconstruct(prefix: int, t: int, s: float) -> float:
    return float(_l().orc_reconstruct(int(prefix), int(t), float(s)))


def sig_encode(x_bf16: np.ndarray, W1, b1, W2=None, b2=None) -> np.ndarray:
    """32-bit signatures of the rows of x (last dim d)."""
    x, px = _c(x_bf16, np.uint16)
    d = x.shape[-1]
    rows = x.size // d
    W1, pW1 = _c(W1, np.float32)
    b1, pb1 = _c(b1, np.float32)
    hidden = 0
    pW2 = pb2 = None
    if W2 is not None:
        hidden = W1.shape[0]
        W2, pW2 = _c(W2, np.float32)
        b2, pb2 = _c(b2, np.float32)
    out = np.empty(rows, np.uint32)
    rc = _l().orc_sig_encode(px, rows, d, pW1, pb1, hidden, pW2, pb2, out.ctypes.data)
    if rc:
        raise ValueError("orc_sig_encode: unsupported size")
    return out.reshape(x.shape[:-1])


def hamming_score(sig: np.ndarray, qsig: np.ndarray) -> np.ndarray:
    """sig uint32 [B][Hkv][n], qsig uint32 [B][Hq] -> int32 [B][Hkv][n]."""
    sig, ps = _c(sig, np.uint32)
    qsig, pq = _c(qsig, np.uint32)
    B, Hkv, n = sig.shape
    Hq = qsig.shape[1]
    out = np.empty((B, Hkv, n), np.int32)
    _l().orc_hamming_score(ps, B, Hq, Hkv, n, pq, out.ctypes.data)
    return out


def plane_build(K: np.ndarray):
    """K bf16 [B][Hkv][n][d] -> planes uint32 [B][Hkv][d][4][2 nb], scales f16 bits
    uint16 [B][Hkv][d][nb], nb = ceil(n / 64) (a partial last block: scale over the
    tokens it holds, bits past n zero)."""
    K, pk = _c(K, np.uint16)
    B, Hkv, n, d = K.shape
    nb = (n + 63) // 64
    planes = np.empty((B, Hkv, d, 4, 2 * nb), np.uint32)
    scales = np.empty((B, Hkv, d, nb), np.uint16)
    if _l().orc_plane_build(pk, B, Hkv, n, d, planes.ctypes.data, scales.ctypes.data):
        raise ValueError("plane_build needs n >= 1")
    return planes, scales


def plan(q: np.ndarray, sigma2: np.ndarray, Hkv: int, mode: int, budget: int) -> np.ndarray:
    """q bf16 [B][Hq][d], sigma2 f32 [Hkv][d] -> plan uint8 [B][Hkv][d]."""
    q, pq = _c(q, np.uint16)
    s2, ps = _c(sigma2, np.float32)
    B, Hq, d = q.shape
    out = np.empty((B, Hkv, d), np.uint8)
    if _l().orc_plan(pq, ps, B, Hq, Hkv, d, mode, budget, out.ctypes.data):
        raise ValueError("plan: bad mode/budget")
    return out


def plane_score(planes, scales, plan_, q, with_l1: bool = False, n: int = None):
    """Scores of the n tokens (default: every position the planes hold) from the
    planes [B][Hkv][d][4][2 nb] and scales [B][Hkv][d][nb], nb = ceil(n / 64)."""
    planes, pp = _c(planes, np.uint32)
    scales, psc = _c(scales, np.uint16)
    plan_, ppl = _c(plan_, np.uint8)
    q, pq = _c(q, np.uint16)
    B, Hkv, d, _, nw = planes.shape
    if n is None:
        n = nw * 32
    if nw != 2 * ((n + 63) // 64) or scales.shape[-1] != nw // 2:
        raise ValueError("plane_score: planes / scales do not hold ceil(n / 64) blocks")
    Hq = q.shape[1]
    out = np.empty((B, Hkv, n), np.float64)
    _l().orc_plane_score(pp, psc, ppl, pq, B, Hq, Hkv, n, d, out.ctypes.data)
    if not with_l1:
        return out
    l1 = np.empty((B, Hkv, n), np.float64)
    _l().orc_plane_score_l1(pp, psc, ppl, pq, B, Hq, Hkv, n, d, l1.ctypes.data)
    return out, l1


def minmax_build(K: np.ndarray) -> np.ndarray:
    """K bf16 [B][Hkv][n][d] -> summ bf16 [B][Hkv][ceil(n/16)][2][d]."""
    K, pk = _c(K, np.uint16)
    B, Hkv, n, d = K.shape
    nblk = (n + 15) // 16
    out = np.empty((B, Hkv, nblk, 2, d), np.uint16)
    _l().orc_minmax_build(pk, B, Hkv, n, d, out.ctypes.data)
    return out


def quest_score(summ, q, with_l1: bool = False):
    summ, ps = _c(summ, np.uint16)
    q, pq = _c(q, np.uint16)
    B, Hkv, nblk, _, d = summ.shape
    Hq = q.shape[1]
    U = np.empty((B, Hkv, nblk), np.float64)
    l1 = np.empty((B, Hkv, nblk), np.float64)
    _l().orc_quest_score(ps, pq, B, Hq, Hkv, nblk, d, U.ctypes.data, l1.ctypes.data)
    return (U, l1) if with_l1 else U


LANDMARK_BLOCK = 8


def landmark_build(K: np.ndarray, blk: int = LANDMARK_BLOCK) -> np.ndarray:
    """K bf16 [B][Hkv][n][d] -> landmarks bf16 [B][Hkv][ceil(n/blk)][d] (block means)."""
    K, pk = _c(K, np.uint16)
    B, Hkv, n, d = K.shape
    out = np.empty((B, Hkv, (n + blk - 1) // blk, d), np.uint16)
    _l().orc_landmark_build(pk, B, Hkv, n, d, blk, out.ctypes.data)
    return out


def landmark_score(L, q, with_l1: bool = False):
    """L bf16 [B][Hkv][nblk][d], q bf16 [B][Hq][d] -> U float64 [B][Hkv][nblk]."""
    L, pl = _c(L, np.uint16)
    q, pq = _c(q, np.uint16)
    B, Hkv, nblk, d = L.shape
    Hq = q.shape[1]
    U = np.empty((B, Hkv, nblk), np.float64)
    l1 = np.empty((B, Hkv, nblk), np.float64)
    _l().orc_landmark_score(pl, pq, B, Hq, Hkv, nblk, d, U.ctypes.data, l1.ctypes.data)
    return (U, l1) if with_l1 else U


def topk(scores: np.ndarray, k: int, sink: int = 0, local: int = 0, block: int = 1,
         n_tokens: int = None):
    """scores [rows..., n_units] (int32, float32 or float64) -> (idx int32
    [rows..., max_count] padded with -1, count int32 [rows...])."""
    kind = {np.dtype(np.int32): 0, np.dtype(np.float32): 1, np.dtype(np.float64): 2}[
        np.asarray(scores).dtype]
    s = np.ascontiguousarray(scores)
    lead_shape = s.shape[:-1]
    n_units = s.shape[-1]
    rows = int(np.prod(lead_shape)) if lead_shape else 1
    if n_tokens is None:
        n_tokens = n_units * block
    max_units = min(n_units, sink + local + k)
    stride = max(1, max_units * block)
    idx = np.full((rows, stride), -1, np.int32)
    count = np.empty(rows, np.int32)
    _l().orc_topk(s.ctypes.data, kind, rows, n_units, k, sink, local, block, n_tokens,
                  idx.ctypes.data, stride, count.ctypes.data)
    return idx.reshape(lead_shape + (stride,)), count.reshape(lead_shape)


def gather_attend(q, K, V, idx, count, scale: float):
    """-> (o float64 [B][Hq][d], lse float64 [B][Hq])."""
    q, pq = _c(q, np.uint16)
    K, pk = _c(K, np.uint16)
    V, pv = _c(V, np.uint16)
    idx, pi = _c(idx, np.int32)
    count, pc = _c(count, np.int32)
    B, Hq, d = q.shape
    Hkv, n = K.shape[1], K.shape[2]
    stride = idx.shape[-1]
    out = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    _l().orc_gather_attend(pq, pk, pv, B, Hq, Hkv, n, d, pi, stride, pc, float(scale),
                           out.ctypes.data, lse.ctypes.data)
    return out, lse


def prefix_copy(src_planes, src_scales, plan_, dst_planes, dst_scales):
    """Copy the planned prefixes (and the active channels' scales) into dst in place."""
    src_planes, pp = _c(src_planes, np.uint32)
    src_scales, ps = _c(src_scales, np.uint16)
    plan_, ppl = _c(plan_, np.uint8)
    assert dst_planes.flags["C_CONTIGUOUS"] and dst_scales.flags["C_CONTIGUOUS"]
    B, Hkv, d, _, nw = src_planes.shape
    _l().orc_prefix_copy(pp, ps, ppl, B, Hkv, nw * 32, d, dst_planes.ctypes.data,
                         dst_scales.ctypes.data)


class Resident:
    """Resident-set state of the delta selection, per row (sequence, KV head):
    slot_unit [rows][R], slot_last [rows][R] (int64), unit_slot [rows][n_units];
    all -1 when empty."""

    def __init__(self, rows: int, R: int, n_units: int):
        self.slot_unit = np.full((rows, R), -1, np.int32)
        self.slot_last = np.full((rows, R), -1, np.int64)
        self.unit_slot = np.full((rows, n_units), -1, np.int32)

    def copy(self):
        r = Resident.__new__(Resident)
        r.slot_unit, r.slot_last, r.unit_slot = (self.slot_unit.copy(), self.slot_last.copy(),
                                                 self.unit_slot.copy())
        return r


def delta_select(state: Resident, scores, idx, count, block: int, n_tokens: int, sink: int,
                 local: int, C: int, step: int, pool_stride: int):
    """One step of the delta selection; updates `state` in place.  scores float32
    [rows][n_units], idx/count the top-k output (tokens).  Returns (plan_slot,
    plan_unit, plan_evict [rows][C], plan_count [rows], pool_idx [rows][pool_stride]
    (-1 past pool_count), pool_count [rows])."""
    scores, psc = _c(scores, np.float32)
    idx, pi = _c(idx, np.int32)
    count, pc = _c(count, np.int32)
    rows, nu = scores.shape
    R = state.slot_unit.shape[1]
    ps = np.full((rows, max(C, 1)), -1, np.int32)
    pu, pe = ps.copy(), ps.copy()
    pcount = np.zeros(rows, np.int32)
    pool = np.full((rows, pool_stride), -1, np.int32)
    pool_count = np.zeros(rows, np.int32)
    for a in (state.slot_unit, state.slot_last, state.unit_slot):
        assert a.flags["C_CONTIGUOUS"]
    rc = _l().orc_delta_select(rows, nu, n_tokens, block, sink, local, psc, pi, idx.shape[-1], pc,
                               C, step, R, state.slot_unit.ctypes.data,
                               state.slot_last.ctypes.data, state.unit_slot.ctypes.data,
                               ps.ctypes.data, pu.ctypes.data, pe.ctypes.data,
                               pcount.ctypes.data, pool.ctypes.data, pool_stride,
                               pool_count.ctypes.data)
    if rc:
        raise ValueError("delta_select: bad block, R, C or step")
    return ps[:, :C], pu[:, :C], pe[:, :C], pcount, pool, pool_count


# ------------------------------------------------------------------------------------
# One sequence split by tokens across shards (HashAttention: Semantic Sparsity for
# Faster Inference, 2.5: contexts beyond one device; a sequence held by several
# devices needs one exchange of top-k candidates and one of attention partials).
# READING: shards are contiguous token ranges cut at multiples of 64 tokens (whole
# bit-plane scale blocks, so each shard's own index gives the unsharded scores);
# the forced windows stay with the shard holding them; the retrieval budget k is
# the sequence's, as unsharded.
# ------------------------------------------------------------------------------------
def shard_bounds(n: int, shards: int):
    """Token boundaries a_0 = 0 < ... < a_S = n of S contiguous shards cut at
    multiples of 64 tokens (64 * floor(nb * s / S), nb = ceil(n / 64))."""
    nb = (n + 63) // 64
    return [min(n, 64 * ((nb * s) // shards)) for s in range(shards + 1)]


def shard_windows(n: int, a: int, b: int, sink: int, local: int):
    """The forced windows of shard [a, b) in its own token indices: (sink_s, local_s),
    the parts of [0, lead) and [tail, n) it holds (lead = min(sink, n),
    tail = max(n - local, lead), as the unsharded top-k takes them)."""
    lead = min(sink, n)
    tail = max(n - local, lead)
    ns = b - a
    sink_s = min(max(lead - a, 0), ns)
    local_s = min(max(b - max(a, tail), 0), ns)
    return sink_s, local_s


def shard_candidates(scores_s, k: int, sink_s: int, local_s: int, a: int):
    """Shard-local top-k of the competing tokens [sink_s, n_s - local_s) of each row,
    in the order (score descending, index ascending): (score [rows][k] float64,
    global index [rows][k] int32 (-1 past the count), count [rows], -1 for a row
    holding a NaN)."""
    s = np.asarray(scores_s, np.float64)
    rows, ns = s.shape
    lo, hi = sink_s, max(ns - local_s, sink_s)
    sc = np.full((rows, k), -np.inf)
    ix = np.full((rows, k), -1, np.int32)
    cnt = np.zeros(rows, np.int32)
    for r in range(rows):
        seg = s[r, lo:hi]
        if np.isnan(seg).any():
            cnt[r] = -1
            continue
        order = sorted(range(len(seg)), key=lambda i: (-seg[i], i))[:k]
        cnt[r] = len(order)
        for t, i in enumerate(order):
            sc[r, t] = seg[i]
            ix[r, t] = a + lo + i
    return sc, ix, cnt


def topk_merge(cand_scores, cand_idx, cand_counts, k: int):
    """The sequence's top-k from every shard's candidates: the first k of their union
    in the order (score descending, global index ascending), written ascending.
    Returns (idx [rows][k] int32, -1 past the count; count [rows], -1 if any shard
    reported a NaN row)."""
    S = len(cand_scores)
    rows = cand_scores[0].shape[0]
    idx = np.full((rows, k), -1, np.int32)
    cnt = np.zeros(rows, np.int32)
    for r in range(rows):
        if any(int(cand_counts[s][r]) < 0 for s in range(S)):
            cnt[r] = -1
            continue
        pool = [(float(cand_scores[s][r, t]), int(cand_idx[s][r, t]))
                for s in range(S) for t in range(int(cand_counts[s][r]))]
        best = sorted(pool, key=lambda x: (-x[0], x[1]))[:k]
        sel = sorted(i for _, i in best)
        cnt[r] = len(sel)
        idx[r, :len(sel)] = sel
    return idx, cnt


def shard_select(sel_idx, sel_counts, a: int, b: int, sink_s: int, local_s: int):
    """Shard [a, b)'s attention set in its own token indices, ascending: its forced
    windows [0, sink_s) and [n_s - local_s, n_s) and the merged top-k's tokens in
    [a, b).  Returns (idx [rows][stride] int32, count [rows]); a NaN row (count -1)
    stays -1."""
    rows = sel_idx.shape[0]
    ns = b - a
    sets = []
    for r in range(rows):
        if sel_counts[r] < 0:
            sets.append(None)
            continue
        mine = [int(t) - a for t in sel_idx[r, :sel_counts[r]] if a <= t < b]
        forced = list(range(sink_s)) + list(range(ns - local_s, ns))
        sets.append(sorted(set(forced) | set(mine)))
    stride = max([1] + [len(x) for x in sets if x is not None])
    idx = np.full((rows, stride), -1, np.int32)
    cnt = np.zeros(rows, np.int32)
    for r, x in enumerate(sets):
        if x is None:
            cnt[r] = -1
            continue
        cnt[r] = len(x)
        idx[r, :len(x)] = x
    return idx, cnt


def attend_combine(outs, lses):
    """Split-softmax combine of per-shard attention over disjoint token sets: with
    L = log sum_s exp(lse_s), o = sum_s exp(lse_s - L) o_s and lse = L; shards with
    an empty set (lse = -inf) weigh 0; all empty gives o = 0, lse = -inf."""
    lse = np.stack([np.asarray(x, np.float64) for x in lses])          # [S][B][Hq]
    o = np.stack([np.asarray(x, np.float64) for x in outs])            # [S][B][Hq][d]
    m = lse.max(axis=0)
    fin = np.isfinite(m)
    w = np.where(fin[None], np.exp(np.where(np.isfinite(lse), lse - np.where(fin, m, 0)[None],
                                            -np.inf)), 0.0)
    tot = w.sum(axis=0)
    out = np.where(fin[..., None], (w[..., None] * o).sum(axis=0) /
                   np.where(tot > 0, tot, 1.0)[..., None], 0.0)
    L = np.where(fin, m + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    return out, L
