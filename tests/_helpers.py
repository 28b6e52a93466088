"""Helpers shared by the GPU parity tests: numpy <-> torch device transfers and
the tolerance contract.

Tolerances (exactly as the parity contract states them):
  * signatures, planes, scales, plans, Hamming scores and Hamming index sets:
    bit-exact;
  * float scores: |s_gpu - s_ref| <= 1e-5 * (sum of |terms| of that score);
  * float index sets: size k, every candidate with s_ref > tau + tol inside,
    none with s_ref < tau - tol (tau = the oracle's k-th score);
  * attention outputs: max |o_gpu - o_ref| <= 2e-3 against the float64 oracle.
"""
import numpy as np
import torch

SCORE_RTOL = 1e-5
ATT_ATOL = 2e-3

_VIEW = {np.dtype(np.uint16): torch.int16, np.dtype(np.uint32): torch.int32,
         np.dtype(np.uint8): torch.uint8, np.dtype(np.float32): torch.float32,
         np.dtype(np.int32): torch.int32, np.dtype(np.int64): torch.int64}
_BACK = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32}


def dev(x: np.ndarray) -> torch.Tensor:
    x = np.ascontiguousarray(x)
    src = x.view(_BACK.get(x.dtype, x.dtype))
    return torch.from_numpy(src).to("cuda")


def host(t: torch.Tensor, dtype) -> np.ndarray:
    a = t.detach().cpu().contiguous().numpy()
    return a.view(dtype)


def empty(shape, dtype) -> torch.Tensor:
    tdt = _VIEW[np.dtype(dtype)]
    return torch.empty(shape, dtype=tdt, device="cuda")


def check_scores(gpu: np.ndarray, ref: np.ndarray, l1: np.ndarray, what: str) -> float:
    err = np.abs(gpu.astype(np.float64) - ref)
    bound = SCORE_RTOL * l1
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} scores outside 1e-5*L1; worst excess "
                           f"{(err - bound).max():.3e}")
    return float((err / np.maximum(l1, 1e-300)).max())


def check_float_topk(idx_gpu, cnt_gpu, idx_ref, cnt_ref, ref_scores, l1, k, sink, local,
                     block=1, n_tokens=None):
    """Float-score index sets under the contract.  Rows are [rows][...]; scores
    [rows][n_units] (double).  Returns how many rows differ from the oracle's
    set (all within tolerance)."""
    rows, n_units = ref_scores.shape
    if n_tokens is None:
        n_tokens = n_units * block
    differ = 0
    for r in range(rows):
        assert cnt_gpu[r] == cnt_ref[r], (r, cnt_gpu[r], cnt_ref[r])
        g = idx_gpu[r, :cnt_gpu[r]]
        o = idx_ref[r, :cnt_ref[r]]
        assert np.all(np.diff(g) > 0), "output not ascending"
        if np.array_equal(g, o):
            continue
        differ += 1
        gu = np.unique(g // block)
        lead = min(sink, n_units)
        tail = max(n_units - local, lead)
        forced = set(range(lead)) | set(range(tail, n_units))
        assert forced <= set(gu.tolist())
        cand_g = np.array(sorted(set(gu.tolist()) - forced))
        assert len(cand_g) == min(k, tail - lead)
        s = ref_scores[r, lead:tail]
        tol = SCORE_RTOL * l1[r, lead:tail]
        tau = np.sort(s)[::-1][k - 1]
        must = np.nonzero(s > tau + tol)[0] + lead
        never = np.nonzero(s < tau - tol)[0] + lead
        assert set(must.tolist()) <= set(cand_g.tolist()), "a clear winner is missing"
        assert not (set(never.tolist()) & set(cand_g.tolist())), "a clear loser is selected"
    return differ
