"""sd_topk_wmax (top-k drawn from the words whose 32-unit maximum reaches a sampled
threshold) against the oracle's top-k, index for index, on seeded score rows
built to take each of its paths: the sampled estimate, the cut words at the
sink and local windows, an estimate that leaves fewer than k candidates, word
and candidate lists that overflow, ties, NaN rows, and the calls it hands to
sd_topk.  The word maxima are the 32-unit maxima of the same rows (their
definition), and in the last test the ones sd_plan_score writes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import dev, empty, host

pytestmark = pytest.mark.gpu

SAMPLE = 2048  # sampled words per row (fewer if the row has fewer)


@pytest.fixture(scope="module")
def sd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_sparse_decode_gb300 import build as b
    b.build()
    import top_sparse_decode_gb300 as m
    m.lib()
    return m


def word_max(s: np.ndarray) -> np.ndarray:
    """Largest of each 32 consecutive scores; NaN if one of them is NaN."""
    rows, n = s.shape
    return s.reshape(rows, n // 32, 32).max(axis=2)  # numpy max propagates NaN


def run_wmax(sd, s, k, sink=0, local=0, wm=None):
    rows, n = s.shape
    sel = sd.make_select(k, sink, local, 1)
    stride = min(n, sink + local + k)
    idx = torch.full((rows, stride), -7, dtype=torch.int32, device="cuda")
    cnt = empty((rows,), np.int32)
    ws_bytes = sd.sd_topk_workspace_size(rows, n, sel)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if ws_bytes else None
    wm = word_max(s) if wm is None else wm
    sd.sd_topk_wmax(dev(s), dev(np.ascontiguousarray(wm, np.float32)), rows, n, sel, idx, stride,
                    cnt, ws)
    torch.cuda.synchronize()
    return host(idx, np.int32), host(cnt, np.int32)


def assert_oracle(sd, s, k, sink=0, local=0):
    gi, gc = run_wmax(sd, s, k, sink, local)
    ri, rc = oracle.topk(s, k, sink, local)
    for r in range(s.shape[0]):
        assert gc[r] == rc[r], (r, gc[r], rc[r])
        assert np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]]), r
    return gc


def sampled_words(W):
    S = min(W, SAMPLE)
    return (np.arange(S, dtype=np.int64) * W) // S


@pytest.mark.parametrize("rows,n,kind,levels,k,sink,local", [
    (8, 1048576, "f32", 0, 512, 0, 0),       # the 1M-token step's shape
    (3, 1048576 + 32, "f32", 0, 512, 4, 64),  # odd words per row; the sink cuts word 0
    (2, 262144, "f32", 0, 1024, 7, 33),      # both windows cut a word
    (2, 262144, "f32", 0, 1, 0, 0),
    (2, 131072, "f32", 0, 1000, 128, 128),
    (2, 262144, "f32ties", 7, 512, 0, 0),    # scores on 7 levels: ties everywhere
    (2, 262144, "f32ties", 256, 512, 0, 0),  # ties among the candidates only
    (2, 100000 - 100000 % 32, "f32ties", 3, 700, 5, 9),
    (2, 8192 + 32, "f32", 0, 512, 0, 0),     # just above the one-CTA row size of sd_topk
    (40, 65536, "f32", 0, 512, 3, 61),       # more rows than resident clusters: a CTA per row
    (48, 131072 + 96, "f32ties", 300, 256, 0, 33),
    (16, 262144, "f32", 0, 1024, 0, 0),
])
def test_topk_wmax_equals_oracle(sd, rows, n, kind, levels, k, sink, local):
    s = synth.make_scores(2000 + n % 977 + k, rows, n, kind, levels)
    assert_oracle(sd, s, k, sink, local)


def test_signed_zeros_and_infinities(sd):
    # -0.0 ranks with +0.0 (ties by unit); infinities are ordinary keys
    n = 65536
    s = np.zeros((2, n), np.float32)
    rng = np.random.default_rng(5)
    neg = rng.random(n) < 0.5
    s[0, neg] = -0.0
    s[1] = rng.standard_normal(n).astype(np.float32)
    s[1, rng.choice(n, 40, replace=False)] = np.inf
    s[1, rng.choice(n, 40, replace=False)] = -np.inf
    assert_oracle(sd, s, 256)
    assert_oracle(sd, s, 30, 3, 5)


def test_estimate_miss_takes_the_exact_path(sd):
    # one large score in each of 100 sampled words: the sample's r-th largest key is
    # one of them, and only ~r units of the row reach it (< k)
    n, k = 1048576, 512
    s = synth.make_scores(41, 2, n, "f32")
    W = n // 32
    hot = sampled_words(W)[::20][:100]
    s[0, hot * 32 + 5] = 100.0 + np.arange(100, dtype=np.float32)
    assert_oracle(sd, s, k)


def test_word_list_overflow_takes_the_exact_path(sd):
    # 8000 words share the row's largest value: every one of them reaches the
    # estimate, more than the candidate word list holds
    n = 1048576
    s = synth.make_scores(42, 1, n, "f32")
    W = n // 32
    words = np.random.default_rng(3).choice(W, 8000, replace=False)
    s[0, words * 32 + 17] = 50.0
    assert_oracle(sd, s, 512)


def test_candidate_overflow_takes_the_exact_path(sd):
    # 2000 words whose 32 units all hold the largest value: 64000 candidates
    n = 1048576
    s = synth.make_scores(43, 1, n, "f32")
    W = n // 32
    words = np.random.default_rng(4).choice(W, 2000, replace=False)
    s[0].reshape(W, 32)[words] = 50.0
    assert_oracle(sd, s, 1024)


def test_constant_rows(sd):
    # every key equal: the top k are the first k competing units
    n = 262144
    s = np.full((2, n), 0.5, np.float32)
    gc = assert_oracle(sd, s, 512, 3, 40)
    assert gc[0] == 3 + 512 + 40


def test_nan_rows(sd):
    n = 262144
    s = synth.make_scores(44, 4, n, "f32")
    s[0, 100000] = np.nan          # competing: the row is NaN
    s[1, 2] = np.nan               # inside the sink, in a word cut by it: not competing
    s[2, n - 1] = np.nan           # inside the local window, in a word cut by it
    s[3, 7] = np.nan               # competing unit of the cut word 0
    gi, gc = run_wmax(sd, s, 512, sink=3, local=5)
    ri, rc = oracle.topk(s, 512, 3, 5)
    assert list(gc) == list(rc) and gc[0] == -1 and gc[3] == -1 and gc[1] > 0 and gc[2] > 0
    for r in (1, 2):
        assert np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]])


def test_nan_in_every_share_of_a_row(sd):
    # a NaN in each sixteenth of a row in turn: whichever CTA holds it flags the row
    n = 1048576
    s = synth.make_scores(47, 16, n, "f32")
    for r in range(16):
        s[r, r * (n // 16) + 12345] = np.nan
    gi, gc = run_wmax(sd, s, 512)
    assert (gc == -1).all()


def test_nan_in_words_outside_the_windows_is_ignored(sd):
    # a NaN word maximum of a word lying entirely in the sink does not count
    n = 262144
    s = synth.make_scores(45, 1, n, "f32")
    s[0, 10] = np.nan
    gi, gc = run_wmax(sd, s, 512, sink=64, local=0)
    ri, rc = oracle.topk(s, 512, 64, 0)
    assert gc[0] == rc[0] > 0 and np.array_equal(gi[0, :gc[0]], ri[0, :rc[0]])


@pytest.mark.parametrize("n,k,sink,local", [(4096, 100, 0, 0),    # short rows: sd_topk
                                            (65536, 2048, 0, 0),  # k above the path's limit
                                            (65536, 512, 32000, 33100),  # at most k compete
                                            (65536, 512, 32000, 33000)])  # fewer words than k
def test_short_windows_and_handed_calls(sd, n, k, sink, local):
    s = synth.make_scores(46 + n + k, 2, n, "f32")
    assert_oracle(sd, s, k, sink, local)


def test_word_maxima_from_plan_score(sd):
    # the maxima the scan writes: bit-exact 32-unit maxima of its own scores, and
    # the top-k drawn from them equals sd_topk's on the same scores
    B, Hkv, G, n = 1, 8, 4, 262144
    cfg = synth.config(4, B=B, Hq=G * Hkv, Hkv=Hkv, n=n)
    inp = synth.make_inputs(cfg, with_v=False)
    shp = sd.make_shape(B, G * Hkv, Hkv, n, 128, n)
    planes = empty((B, Hkv, 128, 4, n // 32), np.uint32)
    scales = empty((B, Hkv, 128, n // 64), np.uint16)
    sd.sd_build_index(sd.SD_IDX_PLANES, shp, dev(inp.K), None, planes, scales)
    scores = empty((B * Hkv, n), np.float32)
    wm = empty((B * Hkv, n // 32), np.float32)
    sd.sd_plan_score(shp, planes, scales, dev(inp.q), dev(inp.sigma2), sd.SD_PLAN_WATERFILL, 56,
                     None, scores, wm)
    torch.cuda.synchronize()
    s = host(scores, np.float32)
    w = host(wm, np.float32)
    assert np.array_equal(w, word_max(s))
    gi, gc = run_wmax(sd, s, 512, 4, 64, wm=w)
    ri, rc = oracle.topk(s, 512, 4, 64)
    for r in range(B * Hkv):
        assert gc[r] == rc[r] and np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]]), r
