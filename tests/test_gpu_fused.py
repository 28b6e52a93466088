"""sd_score_topk (bit-plane scan and top-k in one call) against sd_score followed by
sd_topk on the same inputs: the scores, index sets and counts must be identical,
on the fused path (a sampled threshold, candidates appended by the scan) and on
every way out of it -- an estimate that leaves fewer than k candidates, a list
that overflows, a NaN row, rows too short for the sample, a k too large for it."""
import numpy as np
import pytest
import torch

import synth
from _helpers import dev, empty, host

pytestmark = pytest.mark.gpu

SAMPLE_RUNS = 512  # runs of 32 tokens the threshold sample scores per row


@pytest.fixture(scope="module")
def sd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_sparse_decode_gb300 import build as b
    b.build()
    import top_sparse_decode_gb300 as m
    m.lib()
    return m


def sampled_words(n, sink, local):
    """Word indices the threshold sample reads (the runs' evenly spaced positions)."""
    lead, tail = min(sink, n), max(n - local, min(sink, n))
    w0, w1 = lead // 32, (tail + 31) // 32
    return np.array([w0 + ((2 * g + 1) * (w1 - w0)) // (2 * SAMPLE_RUNS) for g in range(SAMPLE_RUNS)])


def both(sd, K, q, sigma2, B, Hq, Hkv, n, k, sink=0, local=0, budget=56, ncap=0):
    """Runs the two-call path and the fused call on the same index; returns both."""
    ncap = ncap or n
    shp = sd.make_shape(B, Hq, Hkv, n, 128, ncap)
    Kp = np.zeros((B, Hkv, ncap, 128), np.uint16)
    Kp[:, :, :n] = K
    planes = empty((B, Hkv, 128, 4, ncap // 32), np.uint32)
    scales = empty((B, Hkv, 128, ncap // 64), np.uint16)
    sd.sd_build_index(sd.SD_IDX_PLANES, shp, dev(Kp), None, planes, scales)
    qd = dev(q)
    plan = empty((B, Hkv, 128), np.uint8)
    sd.sd_plan(shp, qd, dev(sigma2), sd.SD_PLAN_WATERFILL, budget, plan)
    sel = sd.make_select(k, sink, local)
    rows = B * Hkv
    stride = min(n, sink + local + k)
    # two calls
    s1 = empty((rows, n), np.float32)
    sd.sd_score(sd.SD_IDX_PLANES, shp, planes, scales, qd, plan, s1)
    i1 = torch.full((rows, stride), -7, dtype=torch.int32, device="cuda")
    c1 = empty((rows,), np.int32)
    ws1 = torch.empty(max(1, sd.sd_topk_workspace_size(rows, n, sel)), dtype=torch.uint8,
                      device="cuda")
    sd.sd_topk(sd.SD_SCORE_F32, s1, rows, n, n, sel, i1, stride, c1, ws1)
    # one call
    s2 = empty((rows, n), np.float32)
    i2 = torch.full((rows, stride), -7, dtype=torch.int32, device="cuda")
    c2 = empty((rows,), np.int32)
    ws2 = torch.empty(max(1, sd.sd_score_topk_workspace_size(shp, sel)), dtype=torch.uint8,
                      device="cuda")
    sd.sd_score_topk(shp, planes, scales, qd, plan, sel, s2, i2, stride, c2, ws2)
    torch.cuda.synchronize()
    return (host(s1, np.uint32), host(i1, np.int32), host(c1, np.int32),
            host(s2, np.uint32), host(i2, np.int32), host(c2, np.int32))


def assert_same(r):
    s1, i1, c1, s2, i2, c2 = r
    assert np.array_equal(s1, s2), "scores differ (bit patterns)"
    assert np.array_equal(c1, c2), (c1, c2)
    for row in range(len(c1)):
        if c1[row] > 0:
            assert np.array_equal(i1[row, :c1[row]], i2[row, :c2[row]]), row


def seeded(B, Hq, Hkv, n, cid=4):
    """Seeded keys, queries and calibration (the seed follows the config id)."""
    cfg = synth.config(cid, B=B, Hq=Hq, Hkv=Hkv, n=n)
    inp = synth.make_inputs(cfg, with_v=False)
    return inp.K, inp.q, inp.sigma2


# (a ragged n with n_cap a multiple of 512 stays on the fused path; 20 rows take
# smaller clusters than 8)
@pytest.mark.parametrize("B,Hkv,n,ncap,k,sink,local", [(1, 8, 262144, 0, 512, 4, 64),
                                                       (2, 4, 131072, 0, 256, 0, 0),
                                                       (1, 2, 262144 + 192, 262656, 1000, 7, 33),
                                                       (1, 20, 131072, 0, 512, 16, 128)])
def test_fused_equals_two_calls(sd, B, Hkv, n, ncap, k, sink, local):
    K, q, s2 = seeded(B, 4 * Hkv, Hkv, n)
    assert_same(both(sd, K, q, s2, B, 4 * Hkv, Hkv, n, k, sink, local, ncap=ncap))


@pytest.mark.parametrize("n,k,ncap", [(16384, 512, 0),        # too short for the sample
                                      (262144, 4096, 0),      # k too large for the list
                                      (131072, 512, 131072 + 64)])  # n_cap not a multiple of 512
def test_paths_outside_the_fused_one(sd, n, k, ncap):
    K, q, s2 = seeded(1, 16, 4, n)
    assert_same(both(sd, K, q, s2, 1, 16, 4, n, k, ncap=ncap))


def hot_keys(K, q, Hkv, G, rows_hot, tokens, spread=0.1):
    """Keys of `tokens` replaced by the group-summed query direction, scaled so they
    score about 20 standard deviations above the seeded keys (times 1 + spread *
    u, u uniform per token: spread 0 gives them all one key)."""
    K = K.copy()
    qf = (q.astype(np.uint32) << 16).view(np.float32).reshape(q.shape[0], Hkv, G, 128).sum(2)
    rng = np.random.default_rng(11)
    for h in rows_hot:
        d = qf[0, h] / np.linalg.norm(qf[0, h])
        v = (30.0 * (1.0 + spread * rng.random((len(tokens), 1)))) * d[None, :]
        K[0, h, tokens] = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return K


def test_estimate_miss_falls_back(sd):
    # hot tokens only inside the sampled runs (4 per run): the sample's threshold
    # lands among them, and the row holds far fewer than k tokens above it
    n, Hkv, G = 262144, 4, 4
    K, q, s2 = seeded(1, G * Hkv, Hkv, n, cid=1)
    w = sampled_words(n, 0, 0)
    tokens = (w[:, None] * 32 + np.arange(4)[None, :]).ravel()
    K = hot_keys(K, q, Hkv, G, [0, 2], tokens)
    assert_same(both(sd, K, q, s2, 1, G * Hkv, Hkv, n, 512))


def test_overflowing_list_falls_back(sd):
    # every key of two rows equal: all their scores tie at the threshold, so every
    # token is a candidate -- far more than the list holds
    n, Hkv, G = 262144, 4, 4
    K, q, s2 = seeded(1, G * Hkv, Hkv, n, cid=2)
    K = hot_keys(K, q, Hkv, G, [1, 3], np.arange(n), spread=0.0)
    assert_same(both(sd, K, q, s2, 1, G * Hkv, Hkv, n, 512))


def test_nan_row(sd):
    n, Hkv, G = 131072, 4, 4
    K, q, s2 = seeded(1, G * Hkv, Hkv, n, cid=0)
    q = q.copy()
    q[0, 2 * G + 1, 5] = 0x7FC0  # a NaN in one query head of KV head 2
    r = both(sd, K, q, s2, 1, G * Hkv, Hkv, n, 512)
    assert r[2][2] == -1 and r[5][2] == -1
    assert_same(r)


def test_fused_against_oracle_262k(sd):
    """sd_score_topk against the oracle itself: scores within 1e-5 of their L1 mass,
    index sets equal up to swaps inside that tolerance, at 8 KV heads x 262,144."""
    import oracle
    from _helpers import check_float_topk, check_scores
    B, Hkv, n, k, sink, local = 1, 8, 262144, 512, 4, 64
    K, q, s2 = seeded(B, 4 * Hkv, Hkv, n)
    s1, i1, c1, sf, i2, c2 = both(sd, K, q, s2, B, 4 * Hkv, Hkv, n, k, sink, local)
    rp, rs = oracle.plane_build(K)
    rplan = oracle.plan(q, s2, Hkv, 0, 56)
    ref, l1 = oracle.plane_score(rp, rs, rplan, q, with_l1=True)
    ref, l1 = ref.reshape(B * Hkv, n), l1.reshape(B * Hkv, n)
    check_scores(sf.view(np.float32), ref, l1, "sd_score_topk scores vs oracle")
    ri, rc = oracle.topk(ref, k, sink, local, 1, n)
    check_float_topk(i2, c2, ri, rc, ref, l1, k, sink, local, 1, n)
