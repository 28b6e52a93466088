"""sd_plan_score (the read plan computed inside the bit-plane scan) against sd_plan
followed by sd_score on the same inputs: the plan and the scores must be
identical bit for bit, for every plan mode, budget edge and group size."""
import numpy as np
import pytest
import torch

import synth
from _helpers import dev, empty, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_sparse_decode_gb300 import build as b
    b.build()
    import top_sparse_decode_gb300 as m
    m.lib()
    return m


CASES = [  # (G, Hkv, B, n, ncap, mode, budget)
    (4, 4, 1, 65536, 0, 0, 56), (4, 4, 1, 65536, 0, 0, 0), (4, 4, 1, 65536, 0, 0, 512),
    (4, 4, 1, 65536, 0, 0, 47), (8, 2, 2, 8192 + 192, 8704, 0, 92), (1, 8, 1, 4096, 0, 0, 300),
    (4, 4, 1, 65536, 0, 1, 32), (4, 4, 1, 65536, 0, 1, 0), (4, 4, 1, 65536, 0, 1, 128),
    (2, 4, 2, 16384, 0, 2, 0), (4, 8, 1, 262144, 0, 0, 56),
    (4, 4, 1, 65536, 0, 3, 17), (1, 8, 1, 4096, 0, 3, 128), (8, 2, 2, 8192 + 192, 8704, 3, 5),
    (4, 8, 1, 262144, 0, 3, 0),
]


@pytest.mark.parametrize("G,Hkv,B,n,ncap,mode,budget", CASES)
def test_plan_score_equals_plan_then_score(sd, G, Hkv, B, n, ncap, mode, budget):
    ncap = ncap or n
    cfg = synth.config(4, B=B, Hq=G * Hkv, Hkv=Hkv, n=n)
    inp = synth.make_inputs(cfg, with_v=False)
    shp = sd.make_shape(B, G * Hkv, Hkv, n, 128, ncap)
    Kp = np.zeros((B, Hkv, ncap, 128), np.uint16)
    Kp[:, :, :n] = inp.K
    planes = empty((B, Hkv, 128, 4, ncap // 32), np.uint32)
    scales = empty((B, Hkv, 128, ncap // 64), np.uint16)
    sd.sd_build_index(sd.SD_IDX_PLANES, shp, dev(Kp), None, planes, scales)
    q = dev(inp.q)
    s2 = None if mode == sd.SD_PLAN_TOPQ else dev(inp.sigma2)  # top-q reads no variances
    plan1 = empty((B, Hkv, 128), np.uint8)
    sd.sd_plan(shp, q, s2, mode, budget, plan1)
    s1 = empty((B * Hkv, n), np.float32)
    sd.sd_score(sd.SD_IDX_PLANES, shp, planes, scales, q, plan1, s1)
    plan2 = torch.full((B, Hkv, 128), 77, dtype=torch.uint8, device="cuda")
    s2o = empty((B * Hkv, n), np.float32)
    sd.sd_plan_score(shp, planes, scales, q, s2, mode, budget, plan2, s2o)
    s3 = empty((B * Hkv, n), np.float32)
    sd.sd_plan_score(shp, planes, scales, q, s2, mode, budget, None, s3)  # no plan output
    torch.cuda.synchronize()
    assert np.array_equal(host(plan1, np.uint8), host(plan2, np.uint8))
    assert np.array_equal(host(s1, np.uint32), host(s2o, np.uint32))
    assert np.array_equal(host(s1, np.uint32), host(s3, np.uint32))


def test_plan_score_against_oracle_262k(sd):
    """sd_plan_score against the oracle itself (plan bit-exact, scores within 1e-5 of
    their L1 mass), 8 KV heads x 262,144 tokens at 56 bits."""
    import oracle
    from _helpers import check_scores
    B, Hkv, G, n = 1, 8, 4, 262144
    cfg = synth.config(4, B=B, Hq=G * Hkv, Hkv=Hkv, n=n)
    inp = synth.make_inputs(cfg, with_v=False)
    shp = sd.make_shape(B, G * Hkv, Hkv, n)
    planes = empty((B, Hkv, 128, 4, n // 32), np.uint32)
    scales = empty((B, Hkv, 128, n // 64), np.uint16)
    sd.sd_build_index(sd.SD_IDX_PLANES, shp, dev(inp.K), None, planes, scales)
    plan = empty((B, Hkv, 128), np.uint8)
    scores = empty((B * Hkv, n), np.float32)
    sd.sd_plan_score(shp, planes, scales, dev(inp.q), dev(inp.sigma2), sd.SD_PLAN_WATERFILL, 56,
                     plan, scores)
    torch.cuda.synchronize()
    rp, rs = oracle.plane_build(inp.K)
    rplan = oracle.plan(inp.q, inp.sigma2, Hkv, 0, 56)
    assert np.array_equal(host(plan, np.uint8), rplan)
    ref, l1 = oracle.plane_score(rp, rs, rplan, inp.q, with_l1=True)
    check_scores(host(scores, np.float32), ref.reshape(B * Hkv, n), l1.reshape(B * Hkv, n),
                 "sd_plan_score vs oracle")
