"""The bit-plane step at any n (HashAttention 2.2: signatures -- and here every key
index -- are written as keys arrive; OasisKV method details: compressed-key
update): the scans read a partial last 64-token block, the word-maxima top-k takes
a partial last word, and a decode loop that appends one key per step runs the full
bit-plane step after every append, each checked against the oracle on the oracle's
own index of the first n keys."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import ATT_ATOL, check_float_topk, check_scores, dev, empty, host

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


def padded(x, ncap):
    """K-like [B][H][n][d] -> [B][H][ncap][d], zeros past n (capacity, not keys)."""
    out = np.zeros(x.shape[:2] + (ncap,) + x.shape[3:], x.dtype)
    out[:, :, :x.shape[2]] = x
    return out


@pytest.mark.parametrize("n,ncap", [(4096 + 1, 4608), (4096 + 33, 4608), (64 * 37 + 17, 2560),
                                    (5, 512), (64 * 37 + 17, 64 * 38), (1000, 1024 + 64)])
def test_plan_score_any_n(sd, n, ncap):
    # ncap % 512 == 0: the bulk-copy scan; otherwise the direct-streaming scan
    cfg = synth.config(2, B=2, Hq=8, Hkv=2, n=n)
    inp = synth.make_inputs(cfg, with_v=False)
    shp = sd.make_shape(cfg.B, cfg.Hq, cfg.Hkv, n, n_cap=ncap)
    planes = empty((cfg.B, cfg.Hkv, 128, 4, ncap // 32), np.uint32)
    scales = empty((cfg.B, cfg.Hkv, 128, ncap // 64), np.uint16)
    sd.sd_build_index(sd.SD_IDX_PLANES, shp, dev(padded(inp.K, ncap)), None, planes, scales)
    q = dev(inp.q)
    plan = empty((cfg.B, cfg.Hkv, 128), np.uint8)
    scores = empty((cfg.B * cfg.Hkv, n), np.float32)
    wmax = empty((cfg.B * cfg.Hkv, (n + 31) // 32), np.float32)
    sd.sd_plan_score(shp, planes, scales, q, dev(inp.sigma2), sd.SD_PLAN_WATERFILL, 56, plan,
                     scores, wmax)
    torch.cuda.synchronize()
    rp, rs = oracle.plane_build(inp.K)
    rplan = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, 0, 56)
    assert np.array_equal(host(plan, np.uint8), rplan)
    ref, l1 = oracle.plane_score(rp, rs, rplan, inp.q, with_l1=True, n=n)
    got = host(scores, np.float32).reshape(ref.shape)
    check_scores(got, ref, l1, "any-n plane scores")
    # word maxima over the tokens < n, the last word partial
    rows = got.reshape(cfg.B * cfg.Hkv, n)
    pad = np.full((rows.shape[0], ((n + 31) // 32) * 32), -np.inf, np.float32)
    pad[:, :n] = rows
    assert np.array_equal(host(wmax, np.float32), pad.reshape(rows.shape[0], -1, 32).max(axis=2))


def test_plan_score_any_n_block_per_lane(sd):
    # 8 KV heads x 655,377 tokens: every CTA's range exceeds one 16K-token tile, so
    # the scan's compute lanes own whole 64-token blocks; the last block is partial
    n = 655360 + 17
    ncap = 655360 + 512
    cfg = synth.config(2, B=1, Hq=32, Hkv=8, n=n)
    inp = synth.make_inputs(cfg, with_v=False)
    shp = sd.make_shape(1, 32, 8, n, n_cap=ncap)
    planes = empty((1, 8, 128, 4, ncap // 32), np.uint32)
    scales = empty((1, 8, 128, ncap // 64), np.uint16)
    sd.sd_build_index(sd.SD_IDX_PLANES, shp, dev(padded(inp.K, ncap)), None, planes, scales)
    plan = empty((1, 8, 128), np.uint8)
    scores = empty((8, n), np.float32)
    wmax = empty((8, (n + 31) // 32), np.float32)
    sd.sd_plan_score(shp, planes, scales, dev(inp.q), dev(inp.sigma2), sd.SD_PLAN_WATERFILL, 56,
                     plan, scores, wmax)
    torch.cuda.synchronize()
    rp, rs = oracle.plane_build(inp.K)
    rplan = oracle.plan(inp.q, inp.sigma2, 8, 0, 56)
    assert np.array_equal(host(plan, np.uint8), rplan)
    ref, l1 = oracle.plane_score(rp, rs, rplan, inp.q, with_l1=True, n=n)
    got = host(scores, np.float32)
    check_scores(got, ref.reshape(8, n), l1.reshape(8, n), "any-n plane scores (block per lane)")
    pad = np.full((8, ((n + 31) // 32) * 32), -np.inf, np.float32)
    pad[:, :n] = got
    assert np.array_equal(host(wmax, np.float32), pad.reshape(8, -1, 32).max(axis=2))


@pytest.mark.parametrize("n,k,sink,local", [(20000 + 7, 512, 0, 0), (65536 + 1, 512, 0, 0),
                                            (40000 + 19, 300, 5, 100)])
def test_topk_wmax_any_n(sd, n, k, sink, local):
    rows = 4
    s = synth.make_scores(91, rows, n, "f32")
    pad = np.full((rows, ((n + 31) // 32) * 32), -np.inf, np.float32)
    pad[:, :n] = s
    wm = pad.reshape(rows, -1, 32).max(axis=2)
    sel = sd.make_select(k, sink, local, 1)
    stride = sink + local + k
    idx = empty((rows, stride), np.int32)
    cnt = empty((rows,), np.int32)
    ws_n = sd.sd_topk_workspace_size(rows, n, sel)
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device="cuda")
    sd.sd_topk_wmax(dev(s), dev(wm), rows, n, sel, idx, stride, cnt, ws)
    torch.cuda.synchronize()
    ri, rc = oracle.topk(s, k, sink, local)
    gi, gc = host(idx, np.int32), host(cnt, np.int32)
    assert np.array_equal(gc, rc)
    for r in range(rows):
        assert np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]]), r


def test_decode_loop_of_appends(sd):
    """64 consecutive one-token appends from n = 65,536: after each, the bit-plane
    step (plan in the scan, word-maxima top-k, gather-attend) on n keys equals the
    oracle's step on its own index of those n keys."""
    from top_sparse_decode_gb300.pipeline import DecodeStep, StepConfig
    n0, steps, ncap = 65536, 64, 65536 + 512
    cfg = synth.config(2, B=1, Hq=8, Hkv=2, n=n0 + steps)
    inp = synth.make_inputs(cfg)
    K, V = dev(padded(inp.K, ncap)), dev(padded(inp.V, ncap))
    q, s2 = dev(inp.q), dev(inp.sigma2)
    planes = empty((1, cfg.Hkv, 128, 4, ncap // 32), np.uint32)
    scales = empty((1, cfg.Hkv, 128, ncap // 64), np.uint16)
    sd.sd_build_index(sd.SD_IDX_PLANES, sd.make_shape(1, cfg.Hq, cfg.Hkv, n0, n_cap=ncap), K,
                      None, planes, scales)
    scale = 1 / math.sqrt(cfg.d)
    differ = 0
    for n in range(n0 + 1, n0 + steps + 1):
        shp = sd.make_shape(1, cfg.Hq, cfg.Hkv, n, n_cap=ncap)
        sd.sd_append_index(sd.SD_IDX_PLANES, shp, n - 1, K, None, planes, scales)
        sc = StepConfig(sd.SD_IDX_PLANES, 1, cfg.Hq, cfg.Hkv, n, k=cfg.k, n_cap=ncap)
        step = DecodeStep(sc, K, V, {"planes": planes, "scales": scales}, sigma2=s2)
        step.run(q)
        torch.cuda.synchronize()
        Kn = np.ascontiguousarray(inp.K[:, :, :n])
        rp, rs = oracle.plane_build(Kn)
        rplan = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, 0, 56)
        ref, l1 = oracle.plane_score(rp, rs, rplan, inp.q, with_l1=True, n=n)
        rows = cfg.Hkv
        check_scores(host(step.scores, np.float32), ref.reshape(rows, n), l1.reshape(rows, n),
                     f"scores at n={n}")
        ri, rc = oracle.topk(ref.reshape(rows, n), cfg.k)
        gi, gc = host(step.idx, np.int32), host(step.count, np.int32)
        differ += check_float_topk(gi, gc, ri, rc, ref.reshape(rows, n), l1.reshape(rows, n),
                                   cfg.k, 0, 0)
        ro, _ = oracle.gather_attend(inp.q, Kn, np.ascontiguousarray(inp.V[:, :, :n]),
                                     gi.reshape(1, rows, -1), gc.reshape(1, rows), scale)
        err = np.abs(host(step.out, np.float32) - ro).max()
        assert err <= ATT_ATOL, (n, err)
    assert differ <= steps * rows // 8
