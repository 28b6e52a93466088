"""The sequence-shard kernels (HashAttention 2.5, contexts beyond one device) on one
GPU: candidates, merge, shard set and combine against the oracle's definitions, and
whole 2- and 3-shard steps run from one process (the exchanges are stacks of the
shards' tensors) against the unsharded GPU step (identical selection, scores being
identical per token) and the unsharded oracle step."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import ATT_ATOL, check_float_topk, dev, empty, host

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


@pytest.mark.parametrize("S,k", [(2, 64), (3, 512), (16, 512)])
def test_topk_merge_and_candidates(sd, S, k):
    rows, ns = 5, 3000
    sc_all, ix_all, cn_all = [], [], []
    gs, gi, gc = [], [], []
    for s in range(S):
        scores = synth.make_scores(40 + s, rows, ns, "f32ties", levels=6)
        sink_s, local_s = (3 if s == 0 else 0), (9 if s == S - 1 else 0)
        ri, rc = oracle.topk(scores, k, sink_s, local_s)
        if s == 1:
            rc[2] = -1  # a NaN row reported by one shard
        rsc, rix, rcn = oracle.shard_candidates(scores.astype(np.float64), k, sink_s, local_s,
                                                s * ns)
        rcn[2] = -1 if s == 1 else rcn[2]
        sc_all.append(rsc.astype(np.float32)); ix_all.append(rix); cn_all.append(rcn)
        cs, ci, cc = empty((rows, k), np.float32), empty((rows, k), np.int32), empty((rows,), np.int32)
        sd.sd_shard_candidates(dev(scores), rows, ns, dev(ri), ri.shape[1], dev(rc), sink_s,
                               local_s, s * ns, k, cs, ci, cc)
        torch.cuda.synchronize()
        g_cc = host(cc, np.int32)
        assert np.array_equal(g_cc, rcn)
        for r in range(rows):
            if rcn[r] > 0:  # same entries, in the top-k's (ascending) order
                assert sorted(host(ci, np.int32)[r, :rcn[r]].tolist()) == sorted(rix[r, :rcn[r]].tolist())
        gs.append(cs); gi.append(ci); gc.append(cc)
    mi, mc = oracle.topk_merge(sc_all, ix_all, cn_all, k)
    out, cnt = empty((rows, k), np.int32), empty((rows,), np.int32)
    sd.sd_topk_merge(rows, S, k, torch.stack(gs), torch.stack(gi), torch.stack(gc), out, k, cnt)
    torch.cuda.synchronize()
    assert np.array_equal(host(cnt, np.int32), mc)
    for r in range(rows):
        if mc[r] > 0:
            assert np.array_equal(host(out, np.int32)[r, :mc[r]], mi[r, :mc[r]]), r


def test_shard_select_and_combine(sd):
    rows, k = 3, 40
    a, ns, sink_s, local_s = 2500, 5000, 2, 6
    raw, rcnt = synth.make_index_lists(5, rows, 10000, k, np.array([40, 0, 17]))
    forced = set(range(a, a + sink_s)) | set(range(a + ns - local_s, a + ns))
    sel = np.full((rows, k), -1, np.int32)  # the merge never holds a forced token
    cnt = np.zeros(rows, np.int32)
    for r in range(rows):
        keep = [t for t in raw[r, :rcnt[r]].tolist() if t not in forced]
        sel[r, :len(keep)] = keep
        cnt[r] = len(keep)
    ri, rc = oracle.shard_select(sel, cnt, a, a + ns, sink_s, local_s)
    o_idx, o_cnt = empty((rows, sink_s + local_s + k), np.int32), empty((rows,), np.int32)
    sd.sd_shard_select(rows, dev(sel), sel.shape[1], dev(cnt), a, ns, sink_s, local_s, k, o_idx,
                       sink_s + local_s + k, o_cnt)
    torch.cuda.synchronize()
    assert np.array_equal(host(o_cnt, np.int32), rc)
    for r in range(rows):
        assert np.array_equal(host(o_idx, np.int32)[r, :rc[r]], ri[r, :rc[r]])
    # combine: three shards, one of them empty for some heads
    S, B, Hq = 3, 2, 8
    outs = synth.normal(9, 1, S * B * Hq * 128).reshape(S, B, Hq, 128).astype(np.float32)
    lses = (synth.normal(9, 2, S * B * Hq) * 3).reshape(S, B, Hq).astype(np.float32)
    lses[1, 0, :3] = -np.inf
    lses[:, 1, 5] = -np.inf
    ro, rl = oracle.attend_combine(outs, lses)
    go, gl = empty((B, Hq, 128), np.float32), empty((B, Hq), np.float32)
    sd.sd_attend_combine(S, B, Hq, dev(outs), dev(lses), go, gl)
    torch.cuda.synchronize()
    assert np.abs(host(go, np.float32) - ro).max() < 1e-5
    g = host(gl, np.float32)
    assert np.array_equal(np.isinf(g), np.isinf(rl)) and np.abs(g[np.isfinite(g)] - rl[np.isfinite(rl)]).max() < 1e-5


def padded(x, ncap):
    out = np.zeros(x.shape[:2] + (ncap,) + x.shape[3:], x.dtype)
    out[:, :, :x.shape[2]] = x
    return out


@pytest.mark.parametrize("S,n,k,sink,local", [(2, 131072, 512, 0, 0), (3, 64 * 1000 + 33, 300, 7, 65),
                                              (2, 40000, 1000, 128, 512)])
def test_sharded_step_equals_unsharded(sd, S, n, k, sink, local):
    from top_sparse_decode_gb300.pipeline import DecodeStep, StepConfig, build_index
    from top_sparse_decode_gb300.shard import ShardStep, run_shards_locally, shard_bounds
    cfg = synth.config(2, B=2, Hq=8, Hkv=2, n=n, k=k, sink=sink, local=local)
    inp = synth.make_inputs(cfg)
    q, s2 = dev(inp.q), dev(inp.sigma2)
    full_cap = -(-n // 512) * 512
    scf = StepConfig(sd.SD_IDX_PLANES, cfg.B, cfg.Hq, cfg.Hkv, n, k=k, sink=sink, local=local,
                     n_cap=full_cap)
    Kf, Vf = dev(padded(inp.K, full_cap)), dev(padded(inp.V, full_cap))
    full = DecodeStep(scf, Kf, Vf, build_index(scf, Kf), sigma2=s2)
    full.run(q)
    cut = shard_bounds(n, S)
    steps = []
    for s in range(S):
        a, b = cut[s], cut[s + 1]
        cap = -(-(b - a) // 512) * 512
        Ks = dev(padded(np.ascontiguousarray(inp.K[:, :, a:b]), cap))
        Vs = dev(padded(np.ascontiguousarray(inp.V[:, :, a:b]), cap))
        lc = StepConfig(sd.SD_IDX_PLANES, cfg.B, cfg.Hq, cfg.Hkv, b - a, n_cap=cap)
        steps.append(ShardStep(scf, s, S, Ks, Vs, build_index(lc, Ks), s2, n_cap_s=cap))
    res = run_shards_locally(steps, q)
    torch.cuda.synchronize()
    rows = cfg.B * cfg.Hkv
    # every shard holds the same merged set; it is the unsharded GPU step's competing part
    lead, tail = min(sink, n), max(n - local, min(sink, n))
    fi, fc = host(full.idx, np.int32), host(full.count, np.int32)
    for st in steps:
        mi, mc = host(st.sel_idx, np.int32), host(st.sel_count, np.int32)
        for r in range(rows):
            want = [t for t in fi[r, :fc[r]].tolist() if lead <= t < tail]
            assert mi[r, :mc[r]].tolist() == want, (st.shard, r)
    go = host(res[0][0], np.float32)
    assert np.abs(go - host(full.out, np.float32)).max() < 1e-4
    for o, _ in res[1:]:
        assert np.array_equal(host(o, np.float32), go)
    # and the oracle: unsharded scores, top-k within the score tolerance, attention
    p, sc = oracle.plane_build(inp.K)
    plan = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, 0, 56)
    ref, l1 = oracle.plane_score(p, sc, plan, inp.q, with_l1=True, n=n)
    ri, rc = oracle.topk(ref.reshape(rows, n), k, sink, local)
    check_float_topk(fi, fc, ri, rc, ref.reshape(rows, n), l1.reshape(rows, n), k, sink, local)
    ro, _ = oracle.gather_attend(inp.q, inp.K, inp.V, fi.reshape(cfg.B, cfg.Hkv, -1),
                                 fc.reshape(cfg.B, cfg.Hkv), 1 / math.sqrt(cfg.d))
    assert np.abs(go - ro).max() <= ATT_ATOL
