"""End-to-end parity of one decode step (index build on the KV-write path, then
query map / plan -> score -> top-k -> gather-attend) against the CPU oracle run
on the same seeded inputs, for every workload configuration at full size, in
the launch configuration the benchmark times (pipeline.DecodeStep)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import ATT_ATOL, check_float_topk, check_scores, dev, host

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


def step_config(sd, cfg, kind, plan_mode=0, budget=56):
    from top_sparse_decode_gb300.pipeline import StepConfig
    if kind == sd.SD_IDX_MINMAX:
        return StepConfig(kind, cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.d, k=cfg.blk_k, sink=0,
                          local=cfg.blk_local)
    if kind == sd.SD_IDX_LANDMARK:  # the token budget and windows in 8-token blocks
        return StepConfig(kind, cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.d, k=max(1, cfg.k // 8),
                          sink=(cfg.sink + 7) // 8, local=(cfg.local + 7) // 8)
    # bit planes need a capacity that is a multiple of 64: a ragged n gets a padded one
    ncap = 0 if kind != sd.SD_IDX_PLANES or cfg.n % 64 == 0 else -(-cfg.n // 512) * 512
    return StepConfig(kind, cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.d, k=cfg.k, sink=cfg.sink,
                      local=cfg.local, plan_mode=plan_mode, budget=budget, n_cap=ncap)


def padded(x, ncap):
    """K-like [B][H][n][d] -> [B][H][ncap][d], zeros past n (capacity, not keys)."""
    out = np.zeros(x.shape[:2] + (ncap,) + x.shape[3:], x.dtype)
    out[:, :, :x.shape[2]] = x
    return out


def run_gpu(sd, cfg, inp, kind, plan_mode=0, budget=56, dev_in=None):
    from top_sparse_decode_gb300.pipeline import DecodeStep, build_index
    sc = step_config(sd, cfg, kind, plan_mode, budget)
    if sc.n_cap:
        dev_in = (dev(inp.q), dev(padded(inp.K, sc.n_cap)), dev(padded(inp.V, sc.n_cap)))
    q, K, V = dev_in if dev_in else (dev(inp.q), dev(inp.K), dev(inp.V))
    enc = None
    if kind == sd.SD_IDX_SIG:
        enc = sd.make_encoder(dev(inp.W1), dev(inp.b1),
                              dev(inp.W2) if inp.W2 is not None else None,
                              dev(inp.b2) if inp.b2 is not None else None)
    index = build_index(sc, K, enc)
    step = DecodeStep(sc, K, V, index, enc=enc, sigma2=dev(inp.sigma2))
    step.run(q)
    if step.use_ht:  # the fused Hamming path keeps no scores: score once more to check them
        step.stage_score(q)
    torch.cuda.synchronize()
    return (sc, host(step.idx, np.int32), host(step.count, np.int32),
            host(step.out, np.float32), host(step.lse, np.float32), step, (q, K, V))


def oracle_scores(cfg, inp, kind, plan_mode=0, budget=56):
    if kind == 0:
        sig = oracle.sig_encode(inp.K, inp.W1, inp.b1, inp.W2, inp.b2)
        qs = oracle.sig_encode(inp.q, inp.W1, inp.b1, inp.W2, inp.b2)
        s = oracle.hamming_score(sig, qs)
        return s.reshape(cfg.B * cfg.Hkv, -1), None
    if kind == 1:
        p, sc = oracle.plane_build(inp.K)
        pl = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, plan_mode, budget)
        s, l1 = oracle.plane_score(p, sc, pl, inp.q, with_l1=True, n=cfg.n)
        return s.reshape(cfg.B * cfg.Hkv, -1), l1.reshape(cfg.B * cfg.Hkv, -1)
    if kind == 3:
        s, l1 = oracle.landmark_score(oracle.landmark_build(inp.K), inp.q, with_l1=True)
        return s.reshape(cfg.B * cfg.Hkv, -1), l1.reshape(cfg.B * cfg.Hkv, -1)
    summ = oracle.minmax_build(inp.K)
    s, l1 = oracle.quest_score(summ, inp.q, with_l1=True)
    return s.reshape(cfg.B * cfg.Hkv, -1), l1.reshape(cfg.B * cfg.Hkv, -1)


def check_step(sd, cfg, inp, kind, plan_mode=0, budget=56, dev_in=None):
    sc, gi, gc, go, gl, step, dev_t = run_gpu(sd, cfg, inp, kind, plan_mode, budget, dev_in)
    s, l1 = oracle_scores(cfg, inp, kind, plan_mode, budget)
    ri, rc = oracle.topk(s, sc.k, sc.sink, sc.local, sc.block, cfg.n)
    rows = cfg.B * cfg.Hkv
    same = np.ones(rows, bool)
    if kind == sd.SD_IDX_SIG:
        assert np.array_equal(host(step.scores, np.int32), s)
        assert np.array_equal(gc, rc)
        for r in range(rows):
            assert np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]]), r
    else:
        check_scores(host(step.scores, np.float32), s, l1, "scores")
        gu = [np.unique(gi[r, :gc[r]] // sc.block) for r in range(rows)]
        differ = check_float_topk(gi, gc, ri, rc, s, l1, sc.k, sc.sink, sc.local, sc.block,
                                  cfg.n)
        for r in range(rows):
            same[r] = gc[r] == rc[r] and np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]])
        assert differ == (~same).sum() and differ <= max(1, rows // 16)
    ro, rl = oracle.gather_attend(inp.q, inp.K, inp.V, ri.reshape(cfg.B, cfg.Hkv, -1),
                                  rc.reshape(cfg.B, cfg.Hkv), 1 / math.sqrt(cfg.d))
    same_q = np.repeat(same.reshape(cfg.B, cfg.Hkv), cfg.G, axis=1)
    err = np.abs(go - ro)[same_q].max() if same_q.any() else 0.0
    assert err <= ATT_ATOL, err
    if not same.all():
        # rows whose set legitimately differs (a swap within the score tolerance):
        # the oracle's attention over the GPU's own selected set, on every row
        gsel = np.ascontiguousarray(gi[:, :max(1, gi.shape[1])]).reshape(cfg.B, cfg.Hkv, -1)
        ro2, rl2 = oracle.gather_attend(inp.q, inp.K, inp.V, gsel, gc.reshape(cfg.B, cfg.Hkv),
                                        1 / math.sqrt(cfg.d))
        err2 = np.abs(go - ro2).max()
        assert err2 <= ATT_ATOL, err2
        lfin = np.isfinite(rl2)
        assert np.abs(gl[lfin] - rl2[lfin]).max() <= 1e-4 * max(1.0, np.abs(rl2[lfin]).max())
        err = max(err, err2)
    # side metric: recall of the planted keys / blocks
    planted = inp.planted.reshape(rows, -1)
    hit = 0
    per = sc.block if not cfg.block_mode else 1  # planted tokens -> units
    for r in range(rows):
        units = set((gi[r, :gc[r]] // sc.block).tolist())
        hit += sum(int(p) // per in units for p in planted[r])
    return hit / planted.size, err, dev_t


def test_cfg0_tiny_all_scorers(sd):
    cfg = synth.config(0)
    inp = synth.make_inputs(cfg)
    dev_in = (dev(inp.q), dev(inp.K), dev(inp.V))
    for kind in (sd.SD_IDX_SIG, sd.SD_IDX_PLANES, sd.SD_IDX_MINMAX, sd.SD_IDX_LANDMARK):
        check_step(sd, cfg, inp, kind, dev_in=dev_in)


def test_cfg0_ragged_sizes(sd):
    # n not a multiple of the scan tiles (2048 tokens, 32 Quest blocks) nor of 16
    for n in (64 * 37, 16 * 53 + 7):
        cfg = synth.config(0, n=n, k=40, sink=3, local=17, blk_k=5)
        inp = synth.make_inputs(cfg)
        kinds = [sd.SD_IDX_SIG, sd.SD_IDX_MINMAX, sd.SD_IDX_LANDMARK, sd.SD_IDX_PLANES]
        for kind in kinds:
            check_step(sd, cfg, inp, kind)


def test_degenerate_budget_covers_everything(sd):
    # n <= sink + local + k: every token is selected; the step is dense attention
    cfg = synth.config(0, n=256, k=200, sink=30, local=40)
    inp = synth.make_inputs(cfg)
    check_step(sd, cfg, inp, sd.SD_IDX_SIG)


@pytest.mark.slow
def test_cfg1_hash_32k_full(sd):
    cfg = synth.config(1)
    inp = synth.make_inputs(cfg)
    recall, err, _ = check_step(sd, cfg, inp, sd.SD_IDX_SIG)
    print(f"cfg1 planted recall {recall:.3f}, attention err {err:.2e}")


@pytest.mark.slow
def test_cfg2_fathom_128k_full(sd):
    cfg = synth.config(2)
    inp = synth.make_inputs(cfg)
    dev_in = (dev(inp.q), dev(inp.K), dev(inp.V))
    for mode, budget in [(0, 47), (0, 56), (0, 92), (2, 0), (3, 16), (4, 56)]:
        recall, err, _ = check_step(sd, cfg, inp, sd.SD_IDX_PLANES, mode, budget, dev_in)
        print(f"cfg2 mode {mode} budget {budget}: planted recall {recall:.3f}, err {err:.2e}")


@pytest.mark.slow
def test_cfg3_quest_b64_full(sd):
    cfg = synth.config(3)
    inp = synth.make_inputs(cfg)
    recall, err, _ = check_step(sd, cfg, inp, sd.SD_IDX_MINMAX)
    print(f"cfg3 planted-block recall {recall:.3f}, attention err {err:.2e}")


@pytest.mark.slow
def test_cfg4_longctx_1m_full(sd):
    cfg = synth.config(4)
    inp = synth.make_inputs(cfg)
    dev_in = (dev(inp.q), dev(inp.K), dev(inp.V))
    for kind, mode, budget in [(sd.SD_IDX_PLANES, 0, 56), (sd.SD_IDX_PLANES, 1, 32),
                               (sd.SD_IDX_SIG, 0, 0)]:
        recall, err, _ = check_step(sd, cfg, inp, kind, mode, budget, dev_in)
        print(f"cfg4 kind {kind} mode {mode} budget {budget}: recall {recall:.3f}, err {err:.2e}")
