"""GPU parity of each stage against the CPU oracle, on the same seeded inputs.

Sizes span several CTA tiles and a ragged tail; every call goes through the
C ABI (top_sparse_decode_gb300 is ctypes marshalling only)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import ATT_ATOL, check_scores, dev, empty, host

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


def shape_of(sd, cfg, n_cap=0):
    return sd.make_shape(cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.d, n_cap)


def encoder_of(sd, inp):
    W1 = dev(inp.W1)
    b1 = dev(inp.b1)
    W2 = dev(inp.W2) if inp.W2 is not None else None
    b2 = dev(inp.b2) if inp.b2 is not None else None
    return sd.make_encoder(W1, b1, W2, b2)


# --------------------------------------------------------------------------------------
# S1 signatures and the query map: bit-exact
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("cid,n,hidden", [(0, 4096 + 37, 0), (1, 3000, 128), (1, 1000, 64),
                                          (1, 1000, 32)])
def test_signatures_bit_exact(sd, cid, n, hidden):
    cfg = synth.config(cid, n=n, B=2 if cid == 1 else 1, hidden=hidden)
    inp = synth.make_inputs(cfg, with_v=False)
    if hidden and hidden != 128:  # re-draw a narrower MLP with the same recipe
        inp.W1 = synth.normal_f32(cfg.seed, synth.TID_W1, (hidden, cfg.d), math.sqrt(1 / cfg.d))
        inp.b1 = np.zeros(hidden, np.float32)
        inp.W2 = synth.normal_f32(cfg.seed, synth.TID_W2, (32, hidden), math.sqrt(1 / hidden))
    shp = shape_of(sd, cfg, n_cap=n + 11)
    Kp = np.zeros((cfg.B, cfg.Hkv, n + 11, cfg.d), np.uint16)
    Kp[:, :, :n] = inp.K
    enc = encoder_of(sd, inp)
    sig = empty((cfg.B, cfg.Hkv, n + 11), np.uint32)
    sd.sd_build_index(sd.SD_IDX_SIG, shp, dev(Kp), enc, sig)
    qsig = empty((cfg.B, cfg.Hq), np.uint32)
    sd.sd_encode_query(shp, dev(inp.q), enc, qsig)
    torch.cuda.synchronize()
    ref = oracle.sig_encode(inp.K, inp.W1, inp.b1, inp.W2, inp.b2)
    refq = oracle.sig_encode(inp.q, inp.W1, inp.b1, inp.W2, inp.b2)
    assert np.array_equal(host(sig, np.uint32)[:, :, :n], ref)
    assert np.array_equal(host(qsig, np.uint32), refq)


# --------------------------------------------------------------------------------------
# S5a Hamming scan: bit-exact
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("G,n", [(1, 1023), (2, 4096), (4, 10001), (8, 2048 + 4)])
def test_hamming_scores_bit_exact(sd, G, n):
    B, Hkv = 2, 3
    words = (synth.uniform(40 + G, 1, B * Hkv * n) * 2**32).astype(np.uint64).astype(np.uint32)
    sig = words.reshape(B, Hkv, n)
    qs = (synth.uniform(40 + G, 2, B * Hkv * G) * 2**32).astype(np.uint64).astype(np.uint32)
    qsig = qs.reshape(B, Hkv * G)
    shp = sd.make_shape(B, Hkv * G, Hkv, n)
    out = empty((B, Hkv, n), np.int32)
    sd.sd_score(sd.SD_IDX_SIG, shp, dev(sig), None, dev(qsig), None, out)
    torch.cuda.synchronize()
    assert np.array_equal(host(out, np.int32), oracle.hamming_score(sig, qsig))


# --------------------------------------------------------------------------------------
# S2 bit planes: bit-exact planes and scales
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("n,ncap", [(4096, 4096), (2 * 1024 + 3 * 64, 2 * 1024 + 3 * 64),
                                    (1024 + 64, 4096)])
def test_plane_build_bit_exact(sd, n, ncap):
    cfg = synth.config(2, B=2, Hq=8, Hkv=2, n=n)
    inp = synth.make_inputs(cfg, with_v=False)
    Kp = np.zeros((cfg.B, cfg.Hkv, ncap, cfg.d), np.uint16)
    Kp[:, :, :n] = inp.K
    # a block of zeros (scale 1) and a huge key (scale overflow path is out of range; skip)
    Kp[0, 0, 64:128] = 0
    shp = shape_of(sd, cfg, n_cap=ncap)
    planes = torch.zeros((cfg.B, cfg.Hkv, cfg.d, 4, ncap // 32), dtype=torch.int32, device="cuda")
    scales = torch.zeros((cfg.B, cfg.Hkv, cfg.d, ncap // 64), dtype=torch.int16, device="cuda")
    sd.sd_build_index(sd.SD_IDX_PLANES, shp, dev(Kp), None, planes, scales)
    torch.cuda.synchronize()
    ref_p, ref_s = oracle.plane_build(Kp[:, :, :n].copy())
    assert np.array_equal(host(planes, np.uint32)[..., : n // 32], ref_p)
    assert np.array_equal(host(scales, np.uint16)[..., : n // 64], ref_s)


# --------------------------------------------------------------------------------------
# S3 min/max summaries: bit-exact
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("n", [16 * 8 * 5, 16 * 300 + 5, 17])
def test_minmax_build_bit_exact(sd, n):
    cfg = synth.config(3, B=2, Hq=8, Hkv=2, n=n, planted=2)
    inp = synth.make_inputs(cfg, with_v=False)
    inp.K[0, 0, 3, :8] = 0x8000  # -0.0 mixed with +0.0 below
    inp.K[0, 0, 4, :8] = 0x0000
    shp = shape_of(sd, cfg)
    nblk = (n + 15) // 16
    summ = empty((cfg.B, cfg.Hkv, nblk, 2, cfg.d), np.uint16)
    sd.sd_build_index(sd.SD_IDX_MINMAX, shp, dev(inp.K), None, summ)
    torch.cuda.synchronize()
    assert np.array_equal(host(summ, np.uint16), oracle.minmax_build(inp.K))


# --------------------------------------------------------------------------------------
# S4 read plan: bit-exact
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("G", [1, 4, 8])
def test_plan_bit_exact(sd, G):
    cfg = synth.config(2, B=3, Hq=2 * G, Hkv=2, n=64)
    inp = synth.make_inputs(cfg, with_v=False)
    inp.q[1, :, 5:9] = 0  # zero-gain channels
    inp.q[0, :, 20:24] = inp.q[0, :, 20:21]  # equal query mass: ties to the lower channel
    shp = shape_of(sd, cfg)
    plan = empty((cfg.B, cfg.Hkv, cfg.d), np.uint8)
    q = dev(inp.q)
    s2 = dev(inp.sigma2)
    for mode, budgets in [(sd.SD_PLAN_WATERFILL, [0, 1, 47, 56, 92, 200, 511, 512]),
                          (sd.SD_PLAN_FIXED, [0, 1, 32, 128]), (sd.SD_PLAN_FULL, [0]),
                          (sd.SD_PLAN_TOPQ, [0, 1, 17, 21, 22, 32, 124, 127, 128])]:
        for B in budgets:
            sd.sd_plan(shp, q, None if mode == sd.SD_PLAN_TOPQ else s2, mode, B, plan)
            torch.cuda.synchronize()
            ref = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, mode, B)
            assert np.array_equal(host(plan, np.uint8), ref), (mode, B)


@pytest.mark.parametrize("Hkv,G,B", [(1, 4, 2), (2, 4, 3), (8, 4, 2), (3, 2, 1), (16, 1, 1)])
def test_plan_split_bit_exact(sd, Hkv, G, B):
    """The budget split across KV heads (one CTA per sequence) equals the oracle's
    greedy over every (head, channel) of the sequence, ties to the lower head and
    channel; with one head it is the water-filling plan."""
    cfg = synth.config(2, B=B, Hq=G * Hkv, Hkv=Hkv, n=64)
    inp = synth.make_inputs(cfg, with_v=False)
    inp.q[0, :, 5:9] = 0  # zero-gain channels
    if Hkv > 1:  # equal gains in two heads: ties to the lower head
        inp.sigma2[1] = inp.sigma2[0]
        inp.q[0, G:2 * G] = inp.q[0, :G]
    shp = shape_of(sd, cfg)
    plan = empty((cfg.B, cfg.Hkv, cfg.d), np.uint8)
    q, s2 = dev(inp.q), dev(inp.sigma2)
    for budget in [0, 1, 47, 56, 92, 200, 511, 512]:
        sd.sd_plan(shp, q, s2, sd.SD_PLAN_SPLIT, budget, plan)
        torch.cuda.synchronize()
        ref = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, oracle.PLAN_SPLIT, budget)
        got = host(plan, np.uint8)
        assert np.array_equal(got, ref), budget
        assert np.all(got.astype(np.int64).sum(axis=(1, 2)) == min(Hkv * budget, Hkv * 512))
        if Hkv == 1:
            assert np.array_equal(got, oracle.plan(inp.q, inp.sigma2, 1, oracle.PLAN_WATERFILL,
                                                   budget))


# --------------------------------------------------------------------------------------
# S5b bit-plane scan and S5c Quest bound: within 1e-5 of the L1 mass
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("budget,mode,ncap", [(56, 0, 0), (47, 0, 0), (92, 0, 0), (0, 0, 0),
                                               (32, 1, 0), (0, 2, 0), (56, 0, 4608),
                                               (0, 2, 4608), (17, 3, 0), (17, 3, 4608)])
def test_plane_scores(sd, budget, mode, ncap):
    # n = 4288: one full 4096-token tile and a last tile of 6 words / 3 scale
    # blocks; ncap = 4608 (a multiple of 512) takes the 16-byte staging path
    cfg = synth.config(2, B=2, Hq=8, Hkv=2, n=2 * 2048 + 3 * 64)
    inp = synth.make_inputs(cfg, with_v=False)
    ncap = ncap or cfg.n
    shp = shape_of(sd, cfg, n_cap=ncap)
    ref_p, ref_s = oracle.plane_build(inp.K)
    plan_ref = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, mode, budget)
    ref, l1 = oracle.plane_score(ref_p, ref_s, plan_ref, inp.q, with_l1=True)
    Kp = np.zeros((cfg.B, cfg.Hkv, ncap, cfg.d), np.uint16)
    Kp[:, :, :cfg.n] = inp.K
    planes = empty((cfg.B, cfg.Hkv, cfg.d, 4, ncap // 32), np.uint32)
    scales = empty((cfg.B, cfg.Hkv, cfg.d, ncap // 64), np.uint16)
    sd.sd_build_index(sd.SD_IDX_PLANES, shp, dev(Kp), None, planes, scales)
    plan = empty(plan_ref.shape, np.uint8)
    q = dev(inp.q)
    sd.sd_plan(shp, q, dev(inp.sigma2), mode, budget, plan)
    scores = empty((cfg.B, cfg.Hkv, cfg.n), np.float32)
    sd.sd_score(sd.SD_IDX_PLANES, shp, planes, scales, q, plan, scores)
    torch.cuda.synchronize()
    check_scores(host(scores, np.float32), ref, l1, "plane scores")


@pytest.mark.parametrize("B,Hkv,n,budget,mode", [(1, 8, 262144, 56, 0), (2, 4, 300 * 512 + 192, 56, 0),
                                                 (1, 8, 262144, 80, 1)])
def test_plane_scores_long_ranges(sd, B, Hkv, n, budget, mode):
    # more 512-token units than resident CTAs: each CTA walks several tiles, ranges
    # cross row ends, the next tile is prefetched (at most 64 active channels) or
    # not (80 channels of the fixed plan), and a row may end in a partial unit
    cfg = synth.config(4, B=B, Hq=4 * Hkv, Hkv=Hkv, n=n)
    inp = synth.make_inputs(cfg, with_v=False)
    shp = shape_of(sd, cfg)
    ref_p, ref_s = oracle.plane_build(inp.K)
    plan_ref = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, mode, budget)
    ref, l1 = oracle.plane_score(ref_p, ref_s, plan_ref, inp.q, with_l1=True)
    q = dev(inp.q)
    plan = empty(plan_ref.shape, np.uint8)
    sd.sd_plan(shp, q, dev(inp.sigma2), mode, budget, plan)
    scores = empty((cfg.B, cfg.Hkv, cfg.n), np.float32)
    sd.sd_score(sd.SD_IDX_PLANES, shp, dev(ref_p), dev(ref_s), q, plan, scores)
    torch.cuda.synchronize()
    assert np.array_equal(host(plan, np.uint8), plan_ref)
    check_scores(host(scores, np.float32), ref, l1, "plane scores")


@pytest.mark.parametrize("G,n", [(4, 16 * 1024), (8, 16 * 100 + 9), (1, 16 * 33)])
def test_quest_scores(sd, G, n):
    cfg = synth.config(3, B=3, Hq=2 * G, Hkv=2, n=n, planted=4)
    inp = synth.make_inputs(cfg, with_v=False)
    shp = shape_of(sd, cfg)
    ref_summ = oracle.minmax_build(inp.K)
    ref, l1 = oracle.quest_score(ref_summ, inp.q, with_l1=True)
    summ = empty(ref_summ.shape, np.uint16)
    sd.sd_build_index(sd.SD_IDX_MINMAX, shp, dev(inp.K), None, summ)
    scores = empty(ref.shape, np.float32)
    sd.sd_score(sd.SD_IDX_MINMAX, shp, summ, None, dev(inp.q), None, scores)
    torch.cuda.synchronize()
    check_scores(host(scores, np.float32), ref, l1, "quest scores")


# --------------------------------------------------------------------------------------
# 8-token block landmarks (Fathom's landmark comparison scan): build bit-exact,
# scores within 1e-5 of the L1 mass
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("n,ncap", [(8 * 1000, 0), (8 * 777 + 5, 0), (1, 0), (4101, 4160)])
def test_landmark_build_bit_exact(sd, n, ncap):
    cfg = synth.config(3, B=2, Hq=8, Hkv=2, n=n, planted=0)
    inp = synth.make_inputs(cfg, with_v=False)
    ncap = ncap or n
    Kp = np.zeros((cfg.B, cfg.Hkv, ncap, cfg.d), np.uint16)
    Kp[:, :, :n] = inp.K
    shp = shape_of(sd, cfg, n_cap=ncap)
    L = torch.full((cfg.B, cfg.Hkv, (ncap + 7) // 8, cfg.d), 0x1234, dtype=torch.int16,
                   device="cuda")
    sd.sd_build_index(sd.SD_IDX_LANDMARK, shp, dev(Kp), None, L)
    torch.cuda.synchronize()
    nb = (n + 7) // 8
    got = host(L, np.uint16)
    assert np.array_equal(got[:, :, :nb], oracle.landmark_build(inp.K))
    assert (got[:, :, nb:] == 0x1234).all()  # blocks past n are not written


@pytest.mark.parametrize("G,n", [(4, 8 * 4096), (8, 8 * 100 + 3), (1, 8 * 33), (2, 8 * 5000)])
def test_landmark_scores(sd, G, n):
    cfg = synth.config(3, B=3, Hq=2 * G, Hkv=2, n=n, planted=0)
    inp = synth.make_inputs(cfg, with_v=False)
    shp = shape_of(sd, cfg)
    ref_L = oracle.landmark_build(inp.K)
    ref, l1 = oracle.landmark_score(ref_L, inp.q, with_l1=True)
    L = empty(ref_L.shape, np.uint16)
    sd.sd_build_index(sd.SD_IDX_LANDMARK, shp, dev(inp.K), None, L)
    scores = empty(ref.shape, np.float32)
    sd.sd_score(sd.SD_IDX_LANDMARK, shp, L, None, dev(inp.q), None, scores)
    torch.cuda.synchronize()
    assert np.array_equal(host(L, np.uint16), ref_L)
    check_scores(host(scores, np.float32), ref, l1, "landmark scores")


# --------------------------------------------------------------------------------------
# S6 top-k on identical generated scores: bit-exact against the oracle
# --------------------------------------------------------------------------------------
def run_topk(sd, scores_np, k, sink, local, block=1, n_tokens=None):
    rows, n_units = scores_np.shape
    if n_tokens is None:
        n_tokens = n_units * block
    sel = sd.make_select(k, sink, local, block)
    stride = min(n_units, sink + local + k) * block
    idx = torch.full((rows, stride), -7, dtype=torch.int32, device="cuda")
    cnt = empty((rows,), np.int32)
    ws_bytes = sd.sd_topk_workspace_size(rows, n_units, sel)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda") if ws_bytes else None
    st = sd.SD_SCORE_I32 if scores_np.dtype == np.int32 else sd.SD_SCORE_F32
    sd.sd_topk(st, dev(scores_np), rows, n_units, n_tokens, sel, idx, stride, cnt, ws)
    torch.cuda.synchronize()
    return host(idx, np.int32), host(cnt, np.int32)


TOPK_CASES = [
    # (rows, n_units, kind, levels, k, sink, local)
    (3, 100, "f32", 0, 10, 2, 3),
    (4, 4096, "f32", 0, 64, 4, 64),
    (2, 8192, "f32ties", 7, 512, 0, 0),
    (3, 8192, "int", 128, 300, 16, 16),
    (2, 5000, "const", 0, 4096, 1, 1),
    (2, 8193, "f32", 0, 512, 0, 0),
    (3, 32768, "int", 128, 512, 128, 512),
    (2, 32768, "int", 8, 100, 0, 0),
    (2, 100000, "f32", 0, 512, 0, 0),
    (2, 100000, "f32ties", 3, 1000, 7, 9),
    (2, 20000, "const", 0, 2000, 0, 0),
    (1, 20000, "f32ties", 1, 4096, 0, 0),
]


@pytest.mark.parametrize("rows,n,kind,levels,k,sink,local", TOPK_CASES)
def test_topk_bit_exact_on_shared_scores(sd, rows, n, kind, levels, k, sink, local):
    s = synth.make_scores(1000 + n + k, rows, n, kind, levels)
    gi, gc = run_topk(sd, s, k, sink, local)
    ri, rc = oracle.topk(s, k, sink, local)
    for r in range(rows):
        assert gc[r] == rc[r], (r, gc[r], rc[r])
        assert np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]]), r


def test_topk_estimate_misses_fall_back_to_exact(sd):
    # Long rows: the threshold is estimated from up to 8192 evenly spaced units
    # (unit floor(s * step) with step = M / 8192 in 32.32 fixed point).  (a) 200
    # large scores, all on sampled units: the estimate admits fewer than k
    # candidates.  (b) every unsampled unit large: far more candidates than the
    # selection holds.  Both must still be exact.
    M = 100000
    Ssz = min(M, 8192)
    step = (M << 32) // Ssz
    pos = (np.arange(Ssz, dtype=np.uint64) * np.uint64(step)) >> np.uint64(32)
    pos = pos.astype(np.int64)
    a = np.zeros((1, M), np.float32)
    a[0, pos[::37][:200]] = 1.0
    b = np.full((1, M), 5.0, np.float32)
    b[0, pos] = 1.0
    b[0, 7] = 9.0
    for s in (a, b):
        gi, gc = run_topk(sd, s, 512, 0, 0)
        ri, rc = oracle.topk(s, 512, 0, 0)
        assert gc[0] == rc[0] and np.array_equal(gi[0, :gc[0]], ri[0, :rc[0]])


def test_topk_clustered_winners(sd):
    # the top k sit in one narrow index range (sorting falls back to bitonic)
    s = synth.make_scores(3, 2, 200000, "f32")
    s[:, 50000:53000] += 100.0
    for k in (512, 3000, 4096):
        gi, gc = run_topk(sd, s, k, 1, 1)
        ri, rc = oracle.topk(s, k, 1, 1)
        for r in range(2):
            assert gc[r] == rc[r] and np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]])


def test_topk_block_mode_bit_exact(sd):
    nblk = 1024
    s = synth.make_scores(77, 6, nblk, "f32")
    n_tokens = nblk * 16 - 5  # short last block
    gi, gc = run_topk(sd, s, 128, 0, 1, block=16, n_tokens=n_tokens)
    ri, rc = oracle.topk(s, 128, 0, 1, block=16, n_tokens=n_tokens)
    assert np.array_equal(gc, rc) and gc[0] == 128 * 16 + 11
    for r in range(6):
        assert np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]])


# Rows of at most 2048 competing units take the register kernel (one CTA of 4 warps
# per row, keys in registers, a bitwise search for the k-th largest key, ties that
# span warps); 2049 takes the shared-memory CTA kernel.
REG_TOPK_CASES = [
    # (rows, n_units, kind, levels, k, sink, local)
    (701, 1024, "f32", 0, 128, 0, 1),   # many rows
    (5, 2056, "f32ties", 3, 200, 4, 4),  # M = 2048, the largest warp row
    (3, 2049, "f32", 0, 100, 0, 0),     # M = 2049: the CTA kernel
    (6, 33, "int", 4, 5, 0, 0),
    (7, 129, "f32ties", 2, 64, 0, 0),
    (3, 300, "const", 0, 17, 0, 0),     # every key tied: the lowest units
    (2, 200, "f32", 0, 1, 3, 3),        # k = 1 beside the windows
    (2, 150, "f32", 0, 200, 2, 2),      # k >= M: every unit
    (2, 1, "f32", 0, 1, 0, 0),
    (9, 600, "int", 1, 250, 1, 1),
]


@pytest.mark.parametrize("rows,n,kind,levels,k,sink,local", REG_TOPK_CASES)
def test_topk_reg_rows_bit_exact(sd, rows, n, kind, levels, k, sink, local):
    s = synth.make_scores(2000 + n + k, rows, n, kind, levels)
    gi, gc = run_topk(sd, s, k, sink, local)
    ri, rc = oracle.topk(s, k, sink, local)
    for r in range(rows):
        assert gc[r] == rc[r], (r, gc[r], rc[r])
        assert np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]]), r


def test_topk_reg_rows_block_mode_last_unit(sd):
    # no trailing window: the cut last block competes, and is taken in rows 0, 2, 4
    nblk = 1024
    s = synth.make_scores(78, 5, nblk, "f32")
    s[::2, nblk - 1] = 100.0
    n_tokens = nblk * 16 - 5
    gi, gc = run_topk(sd, s, 128, 0, 0, block=16, n_tokens=n_tokens)
    ri, rc = oracle.topk(s, 128, 0, 0, block=16, n_tokens=n_tokens)
    assert np.array_equal(gc, rc) and gc[0] == 128 * 16 - 5 and gc[1] == 128 * 16
    for r in range(5):
        assert np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]]), r


def test_topk_reg_rows_odd_blocks_and_strides(sd):
    # 6-token blocks (scalar token writes, a division per position in the windows'
    # writer) with a cut last block, and 16-token blocks with a row stride that is not
    # a multiple of 4 entries (no 16-byte stores)
    for blk, extra in ((6, 0), (16, 1), (4, 3)):
        nblk = 700
        s = synth.make_scores(90 + blk, 9, nblk, "f32ties", 5)
        s[::3, nblk - 1] = 10.0  # the cut last block is taken in rows 0, 3, 6
        n_tokens = nblk * blk - (blk - 1)
        sel = sd.make_select(50, 2, 0, blk)
        stride = (2 + 50) * blk + extra
        idx = torch.full((9, stride), -7, dtype=torch.int32, device="cuda")
        cnt = empty((9,), np.int32)
        sd.sd_topk(sd.SD_SCORE_F32, dev(s), 9, nblk, n_tokens, sel, idx, stride, cnt, None)
        torch.cuda.synchronize()
        gi, gc = host(idx, np.int32), host(cnt, np.int32)
        ri, rc = oracle.topk(s, 50, 2, 0, block=blk, n_tokens=n_tokens)
        assert np.array_equal(gc, rc), (blk, gc, rc)
        assert gc[0] == 52 * blk - (blk - 1) and gc[1] == 52 * blk
        for r in range(9):
            assert np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]]), (blk, r)
            assert (gi[r, gc[r]:] == -7).all(), (blk, r)  # nothing written past count


def test_topk_reg_rows_signed_zeros_infinities_nan(sd):
    rng = np.random.default_rng(11)
    s = rng.standard_normal((8, 1000)).astype(np.float32)
    s[0] = np.where(rng.random(1000) < 0.5, np.float32(-0.0), np.float32(0.0))
    s[1, rng.choice(1000, 30, replace=False)] = np.inf
    s[1, rng.choice(1000, 30, replace=False)] = -np.inf
    s[2] = -np.inf
    s[3, 500] = np.nan   # a competing NaN: the row reports -1
    s[4, 1] = np.nan     # inside the leading window: ignored
    s[5, 998] = np.nan   # inside the trailing window: ignored
    gi, gc = run_topk(sd, s, 40, 2, 3)
    ri, rc = oracle.topk(np.where(np.isnan(s), np.float32(0), s), 40, 2, 3)
    assert gc[3] == -1
    for r in (0, 1, 2, 4, 5, 6, 7):
        assert gc[r] == rc[r], (r, gc[r], rc[r])
        assert np.array_equal(gi[r, :gc[r]], ri[r, :rc[r]]), r


def test_topk_nan_row(sd):
    s = synth.make_scores(5, 3, 9000, "f32")
    s[1, 4444] = np.nan
    _, gc = run_topk(sd, s, 10, 0, 0)
    assert gc[1] == -1 and gc[0] == 10 and gc[2] == 10
    s2 = s[:, :500].copy()
    _, gc2 = run_topk(sd, s2, 10, 0, 0)
    assert gc2[0] == 10 and gc2[2] == 10


# --------------------------------------------------------------------------------------
# S7 gather-attend on identical generated index lists: 2e-3 absolute
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("G,max_count", [(4, 1152), (8, 2064), (1, 63), (2, 200), (4, 9000)])
def test_gather_attend(sd, G, max_count):
    cfg = synth.config(1, B=2, Hq=3 * G, Hkv=3, n=max(5000, max_count + 100))
    inp = synth.make_inputs(cfg)
    rows = cfg.B * cfg.Hkv
    counts = np.array([max_count, 1, 0, 65, max_count - 1, 64][:rows])
    idx, cnt = synth.make_index_lists(9, rows, cfg.n, max_count, counts)
    scale = 1 / math.sqrt(cfg.d)
    ref_o, ref_l = oracle.gather_attend(inp.q, inp.K, inp.V, idx.reshape(cfg.B, cfg.Hkv, -1),
                                        cnt.reshape(cfg.B, cfg.Hkv), scale)
    shp = shape_of(sd, cfg)
    out = empty((cfg.B, cfg.Hq, cfg.d), np.float32)
    lse = empty((cfg.B, cfg.Hq), np.float32)
    wsz = sd.sd_gather_attend_workspace_size(shp, max_count)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    sd.sd_gather_attend(shp, dev(inp.q), dev(inp.K), dev(inp.V), dev(idx), max_count, dev(cnt),
                        max_count, scale, out, lse, ws)
    torch.cuda.synchronize()
    o = host(out, np.float32)
    err = np.abs(o - ref_o).max()
    assert err <= ATT_ATOL, err
    lg = host(lse, np.float32)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.abs(lg[fin] - ref_l[fin]).max() <= 1e-4 * max(1, np.abs(ref_l[fin]).max())
