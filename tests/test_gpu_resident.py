"""Delta selection against a resident set and the gather of the admitted units
(sd_delta_select, sd_resident_gather) against the oracle over multi-step drifting
predictions: the plan, the pool rows and the whole resident-set state bit for bit
after every step; the gathered pool pages against the source rows (device and
pinned host sources); and attention over the pool against the oracle's attention
over the same tokens in place."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import ATT_ATOL, dev, host

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


def drifting_scores(rng, rows, nu, step, prev):
    """Scores that drift between steps (so hits, misses and evictions all occur),
    with ties and signed zeros."""
    s = rng.normal(size=(rows, nu)).astype(np.float32) if prev is None else \
        (0.8 * prev + 0.6 * rng.normal(size=(rows, nu))).astype(np.float32)
    s[:, 3::11] = 0.25
    s[:, 5::13] = np.float32(-0.0)
    s[:, 7::13] = np.float32(0.0)
    return s


def run_steps(sd, B, Hkv, n, block, k, sink, local, R, caps, seed, nan_step=None):
    rng = np.random.default_rng(seed)
    rows, nu = B * Hkv, (n + block - 1) // block
    units = min(nu, sink + local + k)
    stride = units * block
    shp = sd.make_shape(B, 4 * Hkv, Hkv, n)
    sel = sd.make_select(k, sink, local, block)
    res = sd.Resident(rows, R, nu)
    ref = oracle.Resident(rows, R, nu)
    pc, pcount = (torch.empty(rows, dtype=torch.int32, device="cuda") for _ in range(2))
    pool = torch.full((rows, stride), -7, dtype=torch.int32, device="cuda")
    prev = None
    for step, C in enumerate(caps):
        # plan arrays [rows][C] (C is their row stride)
        ps, pu, pe = (torch.full((rows, max(C, 1)), -7, dtype=torch.int32, device="cuda")
                      for _ in range(3))
        sc = drifting_scores(rng, rows, nu, step, prev)
        prev = sc
        ri, rc = oracle.topk(sc, k, sink, local, block, n)
        assert ri.shape[1] == stride
        if step == nan_step:
            rc = rc.copy()
            rc[1] = -1
        sd.sd_delta_select(shp, sel, dev(sc), dev(ri), stride, dev(rc), C, step, res, ps, pu, pe,
                           pc, pool, stride, pcount)
        torch.cuda.synchronize()
        rps, rpu, rpe, rpc, rpool, rpcount = oracle.delta_select(ref, sc, ri, rc, block, n, sink,
                                                                local, C, step, stride)
        gpc = host(pc, np.int32)
        assert np.array_equal(gpc, rpc), step
        gps, gpu_, gpe = host(ps, np.int32), host(pu, np.int32), host(pe, np.int32)
        gpool, gcount = host(pool, np.int32), host(pcount, np.int32)
        assert np.array_equal(gcount, rpcount), step
        for r in range(rows):
            a = max(int(rpc[r]), 0)
            assert np.array_equal(gps[r, :a], rps[r, :a]), (step, r)
            assert np.array_equal(gpu_[r, :a], rpu[r, :a]), (step, r)
            assert np.array_equal(gpe[r, :a], rpe[r, :a]), (step, r)
            m = max(int(rpcount[r]), 0)
            assert np.array_equal(gpool[r, :m], rpool[r, :m]), (step, r)
        assert np.array_equal(host(res.slot_unit, np.int32), ref.slot_unit), step
        assert np.array_equal(host(res.slot_last, np.int32), ref.slot_last.astype(np.int32)), step
        assert np.array_equal(host(res.unit_slot, np.int32), ref.unit_slot), step


@pytest.mark.parametrize("B,Hkv,n,block,k,sink,local,R,caps", [
    # 300 units (the last 11 tokens), 64 slots; caps 0, small, beyond every miss
    (3, 4, 16 * 300 - 5, 16, 40, 1, 1, 64, [3, 7, 0, 64, 1, 5, 5, 2, 9, 4]),
    # fewer slots than predicted units: some predicted units never become resident
    (2, 2, 16 * 120, 16, 48, 0, 2, 30, [8, 8, 30, 3, 1, 8]),
    # token units (block 1) and a large cap
    (1, 3, 3000, 1, 200, 4, 16, 256, [256, 40, 40, 0, 100]),
    # the OasisKV shape: 64 x 8 heads, 16,384 tokens, top-128 + 1 local, 129 slots,
    # fetch ratio 0.05 of 128 -> C = 7
    (64, 8, 16384, 16, 128, 0, 1, 129, [7] * 8),
])
def test_delta_select_matches_oracle(sd, B, Hkv, n, block, k, sink, local, R, caps):
    run_steps(sd, B, Hkv, n, block, k, sink, local, R, caps, seed=B * 131 + n)


def test_delta_select_nan_row(sd):
    run_steps(sd, 2, 2, 16 * 100, 16, 20, 0, 1, 24, [5, 5, 5, 5], seed=5, nan_step=2)


def test_delta_select_garbage_state_stays_in_bounds(sd):
    """State arrays holding values out of range: the kernel reads them as 'not
    resident' and every plan entry it writes is in range."""
    B, Hkv, n, block, k, R = 2, 2, 16 * 64, 16, 16, 20
    rows, nu = B * Hkv, n // block
    rng = np.random.default_rng(3)
    res = sd.Resident(rows, R, nu)
    res.slot_unit.copy_(torch.from_numpy(rng.integers(-5, 2 * nu, (rows, R), dtype=np.int32)))
    res.slot_last.copy_(torch.from_numpy(rng.integers(-9, 50, (rows, R), dtype=np.int32)))
    res.unit_slot.copy_(torch.from_numpy(rng.integers(-3, 2 * R, (rows, nu), dtype=np.int32)))
    sc = rng.normal(size=(rows, nu)).astype(np.float32)
    ri, rc = oracle.topk(sc, k, 0, 1, block, n)
    stride = ri.shape[1]
    ps, pu, pe = (torch.full((rows, 8), -7, dtype=torch.int32, device="cuda") for _ in range(3))
    pc, pcount = (torch.empty(rows, dtype=torch.int32, device="cuda") for _ in range(2))
    pool = torch.full((rows, stride), -7, dtype=torch.int32, device="cuda")
    sd.sd_delta_select(sd.make_shape(B, 4 * Hkv, Hkv, n), sd.make_select(k, 0, 1, block), dev(sc),
                       dev(ri), stride, dev(rc), 8, 60, res, ps, pu, pe, pc, pool, stride, pcount)
    torch.cuda.synchronize()
    gpc = host(pc, np.int32)
    for r in range(rows):
        a = int(gpc[r])
        assert 0 <= a <= 8
        assert ((host(ps, np.int32)[r, :a] >= 0) & (host(ps, np.int32)[r, :a] < R)).all()
        assert ((host(pu, np.int32)[r, :a] >= 0) & (host(pu, np.int32)[r, :a] < nu)).all()
    gp = host(pool, np.int32)
    gcount = host(pcount, np.int32)
    for r in range(rows):
        assert ((gp[r, :gcount[r]] >= 0) & (gp[r, :gcount[r]] < R * block)).all()


@pytest.mark.parametrize("pinned", [False, True])
def test_resident_gather_and_attend_over_pool(sd, pinned):
    """Steps of select -> gather (from device or pinned host K/V) -> attend over the
    pool: the pool pages hold the admitted units' rows (zeros past n), untouched
    pages keep their contents, and attention over the pool rows equals the
    oracle's attention over the same tokens in place."""
    B, Hkv, G, n, block, k, local, R = 2, 4, 4, 16 * 200 - 7, 16, 24, 1, 40
    caps = [40, 6, 6, 6]
    rows, nu = B * Hkv, (n + block - 1) // block
    rng = np.random.default_rng(11)
    Kh = (rng.normal(size=(B, Hkv, n, 128)) * 0.5).astype(np.float32)
    Vh = rng.normal(size=(B, Hkv, n, 128)).astype(np.float32)
    q = rng.normal(size=(B, Hkv * G, 128)).astype(np.float32)
    Kt = torch.from_numpy(Kh).to(torch.bfloat16)
    Vt = torch.from_numpy(Vh).to(torch.bfloat16)
    qt = torch.from_numpy(q).to(torch.bfloat16).cuda()
    Ksrc = Kt.pin_memory() if pinned else Kt.cuda()
    Vsrc = Vt.pin_memory() if pinned else Vt.cuda()
    Kb = Kt.view(torch.int16).numpy().view(np.uint16)
    Vb = Vt.view(torch.int16).numpy().view(np.uint16)
    shp = sd.make_shape(B, Hkv * G, Hkv, n)
    sel = sd.make_select(k, 0, local, block)
    units = min(nu, local + k)
    stride = units * block
    res = sd.Resident(rows, R, nu)
    ref = oracle.Resident(rows, R, nu)
    pc, pcount = (torch.empty(rows, dtype=torch.int32, device="cuda") for _ in range(2))
    pool = torch.full((rows, stride), -7, dtype=torch.int32, device="cuda")
    Kp = torch.full((B, Hkv, R * block, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    Vp = torch.full((B, Hkv, R * block, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    pshp = sd.make_shape(B, Hkv * G, Hkv, R * block)
    prev = None
    for step, C in enumerate(caps):
        ps, pu, pe = (torch.full((rows, C), -7, dtype=torch.int32, device="cuda")
                      for _ in range(3))
        sc = drifting_scores(rng, rows, nu, step, prev)
        prev = sc
        ri, rc = oracle.topk(sc, k, 0, local, block, n)
        before = host(Kp.view(torch.int16), np.int16).copy()
        sd.sd_delta_select(shp, sel, dev(sc), dev(ri), ri.shape[1], dev(rc), C, step, res, ps, pu,
                           pe, pc, pool, stride, pcount)
        sd.sd_resident_gather(shp, block, Ksrc, Vsrc, ps, pu, pc, C, R, Kp, Vp)
        torch.cuda.synchronize()
        rps, rpu, _, rpc, rpool, rpcount = oracle.delta_select(ref, sc, ri, rc, block, n, 0, local,
                                                              C, step, stride)
        gk = host(Kp.view(torch.int16), np.int16).view(np.uint16).reshape(rows, R * block, 128)
        gv = host(Vp.view(torch.int16), np.int16).view(np.uint16).reshape(rows, R * block, 128)
        touched = np.zeros((rows, R), bool)
        for r in range(rows):
            for i in range(int(rpc[r])):
                s, u = int(rps[r, i]), int(rpu[r, i])
                touched[r, s] = True
                ln = min(block, n - u * block)
                src_k = Kb.reshape(rows, n, 128)[r, u * block:u * block + ln]
                src_v = Vb.reshape(rows, n, 128)[r, u * block:u * block + ln]
                assert np.array_equal(gk[r, s * block:s * block + ln], src_k), (step, r, i)
                assert np.array_equal(gv[r, s * block:s * block + ln], src_v), (step, r, i)
                assert not gk[r, s * block + ln:(s + 1) * block].any()
        old = before.view(np.uint16).reshape(rows, R, block, 128)
        now = gk.reshape(rows, R, block, 128)
        assert np.array_equal(now[~touched], old[~touched]), step
        # attention over the pool rows against the oracle over the same tokens in place
        tok = np.full((rows, stride), -1, np.int32)
        for r in range(rows):
            rows_r = rpool[r, :rpcount[r]]
            slots, offs = rows_r // block, rows_r % block
            tok[r, :len(rows_r)] = ref.slot_unit[r, slots] * block + offs
        ows = sd.sd_gather_attend_workspace_size(pshp, stride)
        aws = torch.empty(max(ows, 16), dtype=torch.uint8, device="cuda")
        out = torch.empty((B, Hkv * G, 128), dtype=torch.float32, device="cuda")
        lse = torch.empty((B, Hkv * G), dtype=torch.float32, device="cuda")
        sd.sd_gather_attend(pshp, qt, Kp, Vp, pool, stride, pcount, stride, 1 / np.sqrt(128.0),
                            out, lse, aws)
        torch.cuda.synchronize()
        qb = qt.cpu().view(torch.int16).numpy().view(np.uint16)
        o_ref, _ = oracle.gather_attend(qb, Kb, Vb, tok.reshape(B, Hkv, -1),
                                        rpcount.reshape(B, Hkv), 1 / np.sqrt(128.0))
        assert np.abs(host(out, np.float32) - o_ref).max() <= ATT_ATOL, step
