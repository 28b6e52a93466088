"""Offload path (Fathom: host planes are channel-contiguous, one gather copies the
active channels' prefixes into HBM before the scan; OasisKV: UVA gather kernel on
a side stream): sd_offload_gather copies exactly the planned prefixes from pinned
host memory, the scan over them matches the oracle, and the host-side bounded
wait reports a timeout without touching the device."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import check_scores, dev, host

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


@pytest.mark.parametrize("n,budget,mode", [(65536, 56, 0), (4096 + 64, 92, 0), (8192, 32, 1)])
def test_offload_gathers_exactly_the_planned_prefixes(sd, n, budget, mode):
    cfg = synth.config(4, n=n)
    inp = synth.make_inputs(cfg, with_v=False)
    planes, scales = oracle.plane_build(inp.K)
    plan = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, mode, budget)
    hp = torch.from_numpy(planes.view(np.int32)).pin_memory()
    hs = torch.from_numpy(scales.view(np.int16)).pin_memory()
    sentinel_p, sentinel_s = np.uint32(0xA5A5A5A5), np.uint16(0x5A5A)
    dp = torch.full(planes.shape, int(sentinel_p.view(np.int32)), dtype=torch.int32, device="cuda")
    ds = torch.full(scales.shape, int(sentinel_s.view(np.int16)), dtype=torch.int16, device="cuda")
    shp = sd.make_shape(cfg.B, cfg.Hq, cfg.Hkv, n)
    side = torch.cuda.Stream()
    plan_d = dev(plan)
    side.wait_stream(torch.cuda.current_stream())
    sd.sd_offload_gather(shp, hp, hs, plan_d, dp, ds, stream=side)
    done = torch.cuda.Event()
    done.record(side)
    sd.sd_event_wait(done, 30_000_000)
    torch.cuda.current_stream().wait_event(done)
    exp_p = np.full(planes.shape, sentinel_p, np.uint32)
    exp_s = np.full(scales.shape, sentinel_s, np.uint16)
    oracle.prefix_copy(planes, scales, plan, exp_p, exp_s)
    assert np.array_equal(host(dp, np.uint32), exp_p)
    assert np.array_equal(host(ds, np.uint16), exp_s)
    # the scan over the gathered prefixes matches the oracle's scores
    q = dev(inp.q)
    scores = torch.empty((cfg.B * cfg.Hkv, n), dtype=torch.float32, device="cuda")
    sd.sd_score(sd.SD_IDX_PLANES, shp, dp, ds, q, plan_d, scores)
    torch.cuda.synchronize()
    ref, l1 = oracle.plane_score(planes, scales, plan, inp.q, with_l1=True)
    check_scores(host(scores, np.float32).reshape(ref.shape), ref, l1, "offloaded scores")


def test_offload_rejects_pageable_memory(sd):
    cfg = synth.config(4, n=4096)
    shp = sd.make_shape(cfg.B, cfg.Hq, cfg.Hkv, cfg.n)
    pageable = np.zeros((cfg.Hkv, 128, 4, cfg.n // 32), np.uint32)
    sc = np.zeros((cfg.Hkv, 128, cfg.n // 64), np.uint16)
    plan = torch.zeros((1, cfg.Hkv, 128), dtype=torch.uint8, device="cuda")
    dp = torch.empty(pageable.shape, dtype=torch.int32, device="cuda")
    ds = torch.empty(sc.shape, dtype=torch.int16, device="cuda")
    with pytest.raises(sd.SdError) as ei:
        sd.sd_offload_gather(shp, pageable.ctypes.data, sc.ctypes.data, plan, dp, ds)
    assert ei.value.code == sd.SD_ERR_INVALID_ARG


def test_event_wait_times_out_then_completes(sd):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(200_000_000)  # a bounded busy kernel (~0.1 s)
    ev = torch.cuda.Event()
    ev.record(s)
    with pytest.raises(sd.SdError) as ei:
        sd.sd_event_wait(ev, 10)
    assert ei.value.code == sd.SD_ERR_TIMEOUT
    sd.sd_event_wait(ev, 30_000_000)
    assert ev.query()
