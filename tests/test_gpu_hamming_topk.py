"""sd_hamming_topk (Hamming scan and top-k in two passes over the signatures, no
scores) against sd_score(SD_IDX_SIG) followed by sd_topk(SD_SCORE_I32), and against
the oracle's top-k of the oracle's Hamming scores: idx and count identical.  Random
32-bit signatures make ties the common case (a score takes one of 32G + 1 values)."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import empty, host

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


def run_both(sd, B, Hkv, G, n, ncap, k, sink, local, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    sig = torch.randint(-2**31, 2**31 - 1, (B, Hkv, ncap), generator=g, dtype=torch.int32,
                        device="cuda")
    qsig = torch.randint(-2**31, 2**31 - 1, (B, Hkv * G), generator=g, dtype=torch.int32,
                         device="cuda")
    shp = sd.make_shape(B, Hkv * G, Hkv, n, 128, ncap)
    sel = sd.make_select(k, sink, local, 1)
    rows = B * Hkv
    mc = min(n, sink + local + k)
    res = []
    for fused in (False, True):
        idx = torch.full((rows, mc), -7, dtype=torch.int32, device="cuda")
        cnt = empty((rows,), np.int32)
        if fused:
            nb = sd.sd_hamming_topk_workspace_size(shp, sel)
            ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
            sd.sd_hamming_topk(shp, sig, qsig, sel, idx, mc, cnt, ws)
        else:
            sc = torch.empty((rows, n), dtype=torch.int32, device="cuda")
            sd.sd_score(sd.SD_IDX_SIG, shp, sig, None, qsig, None, sc)
            tb = sd.sd_topk_workspace_size(rows, n, sel)
            tws = torch.empty(tb, dtype=torch.uint8, device="cuda") if tb else None
            sd.sd_topk(sd.SD_SCORE_I32, sc, rows, n, n, sel, idx, mc, cnt, tws)
        torch.cuda.synchronize()
        res.append((host(idx, np.int32), host(cnt, np.int32)))
    return res, host(sig, np.uint32), host(qsig, np.uint32)


def assert_same(res):
    (i1, c1), (i2, c2) = res
    assert np.array_equal(c1, c2), (c1, c2)
    for r in range(len(c1)):
        assert np.array_equal(i1[r, :c1[r]], i2[r, :c2[r]]), r


@pytest.mark.parametrize("B,Hkv,G,n,ncap,k,sink,local", [
    (1, 8, 4, 1048576, 1048576, 512, 0, 0),       # the 1M-token step's shape
    (1, 8, 4, 32768, 32768, 512, 128, 512),       # HashAttention's windows
    (2, 4, 8, 65536 + 8, 65536 + 64, 300, 5, 33),  # G = 8, windows cutting 4-token groups
    (1, 4, 1, 40000 + 3, 40000 + 3, 1000, 7, 1),  # G = 1, n % 4 != 0 (scalar loads)
    (1, 2, 2, 9000, 9000, 4096, 0, 0),            # k close to the competing count
    (1, 2, 4, 5000, 5000, 4096, 100, 100),        # k above it: everything competing
    (3, 2, 4, 8192 * 3 + 100, 8192 * 3 + 100, 64, 8191, 8193),
])
def test_hamming_topk_equals_two_calls(sd, B, Hkv, G, n, ncap, k, sink, local):
    res, _, _ = run_both(sd, B, Hkv, G, n, ncap, k, sink, local, 4000 + n % 977 + G)
    assert_same(res)


def test_hamming_topk_against_oracle(sd):
    B, Hkv, G, n, k, sink, local = 1, 2, 4, 20000, 256, 4, 64
    (_, (idx, cnt)), sig, qsig = run_both(sd, B, Hkv, G, n, n, k, sink, local, 4100)
    s = oracle.hamming_score(sig.reshape(B, Hkv, n), qsig).reshape(B * Hkv, n)
    ri, rc = oracle.topk(s, k, sink, local)
    for r in range(B * Hkv):
        assert cnt[r] == rc[r] and np.array_equal(idx[r, :cnt[r]], ri[r, :rc[r]]), r


def test_hamming_topk_repeat_calls(sd):
    # the workspace is reset by each call: a second call gives the same result
    a, _, _ = run_both(sd, 1, 4, 4, 100000, 100000, 512, 0, 0, 4200)
    b, _, _ = run_both(sd, 1, 4, 4, 100000, 100000, 512, 0, 0, 4200)
    assert_same([a[1], b[1]])
