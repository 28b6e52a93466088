"""sd_select_attend (top-k from word maxima and gather-attend in one call) against
sd_topk_wmax followed by sd_gather_attend on the same inputs: idx and count must be
identical and out and lse identical bit for bit (both run the same device code on
the same partition of the selected rows), on the fused launch and on the two-call
path it takes where the fused launch does not apply; one case is also checked
against the oracle's attention."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import ATT_ATOL, dev, empty, host

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


def word_max(s: np.ndarray) -> np.ndarray:
    rows, n = s.shape
    return s.reshape(rows, n // 32, 32).max(axis=2)


def inputs(seed, B, Hkv, G, n, kind="f32", levels=0):
    rows = B * Hkv
    s = synth.make_scores(seed, rows, n, kind, levels)
    g = torch.Generator(device="cuda").manual_seed(seed)
    K = (torch.randn((B, Hkv, n, 128), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    V = torch.randn((B, Hkv, n, 128), generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn((B, Hkv * G, 128), generator=g, device="cuda").to(torch.bfloat16)
    return s, K, V, q


def both(sd, s, K, V, q, B, Hkv, G, n, k, sink=0, local=0):
    rows = B * Hkv
    shp = sd.make_shape(B, Hkv * G, Hkv, n, 128, n)
    sel = sd.make_select(k, sink, local, 1)
    mc = min(n, sink + local + k)
    scale = 1.0 / np.sqrt(128.0)
    sc, wm = dev(s), dev(np.ascontiguousarray(word_max(s), np.float32))
    res = []
    for fused in (False, True):
        idx = torch.full((rows, mc), -7, dtype=torch.int32, device="cuda")
        cnt = empty((rows,), np.int32)
        out = torch.full((B, Hkv * G, 128), 5.0, dtype=torch.float32, device="cuda")
        lse = torch.full((B, Hkv * G), 5.0, dtype=torch.float32, device="cuda")
        if fused:
            nb = sd.sd_select_attend_workspace_size(shp, sel, mc)
            ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
            sd.sd_select_attend(shp, sc, wm, sel, q, K, V, scale, idx, mc, cnt, mc, out, lse, ws)
        else:
            tb = sd.sd_topk_workspace_size(rows, n, sel)
            tws = torch.empty(tb, dtype=torch.uint8, device="cuda") if tb else None
            sd.sd_topk_wmax(sc, wm, rows, n, sel, idx, mc, cnt, tws)
            ab = sd.sd_gather_attend_workspace_size(shp, mc)
            aws = torch.empty(max(ab, 16), dtype=torch.uint8, device="cuda")
            sd.sd_gather_attend(shp, q, K, V, idx, mc, cnt, mc, scale, out, lse, aws)
        torch.cuda.synchronize()
        res.append((host(idx, np.int32), host(cnt, np.int32), host(out, np.float32),
                    host(lse, np.float32)))
    return res


def assert_same(res):
    (i1, c1, o1, l1), (i2, c2, o2, l2) = res
    assert np.array_equal(c1, c2), (c1, c2)
    for r in range(len(c1)):
        if c1[r] > 0:
            assert np.array_equal(i1[r, :c1[r]], i2[r, :c2[r]]), r
    assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32)), "out differs"
    assert np.array_equal(l1.view(np.uint32), l2.view(np.uint32)), "lse differs"


@pytest.mark.parametrize("B,Hkv,G,n,k,sink,local,kind,levels", [
    (1, 8, 4, 1048576, 512, 0, 0, "f32", 0),       # the 1M-token step's shape
    (1, 8, 4, 131072, 512, 128, 512, "f32", 0),    # sink and local windows
    (1, 4, 8, 65536, 256, 5, 33, "f32", 0),        # G = 8, windows cutting words
    (1, 8, 2, 65536, 300, 0, 0, "f32ties", 7),     # ties: the exact path in CTA 0
    (2, 4, 1, 65536, 1000, 0, 0, "f32", 0),        # G = 1, B = 2
    (4, 8, 4, 32768, 512, 0, 0, "f32", 0),         # 32 rows: beyond resident clusters
    (1, 2, 4, 16384, 512, 0, 0, "f32", 0),         # too few words: the two calls
])
def test_select_attend_equals_two_calls(sd, B, Hkv, G, n, k, sink, local, kind, levels):
    s, K, V, q = inputs(3000 + n % 991 + k + G, B, Hkv, G, n, kind, levels)
    assert_same(both(sd, s, K, V, q, B, Hkv, G, n, k, sink, local))


def test_select_attend_nan_row(sd):
    B, Hkv, G, n = 1, 8, 4, 65536
    s, K, V, q = inputs(3100, B, Hkv, G, n)
    s[3, 40000] = np.nan
    res = both(sd, s, K, V, q, B, Hkv, G, n, 512)
    assert res[1][1][3] == -1 and (res[1][1][np.arange(8) != 3] > 0).all()
    assert_same(res)


def test_select_attend_against_oracle(sd):
    B, Hkv, G, n, k = 1, 4, 4, 65536, 256
    s, K, V, q = inputs(3200, B, Hkv, G, n)
    (_, _, _, _), (idx, cnt, out, lse) = both(sd, s, K, V, q, B, Hkv, G, n, k, 4, 64)
    ri, rc = oracle.topk(s, k, 4, 64)
    for r in range(B * Hkv):
        assert cnt[r] == rc[r] and np.array_equal(idx[r, :cnt[r]], ri[r, :rc[r]])
    o_ref, lse_ref = oracle.gather_attend(host(q.view(torch.int16), np.int16).view(np.uint16),
                                          host(K.view(torch.int16), np.int16).view(np.uint16),
                                          host(V.view(torch.int16), np.int16).view(np.uint16),
                                          idx.reshape(B, Hkv, -1), cnt.reshape(B, Hkv),
                                          1.0 / np.sqrt(128.0))
    assert np.abs(out - o_ref).max() <= ATT_ATOL
