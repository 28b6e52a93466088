"""sd_gather_attend_noalloc: gather-attend for callers that cannot allocate device
memory or hand over a workspace (engines whose framework owns every device
allocation, real-time loops that must not take allocator locks or let cudaMalloc
synchronise the device).  When the split-n kernel runs, its partials live in
libsd's static per-GPU array instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row, on different problems,
and checks each result against sd_gather_attend with a caller workspace, within
the attention tolerance of the other parity tests: once as the GB300 runs it (the
16-CTA cluster kernel, which needs no scratch) and once with the split-n kernel
forced (sd_set_fallback_paths), and once on 256 rows, which take the streaming
kernel, so that both calls really write, and the second reuses, the shared array.  This file is collected last so that a run stopping at
the first failure has already run everything else; it also passes on its own in
a fresh process."""
import ctypes
import math

import numpy as np
import pytest
import torch

import synth
from _helpers import ATT_ATOL, dev, empty, host

NOALLOC_LIMIT = 4 << 20


@pytest.fixture(scope="module")
def sd():
    from top_sparse_decode_gb300 import build as b
    b.build()
    import top_sparse_decode_gb300 as m
    m.lib()
    return m


def test_noalloc_rejects_oversized_requests_before_any_cuda_call(sd):
    # 64 x 8 rows x 33 chunks of 4 query heads: ~35 MB of partials > 4 MiB
    shp = sd.make_shape(64, 32, 8, 16384)
    assert sd.sd_gather_attend_workspace_size(shp, 2064) > NOALLOC_LIMIT
    P = 1 << 20  # an aligned placeholder address; never dereferenced
    rc = sd.lib().sd_gather_attend_noalloc(ctypes.byref(shp), P, P, P, P, 2064, P, 2064, 0.1, P,
                                           None, None)
    assert rc == sd.SD_ERR_UNSUPPORTED
    assert "more than" in sd.sd_last_error()


# (G, Hkv, B, n, max_count) of the two calls: a few long rows (the cluster kernel, or
# the split-n kernel when forced), or 256 rows of 320 tokens (the streaming kernel,
# whose ticket and partials then live in the static array)
FEW_ROWS = [(4, 8, 2, 6000, 1152), (8, 3, 2, 3000, 700)]
MANY_ROWS = [(1, 8, 32, 4096, 320), (2, 8, 32, 4096, 320)]


@pytest.mark.gpu
@pytest.mark.parametrize("split_n,problems", [(False, FEW_ROWS), (True, FEW_ROWS),
                                              (False, MANY_ROWS)])
def test_noalloc_matches_workspace_entry_point_twice(sd, split_n, problems):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    prev = sd.sd_set_fallback_paths(split_n)
    try:
        _two_calls(sd, problems)
    finally:
        sd.sd_set_fallback_paths(prev)


def _two_calls(sd, problems):
    for trial, (G, Hkv, B, n, max_count) in enumerate(problems):
        cfg = synth.config(1, B=B, Hq=G * Hkv, Hkv=Hkv, n=n)
        inp = synth.make_inputs(cfg)
        rows = cfg.B * cfg.Hkv
        counts = np.linspace(1, max_count, rows).astype(np.int64)
        idx, cnt = synth.make_index_lists(70 + trial, rows, n, max_count, counts)
        shp = sd.make_shape(cfg.B, cfg.Hq, cfg.Hkv, n)
        need = sd.sd_gather_attend_workspace_size(shp, max_count)
        assert 0 < need <= NOALLOC_LIMIT
        q, K, V, I, C = dev(inp.q), dev(inp.K), dev(inp.V), dev(idx), dev(cnt)
        scale = 1 / math.sqrt(cfg.d)
        out_ref = empty((cfg.B, cfg.Hq, cfg.d), np.float32)
        lse_ref = empty((cfg.B, cfg.Hq), np.float32)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        sd.sd_gather_attend(shp, q, K, V, I, max_count, C, max_count, scale, out_ref, lse_ref, ws)
        out = torch.full((cfg.B, cfg.Hq, cfg.d), float("nan"), device="cuda")
        lse = torch.full((cfg.B, cfg.Hq), float("nan"), device="cuda")
        rc = sd.lib().sd_gather_attend_noalloc(
            ctypes.byref(shp), q.data_ptr(), K.data_ptr(), V.data_ptr(), I.data_ptr(), max_count,
            C.data_ptr(), max_count, ctypes.c_float(scale), out.data_ptr(), lse.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
        assert rc == sd.SD_OK, sd.sd_last_error()
        torch.cuda.synchronize()
        o, r = host(out, np.float32), host(out_ref, np.float32)
        assert np.isfinite(o).all()
        assert np.abs(o - r).max() <= ATT_ATOL
        lg, lr = host(lse, np.float32), host(lse_ref, np.float32)
        assert np.abs(lg - lr).max() <= 1e-4 * max(1.0, np.abs(lr).max())
