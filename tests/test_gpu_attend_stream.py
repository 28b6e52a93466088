"""GPU parity of the gather-attend over many long rows (the streaming kernel: every
warp an online softmax over its range of 16-token groups, K and V loaded straight
into tensor-core fragments, QK^T and PV as MMAs) against the oracle.

sd_gather_attend takes the streaming kernel when the rows hold at least 4 groups of
16 selected tokens per warp of a full grid (8 warps per SM): 256 or 512 rows of
hundreds of tokens here.  Cases: every G, ragged counts (0, 1, 15..17, 63..65, the
maximum, -1, above the maximum), skipped indices (< 0 or >= n), and NaN values in
V: unselected NaN rows must not reach any output, and a row that selects NaN
values must not leak them into the rows processed after it."""
import math

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


def run(sd, cfg, inp, idx, cnt, max_count, V=None):
    shp = sd.make_shape(cfg.B, cfg.Hq, cfg.Hkv, cfg.n, cfg.d)
    out = empty((cfg.B, cfg.Hq, cfg.d), np.float32)
    lse = empty((cfg.B, cfg.Hq), np.float32)
    ws = torch.empty(sd.sd_gather_attend_workspace_size(shp, max_count), dtype=torch.uint8,
                     device="cuda")
    sd.sd_gather_attend(shp, dev(inp.q), dev(inp.K), dev(inp.V if V is None else V), dev(idx),
                        idx.shape[1], dev(cnt), max_count, 1 / math.sqrt(cfg.d), out, lse, ws)
    torch.cuda.synchronize()
    sd.sd_device_status()
    return host(out, np.float32), host(lse, np.float32)


def oracle_of(cfg, inp, idx, cnt, max_count, V=None):
    """The oracle over each row's first min(count, max_count) entries, skipped
    indices removed (the library's reading of an out-of-range index)."""
    rows = cfg.B * cfg.Hkv
    ridx = np.zeros((rows, max(1, max_count)), np.int32)
    rcnt = np.zeros(rows, np.int32)
    for r in range(rows):
        c = max(0, min(int(cnt[r]), max_count))
        sel = idx[r, :c]
        sel = sel[(sel >= 0) & (sel < cfg.n)]
        ridx[r, :len(sel)] = sel
        rcnt[r] = len(sel)
    return oracle.gather_attend(inp.q, inp.K, inp.V if V is None else V,
                                ridx.reshape(cfg.B, cfg.Hkv, -1), rcnt.reshape(cfg.B, cfg.Hkv),
                                1 / math.sqrt(cfg.d))


def compare(o, l, ro, rl):
    nan = np.isnan(ro)
    assert np.array_equal(np.isnan(o), nan)
    err = np.abs(o[~nan] - ro[~nan]).max()
    assert err <= ATT_ATOL, err
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.abs(l[fin] - rl[fin]).max() <= 1e-4 * max(1.0, np.abs(rl[fin]).max())
    return err


EDGE_COUNTS = [0, 1, 15, 16, 17, 63, 64, 65, -1]


@pytest.mark.parametrize("G,B", [(4, 64), (1, 32), (2, 32), (8, 32)])
def test_stream_many_rows(sd, G, B):
    max_count = 400
    cfg = synth.config(1, B=B, Hq=8 * G, Hkv=8, n=2048 + 19)
    inp = synth.make_inputs(cfg)
    rows = cfg.B * cfg.Hkv
    idx, cnt = synth.make_index_lists(31 + G, rows, cfg.n, max_count)
    cnt = cnt.copy()
    cnt[:len(EDGE_COUNTS)] = EDGE_COUNTS
    cnt[len(EDGE_COUNTS)] = max_count
    cnt[len(EDGE_COUNTS) + 1] = max_count + 50  # clamped to max_count
    idx[len(EDGE_COUNTS)] = np.sort(np.random.default_rng(5).choice(cfg.n, max_count, False))
    idx[len(EDGE_COUNTS) + 1] = idx[len(EDGE_COUNTS)]
    # skipped indices inside the counted entries of some rows
    for r in range(20, rows, 37):
        c = int(cnt[r])
        if c > 4:
            idx[r, 1] = -5
            idx[r, c - 2] = cfg.n + 3
    o, l = run(sd, cfg, inp, idx, cnt, max_count)
    ro, rl = oracle_of(cfg, inp, idx, cnt, max_count)
    err = compare(o, l, ro, rl)
    print(f"G={G}: {rows} rows, max err {err:.2e}")


def test_stream_nan_rows_stay_in_their_row(sd):
    max_count = 200
    cfg = synth.config(1, B=64, Hq=32, Hkv=8, n=1024)
    inp = synth.make_inputs(cfg)
    rows = cfg.B * cfg.Hkv
    V = inp.V.copy()
    # tokens 0..255 of every head hold NaN values
    V[:, :, :256, 5] = 0x7FC0
    idx, cnt = synth.make_index_lists(77, rows, cfg.n, max_count)
    cnt = cnt.copy()
    for r in range(rows):
        if r % 3 == 0:  # selects NaN rows throughout
            idx[r, :max_count] = np.arange(max_count)
            cnt[r] = max_count
        else:  # ragged, NaN-free: the rows staged after a NaN row
            cnt[r] = 17 + (r % 5) * 16 + (r % 2)
            idx[r, :cnt[r]] = np.sort(np.random.default_rng(r).choice(
                np.arange(256, cfg.n), cnt[r], False))
    o, l = run(sd, cfg, inp, idx, cnt, max_count, V=V)
    ro, rl = oracle_of(cfg, inp, idx, cnt, max_count, V=V)
    compare(o, l, ro, rl)
    clean = np.repeat((np.arange(rows) % 3 != 0).reshape(cfg.B, cfg.Hkv), cfg.Hq // cfg.Hkv,
                      axis=1)
    assert np.isfinite(o[clean]).all()
    assert np.isnan(o[~clean][:, 5]).all()


@pytest.mark.slow
def test_stream_quest_blocks_full(sd):
    """Batch 64 x 8 KV heads x 16,384 tokens, 128 + 1 blocks of 16 tokens per row."""
    cfg = synth.config(3)
    inp = synth.make_inputs(cfg)
    rows = cfg.B * cfg.Hkv
    nb = 129
    rng = np.random.default_rng(3)
    idx = np.zeros((rows, nb * 16), np.int32)
    for r in range(rows):
        blocks = np.sort(rng.choice(cfg.n // 16 - 1, nb - 1, False))
        blocks = np.append(blocks, cfg.n // 16 - 1)
        idx[r] = (blocks[:, None] * 16 + np.arange(16)).reshape(-1)
    cnt = np.full(rows, nb * 16, np.int32)
    o, l = run(sd, cfg, inp, idx, cnt, nb * 16)
    ro, rl = oracle_of(cfg, inp, idx, cnt, nb * 16)
    err = compare(o, l, ro, rl)
    print(f"Quest blocks: max err {err:.2e}")
