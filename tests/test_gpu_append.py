"""sd_append_index (the KV-write path's incremental index update) against
sd_build_index over the grown length, bit for bit after every append, and against
the oracle at the end: one token at a time across 16- and 64-token block edges,
appends of many tokens at once, appends from an empty index, and the bit-plane
index over lengths that are not multiples of 64 (a partial last block)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import dev, host

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


KINDS = ["sig", "sig_mlp", "planes", "minmax", "landmark"]


def buffers(sd, kind, B, Hkv, ncap, fill):
    """Index buffers filled with a byte pattern (so unwritten parts show)."""
    def full(shape, dtype):
        t = torch.empty(int(np.prod(shape)) * np.dtype(dtype).itemsize, dtype=torch.uint8,
                        device="cuda")
        t.fill_(fill)
        return t
    if kind.startswith("sig"):
        return full((B, Hkv, ncap), np.uint32), None
    if kind == "planes":
        return full((B, Hkv, 128, 4, ncap // 32), np.uint32), full((B, Hkv, 128, ncap // 64),
                                                                 np.uint16)
    if kind == "landmark":
        return full((B, Hkv, (ncap + 7) // 8, 128), np.uint16), None
    return full((B, Hkv, (ncap + 15) // 16, 2, 128), np.uint16), None


def valid(kind, B, Hkv, ncap, n, o0, o1):
    """The parts of the index that describe tokens [0, n), as numpy arrays."""
    if kind.startswith("sig"):
        return [host(o0, np.uint8).view(np.uint32).reshape(B, Hkv, ncap)[:, :, :n]]
    if kind == "planes":
        nb = (n + 63) // 64
        p = host(o0, np.uint8).view(np.uint32).reshape(B, Hkv, 128, 4, ncap // 32)
        s = host(o1, np.uint8).view(np.uint16).reshape(B, Hkv, 128, ncap // 64)
        return [p[..., :2 * nb], s[..., :nb]]
    if kind == "landmark":
        nb = (n + 7) // 8
        lm = host(o0, np.uint8).view(np.uint16).reshape(B, Hkv, (ncap + 7) // 8, 128)
        return [lm[:, :, :nb]]
    nb = (n + 15) // 16
    m = host(o0, np.uint8).view(np.uint16).reshape(B, Hkv, (ncap + 15) // 16, 2, 128)
    return [m[:, :, :nb]]


def kind_id(sd, kind):
    return {"sig": sd.SD_IDX_SIG, "sig_mlp": sd.SD_IDX_SIG, "planes": sd.SD_IDX_PLANES,
            "minmax": sd.SD_IDX_MINMAX, "landmark": sd.SD_IDX_LANDMARK}[kind]


def setup(sd, kind, B, Hkv, ncap):
    cfg = synth.config(1 if kind == "sig_mlp" else 0, B=B, Hq=4 * Hkv, Hkv=Hkv, n=ncap)
    inp = synth.make_inputs(cfg, with_v=False)
    enc = None
    if kind.startswith("sig"):
        enc = sd.make_encoder(dev(inp.W1), dev(inp.b1),
                              dev(inp.W2) if inp.W2 is not None else None,
                              dev(inp.b2) if inp.b2 is not None else None)
    return inp, dev(inp.K), enc


def oracle_index(kind, inp, n):
    K = np.ascontiguousarray(inp.K[:, :, :n])
    if kind.startswith("sig"):
        return [oracle.sig_encode(K, inp.W1, inp.b1, inp.W2, inp.b2)]
    if kind == "planes":
        return list(oracle.plane_build(K))
    if kind == "landmark":
        return [oracle.landmark_build(K)]
    return [oracle.minmax_build(K)]


def equal(a, b):
    return len(a) == len(b) and all(np.array_equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("kind", KINDS)
def test_append_one_token_at_a_time(sd, kind):
    """n grows 1 per step across 16- and 64-token block edges; after every append
    the index equals a fresh build over the same n (each append is one launch)."""
    B, Hkv, ncap = 2, 2, 4224
    inp, K, enc = setup(sd, kind, B, Hkv, ncap)
    k = kind_id(sd, kind)
    n0 = 4030
    a0, a1 = buffers(sd, kind, B, Hkv, ncap, 0xA5)
    sd.sd_build_index(k, sd.make_shape(B, 4 * Hkv, Hkv, n0, 128, ncap), K, enc, a0, a1)
    for n in range(n0 + 1, 4100):
        before = sd.sd_launch_count()
        shp = sd.make_shape(B, 4 * Hkv, Hkv, n, 128, ncap)
        sd.sd_append_index(k, shp, n - 1, K, enc, a0, a1)
        assert sd.sd_launch_count() - before == 1
        f0, f1 = buffers(sd, kind, B, Hkv, ncap, 0x5A)
        sd.sd_build_index(k, shp, K, enc, f0, f1)
        torch.cuda.synchronize()
        assert equal(valid(kind, B, Hkv, ncap, n, a0, a1),
                     valid(kind, B, Hkv, ncap, n, f0, f1)), n
    assert equal(valid(kind, B, Hkv, ncap, 4099, a0, a1), oracle_index(kind, inp, 4099))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("steps", [[0, 1], [0, 64, 65, 1000, 1024, 1025, 3333, 4224],
                                   [17, 17, 18, 2049, 4160]])
def test_append_many_tokens(sd, kind, steps):
    """Appends of several tokens at once (from an empty index, within one block,
    across many tiles, up to n_cap, and n_old == n), checked against the oracle."""
    B, Hkv, ncap = 1, 3, 4224
    inp, K, enc = setup(sd, kind, B, Hkv, ncap)
    k = kind_id(sd, kind)
    a0, a1 = buffers(sd, kind, B, Hkv, ncap, 0xC3)
    n_old = steps[0]
    if n_old:
        sd.sd_build_index(k, sd.make_shape(B, 4 * Hkv, Hkv, n_old, 128, ncap), K, enc, a0, a1)
    for n in steps[1:]:
        before = sd.sd_launch_count()
        shp = sd.make_shape(B, 4 * Hkv, Hkv, n, 128, ncap)
        sd.sd_append_index(k, shp, n_old, K, enc, a0, a1)
        assert sd.sd_launch_count() - before == (1 if n > n_old else 0)
        torch.cuda.synchronize()
        assert equal(valid(kind, B, Hkv, ncap, n, a0, a1), oracle_index(kind, inp, n)), n
        n_old = n


@pytest.mark.parametrize("n", [1, 63, 64, 65, 127, 4095, 4161])
def test_plane_build_partial_block(sd, n):
    """sd_build_index(SD_IDX_PLANES) at any n: the partial last block against the
    oracle; words and scales of blocks past it are left as they were."""
    B, Hkv, ncap = 1, 2, 4224
    inp, K, _ = setup(sd, "planes", B, Hkv, ncap)
    p0, p1 = buffers(sd, "planes", B, Hkv, ncap, 0x77)
    sd.sd_build_index(sd.SD_IDX_PLANES, sd.make_shape(B, 4 * Hkv, Hkv, n, 128, ncap), K, None,
                      p0, p1)
    torch.cuda.synchronize()
    assert equal(valid("planes", B, Hkv, ncap, n, p0, p1), oracle_index("planes", inp, n))
    nb = (n + 63) // 64
    rest = host(p0, np.uint8).view(np.uint32).reshape(B, Hkv, 128, 4, ncap // 32)[..., 2 * nb:]
    assert (rest == 0x77777777).all()
    rest = host(p1, np.uint8).view(np.uint16).reshape(B, Hkv, 128, ncap // 64)[..., nb:]
    assert (rest == 0x7777).all()
