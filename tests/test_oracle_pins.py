"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties an oracle function to something other than itself: a worked
example printed on a page, a closed form or bound, a textbook or library routine
(sort, numpy float16 rounding, dense softmax), or brute force on tiny inputs.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bits_to_word(s: str) -> int:
    return sum(1 << i for i, ch in enumerate(s) if ch == "1")


# ---------------------------------------------------------------------------------
# Hamming score: HashAttention 2.2 worked example (T1)
# ---------------------------------------------------------------------------------
def test_hamming_worked_example():
    g = json.load(open(os.path.join(GOLD, "hamming_worked_example.json")))
    q = bits_to_word(g["query"])
    keys = [bits_to_word(k) for k in g["keys"]]
    for k, x in zip(keys, g["xor"]):
        assert (k ^ q) == bits_to_word(x)
    sig = np.array(keys, np.uint32).reshape(1, 1, -1)
    qsig = np.array([[q]], np.uint32)
    score = oracle.hamming_score(sig, qsig)
    assert (-score[0, 0]).tolist() == g["hamming"]
    idx, cnt = oracle.topk(score.reshape(1, -1), k=g["budget"])
    assert cnt[0] == g["budget"]
    assert idx[0, : cnt[0]].tolist() == g["selected"]


def test_hamming_matches_library_popcount_and_group_sum():
    rng_sig = (synth.uniform(7, 1, 3 * 2 * 300) * 2**32).astype(np.uint64).astype(np.uint32)
    rng_q = (synth.uniform(7, 2, 3 * 8) * 2**32).astype(np.uint64).astype(np.uint32)
    sig = rng_sig.reshape(3, 2, 300)
    qsig = rng_q.reshape(3, 8)  # G = 4
    s = oracle.hamming_score(sig, qsig)
    for b in range(3):
        for h in range(2):
            x = sig[b, h][:, None] ^ qsig[b, h * 4:(h + 1) * 4][None, :]
            ref = -np.bitwise_count(x).astype(np.int64).sum(axis=1)
            assert np.array_equal(s[b, h], ref)
    assert s.min() >= -32 * 4 and s.max() <= 0


# ---------------------------------------------------------------------------------
# Signatures: bits agree with a float64 evaluation wherever the margin exceeds the
# fp32 chain's error bound (HashAttention 2.2, eq. phi)
# ---------------------------------------------------------------------------------
@pytest.mark.parametrize("hidden", [0, 16])
def test_signature_bits_match_exact_sign(hidden):
    d = 128
    x = synth.normal_bf16(11, 1, 400, d)
    xf = synth.bf16_to_f64(x)
    if hidden == 0:
        W1 = synth.normal_f32(11, 2, (32, d), 1.0)
        b1 = synth.normal_f32(11, 3, (32,), 0.5)
        sig = oracle.sig_encode(x, W1, b1)
        pre = xf @ W1.astype(np.float64).T + b1
        mass = np.abs(xf) @ np.abs(W1.astype(np.float64)).T + np.abs(b1)
        rel = d * 2.0**-23
    else:
        W1 = synth.normal_f32(11, 4, (hidden, d), 1 / math.sqrt(d))
        b1 = synth.normal_f32(11, 5, (hidden,), 0.1)
        W2 = synth.normal_f32(11, 6, (32, hidden), 1 / math.sqrt(hidden))
        b2 = synth.normal_f32(11, 7, (32,), 0.1)
        sig = oracle.sig_encode(x, W1, b1, W2, b2)
        hid = np.maximum(xf @ W1.astype(np.float64).T + b1, 0.0)
        pre = hid @ W2.astype(np.float64).T + b2
        mass = (np.abs(xf) @ np.abs(W1.astype(np.float64)).T + np.abs(b1)) @ \
            np.abs(W2.astype(np.float64)).T + np.abs(b2)
        rel = (d + hidden) * 2.0**-22
    bits = ((sig[:, None] >> np.arange(32, dtype=np.uint32)[None, :]) & 1).astype(bool)
    sure = np.abs(pre) > rel * mass
    assert sure.mean() > 0.99
    assert np.array_equal(bits[sure], (pre > 0)[sure])


def test_signature_chain_is_ascending_fmaf_then_bias():
    """Hand-built rows on which the canonical chain -- acc = fma(w_j, x_j, acc), j
    ascending, then + bias -- and its plausible variants give opposite bits.
    (1 + 2^-7)(1 + 2^-23) = 1 + 2^-7 + 2^-23 + 2^-30 rounds to fp32 by dropping 2^-30.
    Against w_0 x_0 = -(1 + 2^-7 + 2^-23) the fused chain keeps +2^-30 (bit 1); a
    separate multiply and add, or the chain taken in descending j, cancels to 0
    (bit 0).  A bias of -1.5 * 2^-30 added after the chain gives -2^-31 (bit 0);
    added first it would vanish below half an ulp of the first product (bit 1)."""
    d = 128
    c = np.float32(1 + 2**-7 + 2**-23)
    w1 = np.float32(1 + 2**-23)
    assert float(c) == 1 + 2**-7 + 2**-23 and float(w1) == 1 + 2**-23
    x = np.zeros((1, d), np.uint16)
    x[0, 0], x[0, 1] = 0x3F80, 0x3F81  # bf16 1.0 and 1 + 2^-7
    W1 = np.zeros((32, d), np.float32)
    b1 = np.zeros(32, np.float32)
    W1[0, :2] = (-c, w1)   # fused ascending chain: +2^-30
    W1[1, :2] = (c, -w1)   # -2^-30
    W1[2, :2] = (-c, w1)
    b1[2] = np.float32(-1.5 * 2**-30)
    W1[3, 1] = w1          # a plain positive product
    sig = int(oracle.sig_encode(x, W1, b1)[0])
    assert [(sig >> o) & 1 for o in range(4)] == [1, 0, 0, 1]
    assert sig >> 4 == 0   # all-zero rows give +0 -> bit 0
    # the same residue through an MLP's hidden unit: ReLU(2^-30) = 2^-30 feeds
    # output 0 with weight 1; a mul+add hidden chain would feed 0
    hidden = 16
    H1 = np.zeros((hidden, d), np.float32)
    H1[0, :2] = (-c, w1)
    H2 = np.zeros((32, hidden), np.float32)
    H2[0, 0] = 1.0
    H2[1, 0] = -1.0
    sig2 = int(oracle.sig_encode(x, H1, np.zeros(hidden, np.float32), H2,
                                 np.zeros(32, np.float32))[0])
    assert sig2 == 1


def test_signature_zero_gives_zero_bit():
    d = 128
    x = np.zeros((2, d), np.uint16)
    x[1] = 0x8000  # -0.0
    W1 = synth.normal_f32(3, 1, (32, d), 1.0)
    sig = oracle.sig_encode(x, W1, np.zeros(32, np.float32))
    assert sig.tolist() == [0, 0]


# ---------------------------------------------------------------------------------
# Bit planes (Fathom "bit planes per channel")
# ---------------------------------------------------------------------------------
def test_f16_rounding_matches_numpy():
    u = synth.uniform(5, 1, 200000)
    # magnitudes from 2^-30 to 2^17 so subnormal, normal and overflow paths are hit
    x = (np.exp2(u * 47 - 30) * np.where(synth.uniform(5, 2, 200000) < 0.5, -1, 1)).astype(np.float32)
    extra = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 2**-24, 2**-25, 1.5 * 2**-25,
                      2**-14, 6.1e-5, 1.0 + 2**-11, 1.0 + 3 * 2**-11], np.float32)
    x = np.concatenate([x, extra])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)
    back = np.array([oracle.f16_to_f32(int(h)) for h in ref[:2000]], np.float32)
    assert np.array_equal(back, ref[:2000].view(np.float16).astype(np.float32))


def _decode_codes(planes):
    return ((planes[..., 0, :, None] >> np.arange(32, dtype=np.uint32)) & 1) * 8 + \
        ((planes[..., 1, :, None] >> np.arange(32, dtype=np.uint32)) & 1) * 4 + \
        ((planes[..., 2, :, None] >> np.arange(32, dtype=np.uint32)) & 1) * 2 + \
        ((planes[..., 3, :, None] >> np.arange(32, dtype=np.uint32)) & 1)


def test_plane_codes_are_nearest_grid_points_all_bf16():
    """Brute force over every finite bf16 value in range against one scale: the
    code is the nearest point of the grid s*(c-8), ties to the even rint."""
    all_bf16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        vals = synth.bf16_to_f64(all_bf16)
    finite = np.isfinite(vals)
    # one 64-token block per channel: put the block absmax 7*s at token 0
    s_target = 0.375  # exact in f16; absmax = 2.625 is exact in bf16
    amax = np.float64(7 * s_target)
    sel = all_bf16[finite & (np.abs(vals) <= amax)]
    n_tok = 64 * ((len(sel) + 62) // 63)
    d = 1
    K = np.zeros((1, 1, n_tok, d), np.uint16)
    flat = K.reshape(-1)
    # each block: token 0 holds +absmax, the other 63 hold values under test
    vals_iter = list(sel)
    pos = 0
    for blk in range(n_tok // 64):
        flat[blk * 64] = synth.to_bf16(np.array([amax]))[0]
        for t in range(1, 64):
            flat[blk * 64 + t] = vals_iter[pos] if pos < len(vals_iter) else 0
            pos += 1
    planes, scales = oracle.plane_build(K)
    assert np.all(scales == np.float16(s_target).view(np.uint16))
    codes = _decode_codes(planes)[0, 0, 0].reshape(-1)
    k = synth.bf16_to_f64(flat)
    grid = s_target * (np.arange(16) - 8.0)
    dist = np.abs(k[:, None] - grid[None, :])
    best = dist.min(axis=1)
    assert np.all(dist[np.arange(len(k)), codes] == best)
    tie = (dist == best[:, None]).sum(axis=1) > 1
    # ties only between two neighbours: rint picks the even (k/s) integer, i.e. even code
    assert np.all(codes[tie] % 2 == 0)


def test_plane_scale_rule_and_prefix_invariant():
    cfg = synth.config(0, n=256)
    inp = synth.make_inputs(cfg, with_v=False)
    planes, scales = oracle.plane_build(inp.K)
    K = synth.bf16_to_f64(inp.K)[0, 0]  # [n][d]
    n, d = K.shape
    # scale = f16_rn(absmax/7) computed in fp32, via numpy's own float16 rounding
    amax = np.abs(K.reshape(n // 64, 64, d)).max(axis=1).astype(np.float32)  # [nb][d]
    s_ref = (amax / np.float32(7)).astype(np.float16)
    s_ref[s_ref == 0] = 1
    assert np.array_equal(scales[0, 0].T, s_ref.view(np.uint16))
    codes = _decode_codes(planes)[0, 0].reshape(d, n)
    s = np.repeat(s_ref.astype(np.float64), 64, axis=0).T  # [d][n]
    # 4-bit dequantisation error bound |k - s(c-8)| <= s/2 (inside the clamp range)
    assert np.all(np.abs(K.T - s * (codes - 8.0)) <= s / 2 * (1 + 1e-12))
    # prefix invariant: the first t planes are the t-bit code, and the midpoint
    # reconstruction of [-8s, 8s) cut into 2^t bins stays within half a t-bit step
    for t in range(5):
        pref = (codes >> (4 - t)) << (4 - t)
        for c, p, sv in [(int(codes[j, i]), int(pref[j, i]), float(s[j, i]))
                         for j in (0, 5, 77) for i in (0, 63, 64, 200)]:
            khat = oracle.reconstruct(p, t, sv)
            khat4 = oracle.reconstruct(c, 4, sv)
            assert khat4 == sv * (c - 8)
            if t == 0:
                assert khat == 0.0
            if t < 4:
                width = sv * 2 ** (4 - t)
                assert khat == pytest.approx(-8 * sv + (p >> (4 - t)) * width + width / 2)
                assert abs(khat - khat4) <= sv * 2 ** (3 - t)


@pytest.mark.parametrize("n", [5, 64 * 2 + 37, 64 * 3 + 63])
def test_plane_partial_block_rule(n):
    """A last block holding r < 64 tokens: its scale is f16_rn(absmax/7) over those r
    tokens (numpy's float16 rounding), their codes are within half a step, the bits
    of the positions past n are zero, and the full blocks before it do not depend on
    the tokens after them (appending keys never changes a closed block)."""
    cfg = synth.config(0, n=256)
    inp = synth.make_inputs(cfg, with_v=False)
    Kn = np.ascontiguousarray(inp.K[:, :, :n])
    planes, scales = oracle.plane_build(Kn)
    nb = (n + 63) // 64
    assert planes.shape[-1] == 2 * nb and scales.shape[-1] == nb
    K = synth.bf16_to_f64(Kn)[0, 0]  # [n][d]
    d = K.shape[1]
    c0 = (nb - 1) * 64
    amax = np.abs(K[c0:]).max(axis=0).astype(np.float32)
    s_ref = (amax / np.float32(7)).astype(np.float16)
    s_ref[s_ref == 0] = 1
    assert np.array_equal(scales[0, 0, :, nb - 1], s_ref.view(np.uint16))
    codes = _decode_codes(planes)[0, 0].reshape(d, -1)  # [d][64 nb]
    s = s_ref.astype(np.float64)[:, None]
    assert np.all(np.abs(K[c0:].T - s * (codes[:, c0:n] - 8.0)) <= s / 2 * (1 + 1e-12))
    assert not codes[:, n:].any()  # padding: every plane bit past n is 0
    if nb > 1:
        pf, sf = oracle.plane_build(np.ascontiguousarray(inp.K[:, :, :c0]))
        assert np.array_equal(planes[..., :2 * (nb - 1)], pf)
        assert np.array_equal(scales[..., :nb - 1], sf)


def test_plane_zero_block_scale_is_one():
    K = np.zeros((1, 1, 64, 128), np.uint16)
    planes, scales = oracle.plane_build(K)
    assert np.all(scales == 0x3C00)
    codes = _decode_codes(planes)[0, 0]
    assert np.all(codes == 8)


# ---------------------------------------------------------------------------------
# Water-filling plan (Fathom "per-query reverse water-filling")
# ---------------------------------------------------------------------------------
def _brute_plan_objective(w, B):
    best = -1.0
    for alloc in itertools.product(range(5), repeat=len(w)):
        if sum(alloc) != B:
            continue
        val = sum(wj * (1 - 4.0 ** -bj) for wj, bj in zip(w, alloc))
        best = max(best, val)
    return best


def _gains(q, sigma2, h, G):
    qf = synth.bf16_to_f64(q).astype(np.float32)
    acc = np.zeros(q.shape[-1], np.float32)
    for g in range(G):
        acc = acc + qf[0, h * G + g] * qf[0, h * G + g]
    return (acc * sigma2[h]).astype(np.float64)


@pytest.mark.parametrize("d,G", [(4, 1), (5, 2), (6, 4)])
def test_waterfill_is_optimal_by_brute_force(d, G):
    for trial in range(3):
        q = synth.normal_bf16(100 + trial, 1, G, d).reshape(1, G, d)
        sigma2 = (synth.uniform(100 + trial, 2, d) * 4 + 0.01).astype(np.float32).reshape(1, d)
        w = _gains(q, sigma2, 0, G)
        prev = np.zeros(d, np.int64)
        for B in range(0, 4 * d + 3):
            p = oracle.plan(q, sigma2, 1, oracle.PLAN_WATERFILL, B)[0, 0].astype(np.int64)
            assert p.sum() == min(B, 4 * d) and p.max() <= 4
            assert np.all(p >= prev)  # nested in B
            prev = p
            if B <= 4 * d:
                val = float(np.sum(w * (1 - 4.0 ** -p)))
                assert val == pytest.approx(_brute_plan_objective(w, B), rel=1e-12, abs=1e-300)


@pytest.mark.parametrize("Hkv,d,G", [(2, 2, 1), (2, 3, 2), (3, 2, 2)])
def test_budget_split_is_optimal_by_brute_force(Hkv, d, G):
    """The cross-head split (Fathom's marginal-gain rule over every KV head of a
    sequence under their summed budget) maximises sum over (h, j) of
    w_hj (1 - 4^-b_hj) among all allocations of Hkv * B bits: brute force over
    every allocation; nested in B; the bits of every head within [0, 4]."""
    for trial in range(2):
        q = synth.normal_bf16(300 + trial, 1, Hkv * G, d).reshape(1, Hkv * G, d)
        sigma2 = (synth.uniform(300 + trial, 2, Hkv * d) * 4 + 0.01).astype(np.float32)
        sigma2 = sigma2.reshape(Hkv, d)
        w = np.concatenate([_gains(q, sigma2, h, G) for h in range(Hkv)])
        prev = np.zeros(Hkv * d, np.int64)
        for B in range(0, 4 * d + 1):
            p = oracle.plan(q, sigma2, Hkv, oracle.PLAN_SPLIT, B)[0].reshape(-1).astype(np.int64)
            assert p.sum() == Hkv * B and p.max() <= 4
            assert np.all(p >= prev)
            prev = p
            val = float(np.sum(w * (1 - 4.0 ** -p)))
            assert val == pytest.approx(_brute_plan_objective(w, Hkv * B), rel=1e-12, abs=1e-300)


def test_budget_split_one_head_is_waterfill_and_moves_bits_between_heads():
    cfg = synth.config(2, B=2, Hq=8, Hkv=2, n=64)
    inp = synth.make_inputs(cfg, with_v=False)
    q1 = np.ascontiguousarray(inp.q[:, :4])
    s1 = np.ascontiguousarray(inp.sigma2[:1])
    for B in (0, 7, 56, 300, 512):
        assert np.array_equal(oracle.plan(q1, s1, 1, oracle.PLAN_SPLIT, B),
                              oracle.plan(q1, s1, 1, oracle.PLAN_WATERFILL, B))
    # a head whose gains are 16x larger takes more of the shared budget
    s2 = inp.sigma2.copy()
    s2[1] *= 16.0
    p = oracle.plan(inp.q, s2, 2, oracle.PLAN_SPLIT, 56).astype(np.int64)
    per_head = p.sum(axis=-1)
    assert np.all(per_head.sum(axis=-1) == 2 * 56)
    assert np.all(per_head[:, 1] > per_head[:, 0])


def test_budget_split_ties_go_to_lower_head_then_channel():
    # every gain equal: the bits go to head 0's channels first (lower j first, each
    # channel's b = 0 pairs before any b = 1), then head 1's
    d, G, Hkv = 4, 1, 2
    q = np.full((1, Hkv * G, d), 0x3F80, np.uint16)  # bf16 1.0
    sigma2 = np.ones((Hkv, d), np.float32)
    p = oracle.plan(q, sigma2, Hkv, oracle.PLAN_SPLIT, 3)[0]
    # 6 bits of equal gain at b = 0: head 0 channels 0..3, then head 1 channels 0..1
    assert p.tolist() == [[1, 1, 1, 1], [1, 1, 0, 0]]


def test_waterfill_ties_go_to_lower_channel():
    d = 4
    q = np.zeros((1, 1, d), np.uint16)
    q[0, 0] = synth.to_bf16(np.array([1.0, 1.0, 2.0, 0.0]))
    sigma2 = np.array([[1.0, 1.0, 0.25, 3.0]], np.float32)  # gains 1, 1, 1, 0
    got = [oracle.plan(q, sigma2, 1, oracle.PLAN_WATERFILL, B)[0, 0].tolist() for B in range(8)]
    assert got[1] == [1, 0, 0, 0]
    assert got[3] == [1, 1, 1, 0]
    assert got[4] == [2, 1, 1, 0]
    assert got[7] == [3, 2, 2, 0]
    # an exact tie between a second bit of channel 0 (w/4) and a first bit of channel 1
    q[0, 0] = synth.to_bf16(np.array([2.0, 1.0, 0.0, 0.0]))
    sigma2 = np.array([[1.0, 1.0, 1.0, 1.0]], np.float32)  # gains 4, 1, 0, 0
    assert oracle.plan(q, sigma2, 1, oracle.PLAN_WATERFILL, 2)[0, 0].tolist() == [2, 0, 0, 0]
    assert oracle.plan(q, sigma2, 1, oracle.PLAN_WATERFILL, 3)[0, 0].tolist() == [2, 1, 0, 0]
    # zero gains: bits go to the lowest channels, 4 at a time
    q[:] = 0
    assert oracle.plan(q, sigma2, 1, oracle.PLAN_WATERFILL, 6)[0, 0].tolist() == [4, 2, 0, 0]


def test_fixed_and_full_plans():
    cfg = synth.config(4, n=64, B=2)
    inp = synth.make_inputs(cfg, with_v=False)
    p = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, oracle.PLAN_FIXED, 32)
    for h in range(cfg.Hkv):
        top = np.argsort(-inp.sigma2[h].astype(np.float64), kind="stable")[:32]
        ref = np.zeros(cfg.d, np.uint8)
        ref[top] = 4
        assert np.array_equal(p[0, h], ref) and np.array_equal(p[1, h], ref)
    f = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, oracle.PLAN_FULL, 0)
    assert np.all(f == 4)


def test_topq_plan_is_sparq_rule():
    """SparQ-style plan: with one query head per group it is exactly the top-r |q_j|
    rule (q^2 of a bf16 value is exact in fp32, so the ranking is |q|'s), ties to
    the lower channel; with a group, every planned channel's query mass is at least
    every unplanned one's, r channels get 4 bits, the rest 0."""
    cfg = synth.config(4, n=64, B=2, Hq=8, Hkv=8)  # G = 1
    inp = synth.make_inputs(cfg, with_v=False)
    p = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, oracle.PLAN_TOPQ, 17)
    qf = synth.bf16_to_f64(inp.q)
    for b in range(cfg.B):
        for h in range(cfg.Hkv):
            top = np.argsort(-np.abs(qf[b, h]), kind="stable")[:17]
            ref = np.zeros(cfg.d, np.uint8)
            ref[top] = 4
            assert np.array_equal(p[b, h], ref), (b, h)
    cfg = synth.config(4, n=64, B=1)  # G = 4
    inp = synth.make_inputs(cfg, with_v=False)
    p = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, oracle.PLAN_TOPQ, 17)
    qf = synth.bf16_to_f64(inp.q).reshape(cfg.B, cfg.Hkv, cfg.G, cfg.d)
    u = (qf ** 2).sum(axis=2)  # exact in double
    for h in range(cfg.Hkv):
        sel = p[0, h] == 4
        assert sel.sum() == 17 and set(np.unique(p[0, h])) <= {0, 4}
        assert u[0, h][sel].min() >= u[0, h][~sel].max()
    # budgets 0 and d
    assert np.all(oracle.plan(inp.q, inp.sigma2, cfg.Hkv, oracle.PLAN_TOPQ, 0) == 0)
    assert np.all(oracle.plan(inp.q, inp.sigma2, cfg.Hkv, oracle.PLAN_TOPQ, cfg.d) == 4)


# ---------------------------------------------------------------------------------
# Bit-plane score
# ---------------------------------------------------------------------------------
def test_plane_score_full_plan_is_dequantised_dot_and_bounded():
    cfg = synth.config(0, n=512)
    inp = synth.make_inputs(cfg, with_v=False)
    planes, scales = oracle.plane_build(inp.K)
    full = oracle.plan(inp.q, inp.sigma2, 1, oracle.PLAN_FULL, 0)
    sc = oracle.plane_score(planes, scales, full, inp.q)[0, 0]
    qf = synth.bf16_to_f64(inp.q)[0]          # [G][d]
    Kf = synth.bf16_to_f64(inp.K)[0, 0]       # [n][d]
    sv = np.repeat(scales[0, 0].view(np.float16).astype(np.float64), 64, axis=1).T  # [n][d]
    exact = Kf @ qf.sum(axis=0)
    bound = (sv / 2) @ np.abs(qf).sum(axis=0)
    assert np.all(np.abs(sc - exact) <= bound * (1 + 1e-9))
    zero = oracle.plan(inp.q, inp.sigma2, 1, oracle.PLAN_WATERFILL, 0)
    assert np.all(oracle.plane_score(planes, scales, zero, inp.q) == 0.0)


def test_plane_score_single_channel_prefix():
    cfg = synth.config(0, n=128)
    inp = synth.make_inputs(cfg, with_v=False)
    planes, scales = oracle.plane_build(inp.K)
    qf = synth.bf16_to_f64(inp.q)[0]
    codes = _decode_codes(planes)[0, 0].reshape(cfg.d, cfg.n)
    for j, t in [(3, 1), (9, 2), (40, 3), (127, 4)]:
        p = np.zeros((1, 1, cfg.d), np.uint8)
        p[0, 0, j] = t
        sc = oracle.plane_score(planes, scales, p, inp.q)[0, 0]
        sv = np.repeat(scales[0, 0, j].view(np.float16).astype(np.float64), 64)
        pref = (codes[j] >> (4 - t)) << (4 - t)
        width = sv * 2.0 ** (4 - t)
        if t < 4:   # midpoint of bin (pref >> (4-t)) of [-8s, 8s) cut into 2^t bins
            mid = -8 * sv + (pref >> (4 - t)) * width + width / 2
        else:       # the 4-bit grid value
            mid = sv * (codes[j] - 8.0)
        assert np.allclose(sc, qf[:, j].sum() * mid, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------------
# Quest bound (OasisKV prerequisites: Quest-style block summaries)
# ---------------------------------------------------------------------------------
def test_minmax_matches_library_reductions():
    cfg = synth.config(0, n=200)  # ragged tail block
    inp = synth.make_inputs(cfg, with_v=False)
    summ = oracle.minmax_build(inp.K)
    Kf = synth.bf16_to_f64(inp.K)[0, 0]
    for c in range(summ.shape[2]):
        blk = Kf[c * 16: min((c + 1) * 16, cfg.n)]
        assert np.array_equal(synth.bf16_to_f64(summ[0, 0, c, 0]), blk.min(axis=0))
        assert np.array_equal(synth.bf16_to_f64(summ[0, 0, c, 1]), blk.max(axis=0))


def test_minmax_signed_zero_rule():
    K = np.zeros((1, 1, 16, 128), np.uint16)
    K[0, 0, 3, 0] = 0x8000  # one -0.0 among +0.0
    summ = oracle.minmax_build(K)
    assert summ[0, 0, 0, 0, 0] == 0x8000 and summ[0, 0, 0, 1, 0] == 0x0000


def test_quest_bound_dominates_every_in_block_dot():
    cfg = synth.config(3, B=2, Hkv=2, Hq=8, n=16 * 40 + 5, planted=3)
    inp = synth.make_inputs(cfg, with_v=False)
    summ = oracle.minmax_build(inp.K)
    U = oracle.quest_score(summ, inp.q)
    qf = synth.bf16_to_f64(inp.q)
    Kf = synth.bf16_to_f64(inp.K)
    G = cfg.G
    for b in range(cfg.B):
        for h in range(cfg.Hkv):
            qs = qf[b, h * G:(h + 1) * G].sum(axis=0)
            dots = Kf[b, h] @ qs
            for c in range(U.shape[2]):
                blk = dots[c * 16: min((c + 1) * 16, cfg.n)]
                assert np.all(blk <= U[b, h, c] + 1e-9 * (1 + abs(U[b, h, c])))
    # tightness: a block of identical keys gives exactly their dot
    K1 = np.repeat(inp.K[:1, :1, :1], 16, axis=2)
    U1 = oracle.quest_score(oracle.minmax_build(K1), inp.q[:1, :G])
    assert U1[0, 0, 0] == pytest.approx(float(Kf[0, 0, 0] @ qf[0, :G].sum(axis=0)), rel=1e-12)


def _khat_by_bins(planes, scales, plan_, n):
    """khat_ij(t_j) [B][Hkv][d][n] decoded by numpy from the planes: the first t_j
    planes give the bin (code >> (4 - t)) of [-8 s, 8 s) cut into 2^t bins; the
    reconstruction is its midpoint for t < 4 and the 4-bit grid value s (code - 8)
    for t = 4 (an unread channel, t = 0, is the midpoint of [-8 s, 8 s), 0)."""
    codes = _decode_codes(planes)
    B, Hkv, d = planes.shape[:3]
    codes = codes.reshape(B, Hkv, d, -1)[..., :n].astype(np.int64)
    s = np.repeat(scales.view(np.float16).astype(np.float64), 64, axis=-1)[..., :n]
    t = plan_.astype(np.int64)[..., None]
    width = s * 2.0 ** (4 - t)
    mid = -8 * s + (codes >> (4 - t)) * width + width / 2
    return np.where(t == 4, s * (codes - 8.0), mid)


@pytest.mark.parametrize("n,mode,budget", [(64 * 5, oracle.PLAN_WATERFILL, 56),
                                           (64 * 5 + 23, oracle.PLAN_WATERFILL, 92),
                                           (64 * 3 + 1, oracle.PLAN_WATERFILL, 7),
                                           (64 * 4 + 40, "random", 0)])
def test_plane_score_and_l1_mass_by_numpy_decoding(n, mode, budget):
    """The bit-plane score sum_g sum_j q_gj khat_ij(t_j) and its tolerance mass
    sum_g sum_j |q_gj khat_ij(t_j)| against numpy over independently decoded
    codes, for water-filled and arbitrary plans, with a partial last block.  A
    mass formed from |q~_j| (group-summed first), or from |q| |s| 8, or with a term
    dropped, fails here."""
    cfg = synth.config(0, n=n, B=2, Hq=8, Hkv=2)
    inp = synth.make_inputs(cfg, with_v=False)
    planes, scales = oracle.plane_build(inp.K)
    if mode == "random":
        u = synth.uniform(77, 1, cfg.B * cfg.Hkv * cfg.d)
        plan_ = np.floor(u * 5).astype(np.uint8).reshape(cfg.B, cfg.Hkv, cfg.d)
    else:
        plan_ = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, mode, budget)
    sc, l1 = oracle.plane_score(planes, scales, plan_, inp.q, with_l1=True, n=n)
    kh = _khat_by_bins(planes, scales, plan_, n)                    # [B][H][d][n]
    q = synth.bf16_to_f64(inp.q).reshape(cfg.B, cfg.Hkv, cfg.G, cfg.d)
    ref = np.einsum("bhgj,bhjn->bhn", q, kh)
    mass = np.einsum("bhgj,bhjn->bhn", np.abs(q), np.abs(kh))
    assert np.allclose(sc, ref, rtol=0, atol=1e-12 * mass.max())
    assert np.allclose(l1, mass, rtol=1e-12, atol=0)
    # the mass is not the looser |q~| form unless every group's signs agree
    qt = np.abs(q.sum(axis=2))
    loose = np.einsum("bhj,bhjn->bhn", qt, np.abs(kh))
    assert np.all(l1 >= loose * (1 - 1e-12)) and np.any(l1 > loose * (1 + 1e-6))


def test_quest_l1_mass_is_sum_of_abs_bound_terms():
    """The Quest tolerance mass sum_g sum_j |max(q_gj min_j, q_gj max_j)| against
    numpy over the summaries; it bounds |U| and equals U on a block whose every
    term is non-negative (q and the keys of one sign)."""
    cfg = synth.config(3, B=2, Hkv=2, Hq=8, n=16 * 9 + 3, planted=2)
    inp = synth.make_inputs(cfg, with_v=False)
    summ = oracle.minmax_build(inp.K)
    U, l1 = oracle.quest_score(summ, inp.q, with_l1=True)
    q = synth.bf16_to_f64(inp.q).reshape(cfg.B, cfg.Hkv, cfg.G, 1, cfg.d)
    mn = synth.bf16_to_f64(summ[:, :, :, 0])[:, :, None]   # [B][H][1][c][d]
    mx = synth.bf16_to_f64(summ[:, :, :, 1])[:, :, None]
    terms = np.maximum(q * mn, q * mx)                      # [B][H][G][c][d]
    assert np.allclose(U, terms.sum(axis=(2, 4)), rtol=0, atol=1e-12 * np.abs(terms).sum())
    assert np.allclose(l1, np.abs(terms).sum(axis=(2, 4)), rtol=1e-12, atol=0)
    assert np.all(np.abs(U) <= l1 * (1 + 1e-12))
    Kp = np.abs(synth.bf16_to_f64(inp.K[:1, :1, :16]))
    qp = np.abs(synth.bf16_to_f64(inp.q[:1, :cfg.G]))
    Up, lp = oracle.quest_score(oracle.minmax_build(synth.to_bf16(Kp)), synth.to_bf16(qp),
                                with_l1=True)
    assert Up[0, 0, 0] == pytest.approx(lp[0, 0, 0], rel=1e-12)


# ---------------------------------------------------------------------------------
# Top-k with forced windows (HashAttention 2.1 TOPK, 3.1; OasisKV method details)
# ---------------------------------------------------------------------------------
def _brute_topk(s, k, sink, local, block, n_tokens):
    n = len(s)
    lead = min(sink, n)
    tail = max(n - local, lead)
    cand = list(range(lead, tail))
    if len(cand) > k:
        cand = sorted(cand, key=lambda u: (-float(s[u]), u))[:k]
    units = sorted(list(range(lead)) + cand + list(range(tail, n)))
    out = []
    for u in units:
        out.extend(range(u * block, min((u + 1) * block, n_tokens)))
    return out


@pytest.mark.parametrize("kind", ["f32", "f32ties", "int", "const"])
def test_topk_brute_force_small(kind):
    for n in [1, 5, 17, 40, 130]:
        s = synth.make_scores(31 + n, 4, n, kind, levels=5)
        for k, sink, local in [(1, 0, 0), (3, 2, 2), (8, 0, 4), (50, 4, 4), (200, 1, 1)]:
            idx, cnt = oracle.topk(s, k, sink, local)
            for r in range(4):
                ref = _brute_topk(s[r], k, sink, local, 1, n)
                assert cnt[r] == len(ref)
                assert idx[r, :cnt[r]].tolist() == ref


def test_topk_block_mode_and_ragged_tail():
    s = synth.make_scores(5, 3, 21, "f32").astype(np.float64)
    n_tokens = 16 * 20 + 7
    idx, cnt = oracle.topk(s, k=4, sink=0, local=1, block=16, n_tokens=n_tokens)
    for r in range(3):
        ref = _brute_topk(s[r], 4, 0, 1, 16, n_tokens)
        assert cnt[r] == 4 * 16 + 7 and idx[r, :cnt[r]].tolist() == ref


def test_topk_all_ties_take_lowest_indices_and_signed_zero():
    s = np.zeros((2, 100), np.float32)
    s[1, ::2] = np.float32(-0.0)
    idx, cnt = oracle.topk(s, k=10)
    assert idx[0, :10].tolist() == list(range(10)) and idx[1, :10].tolist() == list(range(10))


def test_topk_nan_row_reports_error():
    s = np.zeros((2, 50), np.float32)
    s[1, 7] = np.nan
    _, cnt = oracle.topk(s, k=5)
    assert cnt[0] == 5 and cnt[1] == -1


def test_budget_arithmetic_hashattention_and_oasiskv():
    g = json.load(open(os.path.join(GOLD, "byte_model.json")))
    n, m, fixed = g["n"], g["m"], g["fixed"]
    assert n // g["sparsity"] == m
    s = synth.make_scores(9, 1, n, "f32")
    _, cnt = oracle.topk(s, k=m, sink=fixed // 2, local=fixed // 2)
    assert cnt[0] == g["total"]
    assert round(100.0 * cnt[0] / n, 2) == g["read_fraction_pct"]
    nblk = 1024
    sb = synth.make_scores(10, 1, nblk, "f32")
    _, cb = oracle.topk(sb, k=g["blocks"] - 1, local=1, block=g["block_tokens"],
                        n_tokens=nblk * 16)
    assert cb[0] == g["tokens_per_head"]


# ---------------------------------------------------------------------------------
# Gather-attend (HashAttention 2.1, corrected o_hat)
# ---------------------------------------------------------------------------------
def test_gather_attend_full_set_equals_dense_softmax():
    cfg = synth.config(0, n=300, Hq=8, Hkv=2)
    inp = synth.make_inputs(cfg)
    B, Hkv, n = cfg.B, cfg.Hkv, cfg.n
    idx = np.tile(np.arange(n, dtype=np.int32), (B, Hkv, 1))
    cnt = np.full((B, Hkv), n, np.int32)
    scale = 1 / math.sqrt(cfg.d)
    o, lse = oracle.gather_attend(inp.q, inp.K, inp.V, idx, cnt, scale)
    qf, Kf, Vf = (synth.bf16_to_f64(x) for x in (inp.q, inp.K, inp.V))
    for g in range(cfg.Hq):
        h = g // cfg.G
        z = Kf[0, h] @ qf[0, g] * scale
        a = np.exp(z - z.max())
        ref = (a / a.sum()) @ Vf[0, h]
        assert np.allclose(o[0, g], ref, rtol=1e-12, atol=1e-12)
        assert lse[0, g] == pytest.approx(z.max() + math.log(a.sum()), rel=1e-12)


def test_gather_attend_single_row_and_empty():
    cfg = synth.config(0, n=64)
    inp = synth.make_inputs(cfg)
    idx = np.array([[[17, -1]]], np.int32)
    o, lse = oracle.gather_attend(inp.q, inp.K, inp.V, idx, np.array([[1]], np.int32), 0.1)
    v = synth.bf16_to_f64(inp.V)[0, 0, 17]
    assert np.array_equal(o[0, 0], v) and np.array_equal(o[0, 3], v)
    o, lse = oracle.gather_attend(inp.q, inp.K, inp.V, idx, np.array([[0]], np.int32), 0.1)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_prefix_copy_copies_exactly_the_planned_prefix():
    cfg = synth.config(0, n=128)
    inp = synth.make_inputs(cfg, with_v=False)
    planes, scales = oracle.plane_build(inp.K)
    p = oracle.plan(inp.q, inp.sigma2, 1, oracle.PLAN_WATERFILL, 56)
    dp = np.zeros_like(planes)
    ds = np.zeros_like(scales)
    oracle.prefix_copy(planes, scales, p, dp, ds)
    for j in range(cfg.d):
        t = int(p[0, 0, j])
        assert np.array_equal(dp[0, 0, j, :t], planes[0, 0, j, :t])
        assert np.all(dp[0, 0, j, t:] == 0)
        assert np.array_equal(ds[0, 0, j], scales[0, 0, j] if t else np.zeros_like(ds[0, 0, j]))


# ---------------------------------------------------------------------------------
# F3 delta selection against a resident set (OasisKV, method details)
# ---------------------------------------------------------------------------------
def _expand(units, block, n_tokens):
    return [t for u in sorted(units) for t in range(u * block, min((u + 1) * block, n_tokens))]


def test_delta_select_worked_example():
    """The hand-worked six-step sequence of tests/golden (one KV head, 3 slots,
    16-token units, a forced local unit, ties, -0.0, C = 0 and a NaN row)."""
    g = json.load(open(os.path.join(GOLD, "delta_select_worked_example.json")))
    R, block, n_tok, nu = g["R"], g["block"], g["n_tokens"], g["n_units"]
    st = oracle.Resident(1, R, nu)
    for step, s in enumerate(g["steps"]):
        sc = np.array([[float(x) for x in s["scores"]]], np.float32)
        if s["P"] is None:
            idx, cnt = np.zeros((1, 8), np.int32), np.array([-1], np.int32)
        else:
            toks = _expand(s["P"], block, n_tok)
            idx, cnt = np.array([toks], np.int32), np.array([len(toks)], np.int32)
        ps, pu, pe, pc, pool, pcount = oracle.delta_select(st, sc, idx, cnt, block, n_tok,
                                                          g["sink"], g["local"], s["C"], step,
                                                          64)
        if s["plan"] is None:
            assert pc[0] == -1 and pcount[0] == -1
        else:
            assert pc[0] == len(s["plan"])
            got = [[int(ps[0, i]), int(pu[0, i]), int(pe[0, i])] for i in range(pc[0])]
            assert got == s["plan"], (step, got)
            rows = [r for a, b in s["pool"] for r in range(a, b)]
            assert pcount[0] == len(rows) and list(pool[0, :pcount[0]]) == rows, step
        assert list(st.slot_unit[0]) == s["slot_unit"], step
        assert list(st.slot_last[0]) == s["slot_last"], step
        us = np.full(nu, -1)
        for slot, u in enumerate(s["slot_unit"]):
            if u >= 0:
                us[u] = slot
        assert np.array_equal(st.unit_slot[0], us), step


def test_delta_select_invariants_random():
    """Random drifting predictions over many steps: at most C admissions per row and
    step, hits keep their slot, the map stays a bijection, every admitted miss ranks
    ahead of every miss left out, every evicted target is no more recently selected
    than any slot kept outside the prediction, and the pool rows are exactly the
    resident predicted units' tokens."""
    rng = np.random.default_rng(7)
    rows, nu, block, R, k, sink, local = 6, 96, 16, 20, 12, 1, 2
    n_tok = nu * block - 5
    st = oracle.Resident(rows, R, nu)
    for step in range(40):
        C = int(rng.integers(0, 6))
        sc = rng.normal(size=(rows, nu)).astype(np.float32)
        sc[:, ::7] = 0.5  # ties
        ri, rc = oracle.topk(sc, k, sink, local, block, n_tok)
        before = st.copy()
        ps, pu, pe, pc, pool, pcount = oracle.delta_select(st, sc, ri, rc, block, n_tok, sink,
                                                          local, C, step, ri.shape[1])
        for r in range(rows):
            P = sorted({int(t) // block for t in ri[r, :rc[r]] if t % block == 0})
            hits = [u for u in P if before.unit_slot[r, u] >= 0]
            miss = [u for u in P if before.unit_slot[r, u] < 0]
            a = int(pc[r])
            free = [s for s in range(R) if before.slot_unit[r, s] not in P]
            assert a == min(C, len(miss), len(free))
            for u in hits:
                assert st.unit_slot[r, u] == before.unit_slot[r, u]
                assert st.slot_last[r, st.unit_slot[r, u]] == step
            res = st.unit_slot[r] >= 0
            assert res.sum() == (st.slot_unit[r] >= 0).sum()
            for s in range(R):
                if st.slot_unit[r, s] >= 0:
                    assert st.unit_slot[r, st.slot_unit[r, s]] == s

            def key(u):  # admission order: forced first, then score desc, unit asc
                forced = u < sink or u >= nu - local
                return (0, u) if forced else (1, -float(sc[r, u]), u)
            admitted = [int(x) for x in pu[r, :a]]
            assert admitted == sorted(miss, key=key)[:a]
            evicted = [int(x) for x in ps[r, :a]]
            kept = [s for s in free if s not in evicted]
            for s in evicted:
                assert pe[r, evicted.index(s)] == before.slot_unit[r, s]
                for s2 in kept:
                    assert (before.slot_last[r, s], s) < (before.slot_last[r, s2], s2)
            rows_exp = [int(st.unit_slot[r, u]) * block + t for u in P if st.unit_slot[r, u] >= 0
                        for t in range(min(block, n_tok - u * block))]
            assert list(pool[r, :pcount[r]]) == rows_exp


# ---------------------------------------------------------------------------------
# F2 8-token block landmarks (Fathom, results: the block-landmark comparison scan)
# ---------------------------------------------------------------------------------
def test_landmark_is_block_mean():
    """Keys on a coarse grid (every fp32 sum exact) and block counts that are powers
    of two (every quotient exact): the landmark equals the numpy mean of the held
    tokens rounded once to bf16, for full blocks and a short last block of 4."""
    rng = np.random.default_rng(21)
    n, d = 8 * 5 + 4, 16
    vals = rng.integers(-64, 65, size=(1, 2, n, d)).astype(np.float64) / 8.0
    K = synth.to_bf16(vals)
    L = synth.bf16_to_f64(oracle.landmark_build(K))
    k = synth.bf16_to_f64(K)
    for c in range(6):
        blkv = k[:, :, 8 * c:min(8 * c + 8, n)]
        ref = synth.bf16_to_f64(synth.to_bf16(blkv.mean(axis=2)))
        assert np.array_equal(L[:, :, c], ref), c


def test_landmark_of_identical_keys_is_the_key():
    rng = np.random.default_rng(22)
    row = synth.to_bf16(rng.normal(size=128) * 3)
    K = np.broadcast_to(row, (1, 1, 24, 128)).copy()
    L = oracle.landmark_build(K)
    assert np.array_equal(L[0, 0], np.broadcast_to(row, (3, 128)))


def test_landmark_score_is_group_dot_product():
    """U = sum_g <q_g, L> against numpy's matmul; a one-hot query reads one channel."""
    cfg = synth.config(0, n=8 * 40, Hq=8, Hkv=2, B=2)
    inp = synth.make_inputs(cfg, with_v=False)
    L = oracle.landmark_build(inp.K)
    U, l1 = oracle.landmark_score(L, inp.q, with_l1=True)
    q = synth.bf16_to_f64(inp.q).reshape(2, 2, 4, 128)
    Lf = synth.bf16_to_f64(L)
    ref = np.einsum("bhgj,bhcj->bhc", q, Lf)
    assert np.allclose(U, ref, rtol=0, atol=1e-9 * np.abs(ref).max())
    assert np.allclose(l1, np.einsum("bhgj,bhcj->bhc", np.abs(q), np.abs(Lf)), rtol=1e-12)
    onehot = np.zeros((1, 1, 128), np.float64)
    onehot[0, 0, 37] = 1.0
    U1 = oracle.landmark_score(L[:1, :1], synth.to_bf16(onehot))
    assert np.array_equal(U1[0, 0], Lf[0, 0, :, 37])


# ---------------------------------------------------------------------------------
# One sequence split by tokens (HashAttention 2.5, contexts beyond one device): the
# shards' candidates merged and their attention combined equal the unsharded step
# ---------------------------------------------------------------------------------
@pytest.mark.parametrize("S,n,k,sink,local", [(2, 64 * 20 + 17, 40, 3, 17), (3, 64 * 9, 30, 0, 0),
                                              (4, 64 * 7 + 1, 25, 70, 5), (2, 300, 400, 4, 4)])
def test_sharded_oracle_step_equals_unsharded(S, n, k, sink, local):
    cfg = synth.config(0, n=n, B=2, Hq=8, Hkv=2, k=k, sink=sink, local=local)
    inp = synth.make_inputs(cfg)
    planes, scales = oracle.plane_build(inp.K)
    plan = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, oracle.PLAN_WATERFILL, 56)
    s = oracle.plane_score(planes, scales, plan, inp.q, n=n).reshape(4, n)
    ri, rc = oracle.topk(s, k, sink, local)
    ro, rl = oracle.gather_attend(inp.q, inp.K, inp.V, ri.reshape(2, 2, -1), rc.reshape(2, 2),
                                  1 / math.sqrt(cfg.d))
    cut = oracle.shard_bounds(n, S)
    assert cut[0] == 0 and cut[-1] == n and all(c % 64 == 0 for c in cut[:-1])
    cands, outs, lses = [], [], []
    for sh in range(S):
        a, b = cut[sh], cut[sh + 1]
        Ks = np.ascontiguousarray(inp.K[:, :, a:b])
        ps, ss = oracle.plane_build(Ks)
        s_s = oracle.plane_score(ps, ss, plan, inp.q, n=b - a).reshape(4, b - a)
        assert np.array_equal(s_s, s[:, a:b])  # whole scale blocks: the same scores
        cands.append(oracle.shard_candidates(s_s, k, *oracle.shard_windows(n, a, b, sink, local), a))
    mi, mc = oracle.topk_merge([c[0] for c in cands], [c[1] for c in cands],
                               [c[2] for c in cands], k)
    union = [[] for _ in range(4)]
    for sh in range(S):
        a, b = cut[sh], cut[sh + 1]
        li, lc = oracle.shard_select(mi, mc, a, b, *oracle.shard_windows(n, a, b, sink, local))
        for r in range(4):
            union[r] += [int(t) + a for t in li[r, :lc[r]]]
        o, l = oracle.gather_attend(inp.q, np.ascontiguousarray(inp.K[:, :, a:b]),
                                    np.ascontiguousarray(inp.V[:, :, a:b]),
                                    li.reshape(2, 2, -1), lc.reshape(2, 2), 1 / math.sqrt(cfg.d))
        outs.append(o)
        lses.append(l)
    # the shards' sets, shifted to global indices, partition the unsharded set
    for r in range(4):
        assert sorted(union[r]) == ri[r, :rc[r]].tolist()
    o, l = oracle.attend_combine(outs, lses)
    assert np.abs(o - ro).max() < 1e-12 and np.abs(l - rl).max() < 1e-12


def test_attend_combine_special_cases():
    o1 = np.ones((1, 1, 4))
    o2 = np.full((1, 1, 4), 3.0)
    # equal masses: the mean; one empty shard: the other; all empty: 0 and -inf
    o, l = oracle.attend_combine([o1, o2], [np.zeros((1, 1)), np.zeros((1, 1))])
    assert np.allclose(o, 2.0) and np.allclose(l, math.log(2.0))
    o, l = oracle.attend_combine([o1, o2], [np.full((1, 1), -np.inf), np.full((1, 1), 0.5)])
    assert np.allclose(o, 3.0) and np.allclose(l, 0.5)
    o, l = oracle.attend_combine([o1, o2], [np.full((1, 1), -np.inf)] * 2)
    assert np.all(o == 0.0) and np.all(l == -np.inf)


def test_topk_merge_nan_and_short_rows():
    sc = [np.array([[3.0, 1.0, -np.inf]]), np.array([[2.0, -np.inf, -np.inf]])]
    ix = [np.array([[10, 4, -1]], np.int32), np.array([[70, -1, -1]], np.int32)]
    mi, mc = oracle.topk_merge(sc, ix, [np.array([2]), np.array([1])], 3)
    assert mc.tolist() == [3] and mi[0].tolist() == [4, 10, 70]
    mi, mc = oracle.topk_merge(sc, ix, [np.array([2]), np.array([-1])], 3)
    assert mc.tolist() == [-1]
