"""The C-ABI library loads and exports every entry point include/sd.h declares;
argument checks fail with the documented codes before anything reaches CUDA.
No GPU needed: every call here is rejected by the host-side checks."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sd():
    from top_sparse_decode_gb300 import build as b
    b.build()
    import top_sparse_decode_gb300 as sdmod
    sdmod.lib()
    return sdmod


def header_functions():
    text = open(os.path.join(ROOT, "include", "sd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[\w\s\*]+?\b(sd_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_path():
    names = header_functions()
    for must in ["sd_build_index", "sd_append_index", "sd_encode_query", "sd_plan", "sd_score", "sd_topk",
                 "sd_gather_attend", "sd_offload_gather", "sd_last_error"]:
        assert must in names


def test_library_exports_every_declared_symbol(sd):
    lib = sd.lib()
    for name in header_functions():
        assert hasattr(lib, name), name
    from top_sparse_decode_gb300 import _abi
    assert sorted(_abi.SIGNATURES) == header_functions()
    for name in header_functions():
        assert callable(getattr(sd, name)), name
    assert sd.sd_version() == 104  # 1.04: sd_copy


def test_shape_checks(sd):
    bad = [sd.make_shape(1, 4, 1, 4096, d=64),      # d != 128
           sd.make_shape(1, 12, 4, 4096),           # G = 3
           sd.make_shape(1, 4, 3, 4096),            # hq % hkv
           sd.make_shape(0, 4, 1, 4096),            # batch 0
           sd.make_shape(1, 4, 1, 4096, n_cap=100)]  # n_cap < n
    codes = [sd.SD_ERR_UNSUPPORTED, sd.SD_ERR_UNSUPPORTED, sd.SD_ERR_INVALID_ARG,
             sd.SD_ERR_INVALID_ARG, sd.SD_ERR_INVALID_ARG]
    lib = sd.lib()
    for shp, code in zip(bad, codes):
        rc = lib.sd_plan(ctypes.byref(shp), 16, 16, 0, 56, 16, None)
        assert rc == code, (shp.d, shp.hq, shp.hkv, rc)
        assert sd.sd_last_error()


def test_argument_checks(sd):
    lib = sd.lib()
    shp = sd.make_shape(1, 4, 1, 4096)
    P = 1 << 20  # a fake, aligned address; never dereferenced
    # planes need n % 64 == 0
    shp_r = sd.make_shape(1, 4, 1, 4000)
    assert lib.sd_build_index(1, ctypes.byref(shp_r), P, None, P, P, None) == sd.SD_ERR_UNSUPPORTED
    # misaligned K
    assert lib.sd_build_index(2, ctypes.byref(shp), P + 2, None, P, None, None) == sd.SD_ERR_INVALID_ARG
    # unknown kind
    assert lib.sd_build_index(7, ctypes.byref(shp), P, None, P, None, None) == sd.SD_ERR_INVALID_ARG
    # signatures need an encoder; hidden 100 unsupported
    assert lib.sd_build_index(0, ctypes.byref(shp), P, None, P, None, None) == sd.SD_ERR_INVALID_ARG
    enc = sd._abi.SdEncoder(P, None, 100, P, None)
    assert lib.sd_build_index(0, ctypes.byref(shp), P, ctypes.byref(enc), P, None, None) == \
        sd.SD_ERR_UNSUPPORTED
    # appends: n_old in [0, n], planes need n_cap % 64 == 0 (any n), scales required
    shp_a = sd.make_shape(1, 4, 1, 4001, 128, 4032)
    assert lib.sd_append_index(2, ctypes.byref(shp_a), 4002, P, None, P, None, None) == \
        sd.SD_ERR_INVALID_ARG
    assert lib.sd_append_index(2, ctypes.byref(shp_a), -1, P, None, P, None, None) == \
        sd.SD_ERR_INVALID_ARG
    assert lib.sd_append_index(1, ctypes.byref(shp_a), 4000, P, None, P, None, None) == \
        sd.SD_ERR_INVALID_ARG
    shp_b = sd.make_shape(1, 4, 1, 4001, 128, 4040)
    assert lib.sd_append_index(1, ctypes.byref(shp_b), 4000, P, None, P, P, None) == \
        sd.SD_ERR_UNSUPPORTED
    assert lib.sd_append_index(0, ctypes.byref(shp_a), 4000, P, None, P, None, None) == \
        sd.SD_ERR_INVALID_ARG
    assert lib.sd_append_index(7, ctypes.byref(shp_a), 4000, P, None, P, None, None) == \
        sd.SD_ERR_INVALID_ARG
    assert lib.sd_append_index(2, ctypes.byref(shp_a), 4000, P + 8, None, P, None, None) == \
        sd.SD_ERR_INVALID_ARG
    # n_old == n appends nothing and launches nothing
    assert lib.sd_append_index(2, ctypes.byref(shp_a), 4001, P, None, P, None, None) == sd.SD_OK
    # delta selection: block, slots, cap, step, strides; gather: block and slots
    res = sd._abi.SdResident(16, P, P, P)
    selb16 = sd.make_select(8, 0, 1, 16)
    shp_d = sd.make_shape(2, 8, 2, 1600)

    def ds(sel=selb16, cap=4, step=0, r=res, istride=9 * 16, pstride=9 * 16):
        return lib.sd_delta_select(ctypes.byref(shp_d), ctypes.byref(sel), P, P, istride, P, cap,
                                   step, ctypes.byref(r), P, P, P, P, P, pstride, P, None)
    assert ds(sel=sd.make_select(8, 0, 1, 0)) == sd.SD_ERR_INVALID_ARG
    assert ds(cap=-1) == sd.SD_ERR_INVALID_ARG
    assert ds(step=-1) == sd.SD_ERR_INVALID_ARG
    assert ds(step=0x7FFFFFFF) == sd.SD_ERR_INVALID_ARG
    assert ds(istride=9 * 16 - 1) == sd.SD_ERR_INVALID_ARG
    assert ds(pstride=9 * 16 - 1) == sd.SD_ERR_INVALID_ARG
    assert ds(r=sd._abi.SdResident(0, P, P, P)) == sd.SD_ERR_UNSUPPORTED
    assert ds(r=sd._abi.SdResident(5000, P, P, P)) == sd.SD_ERR_UNSUPPORTED
    assert ds(r=sd._abi.SdResident(16, P, None, P)) == sd.SD_ERR_INVALID_ARG
    shp_big = sd.make_shape(1, 1, 1, 1 << 16)
    sel_big = sd.make_select(4096, 4096, 4096, 1)  # 12,288 predicted units
    assert lib.sd_delta_select(ctypes.byref(shp_big), ctypes.byref(sel_big), P, P, 1 << 20, P, 4,
                               0, ctypes.byref(res), P, P, P, P, P, 1 << 20, P, None) == \
        sd.SD_ERR_UNSUPPORTED
    assert lib.sd_resident_gather(ctypes.byref(shp_d), 0, P, P, P, P, P, 4, 16, P, P, None) == \
        sd.SD_ERR_INVALID_ARG
    assert lib.sd_resident_gather(ctypes.byref(shp_d), 16, P, P, P, P, P, 4, 0, P, P, None) == \
        sd.SD_ERR_UNSUPPORTED
    assert lib.sd_resident_gather(ctypes.byref(shp_d), 16, P + 8, P, P, P, P, 4, 16, P, P,
                                  None) == sd.SD_ERR_INVALID_ARG
    # plan budgets
    assert lib.sd_plan(ctypes.byref(shp), P, P, 0, 513, P, None) == sd.SD_ERR_INVALID_ARG
    assert lib.sd_plan(ctypes.byref(shp), P, P, 1, 129, P, None) == sd.SD_ERR_INVALID_ARG
    assert lib.sd_plan(ctypes.byref(shp), P, P, 5, 1, P, None) == sd.SD_ERR_INVALID_ARG
    # top-q: at most d channels, q required, sigma2 not
    assert lib.sd_plan(ctypes.byref(shp), P, None, 3, 129, P, None) == sd.SD_ERR_INVALID_ARG
    assert lib.sd_plan(ctypes.byref(shp), P, None, 3, -1, P, None) == sd.SD_ERR_INVALID_ARG
    assert lib.sd_plan(ctypes.byref(shp), None, None, 3, 17, P, None) == sd.SD_ERR_INVALID_ARG
    assert lib.sd_plan(ctypes.byref(shp), P, None, 1, 17, P, None) == sd.SD_ERR_INVALID_ARG
    assert lib.sd_plan_score(ctypes.byref(shp), P, P, P, None, 3, 129, None, P, None, None) == \
        sd.SD_ERR_INVALID_ARG
    assert lib.sd_plan_score(ctypes.byref(shp), P, P, P, None, 0, 56, None, P, None, None) == \
        sd.SD_ERR_INVALID_ARG
    # top-k limits and strides
    sel = sd.make_select(5000)
    assert lib.sd_topk(1, P, 1, 100, 100, ctypes.byref(sel), P, 5000, P, None, 0, None) == \
        sd.SD_ERR_UNSUPPORTED
    sel = sd.make_select(10, 2, 2)
    assert lib.sd_topk(1, P, 1, 100, 100, ctypes.byref(sel), P, 13, P, None, 0, None) == \
        sd.SD_ERR_INVALID_ARG
    assert lib.sd_topk(3, P, 1, 100, 100, ctypes.byref(sel), P, 14, P, None, 0, None) == \
        sd.SD_ERR_INVALID_ARG
    # long rows need a workspace
    need = sd.sd_topk_workspace_size(2, 100000, sel)
    assert need > 0 and sd.sd_topk_workspace_size(2, 1000, sel) == 0
    assert lib.sd_topk(1, P, 2, 100000, 100000, ctypes.byref(sel), P, 14, P, P, need - 1, None) \
        == sd.SD_ERR_WORKSPACE
    # block mode: n_tokens must match n_units * block
    selb = sd.make_select(4, 0, 1, 16)
    assert lib.sd_topk(1, P, 1, 10, 200, ctypes.byref(selb), P, 80, P, None, 0, None) == \
        sd.SD_ERR_INVALID_ARG
    # token indices are int32: a row's tokens and its output must stay below 2^31
    selh = sd.make_select(2, 0, 0, 1 << 30)
    assert lib.sd_topk(1, P, 1, 3, (1 << 31) + 5, ctypes.byref(selh), P, 1 << 31, P, None, 0,
                       None) == sd.SD_ERR_UNSUPPORTED
    assert lib.sd_topk(1, P, 1, 2, (1 << 30) + 5, ctypes.byref(selh), P, 1 << 31, P, None, 0,
                       None) == sd.SD_ERR_UNSUPPORTED
    # gather-attend workspace
    wsz = sd.sd_gather_attend_workspace_size(shp, 200)
    assert wsz > 0
    assert lib.sd_gather_attend(ctypes.byref(shp), P, P, P, P, 200, P, 200, 0.1, P, None, P,
                                wsz - 1, None) == sd.SD_ERR_WORKSPACE
    assert lib.sd_gather_attend(ctypes.byref(shp), P, P, P, P, 100, P, 200, 0.1, P, None, P,
                                wsz, None) == sd.SD_ERR_INVALID_ARG
    assert lib.sd_event_wait(None, 10) == sd.SD_ERR_INVALID_ARG


def test_fused_entry_argument_checks(sd):
    """sd_topk_wmax, sd_hamming_topk and sd_select_attend reject bad arguments on the
    host, before any device work."""
    lib = sd.lib()
    P = 1 << 20  # a fake, aligned address; never dereferenced
    shp = sd.make_shape(1, 32, 8, 1 << 20)
    sel = sd.make_select(512)
    # word maxima: n >= 1, scores 16-byte aligned, block 1
    assert lib.sd_topk_wmax(P, P, 8, 0, ctypes.byref(sel), P, 512, P, None, 0, None) == \
        sd.SD_ERR_INVALID_ARG
    assert lib.sd_topk_wmax(P + 4, P, 8, 1 << 20, ctypes.byref(sel), P, 512, P, None, 0,
                            None) == sd.SD_ERR_INVALID_ARG
    selb = sd.make_select(4, 0, 1, 16)
    assert lib.sd_topk_wmax(P, P, 8, 1 << 20, ctypes.byref(selb), P, 80, P, None, 0, None) == \
        sd.SD_ERR_INVALID_ARG
    need = sd.sd_topk_workspace_size(8, 1 << 20, sel)
    assert lib.sd_topk_wmax(P, P, 8, 1 << 20, ctypes.byref(sel), P, 512, P, P, need - 1,
                            None) == sd.SD_ERR_WORKSPACE
    # Hamming scan + top-k: token mode only, k limit, stride, workspace, size limit
    assert lib.sd_hamming_topk(ctypes.byref(shp), P, P, ctypes.byref(selb), P, 80, P, P, 1 << 30,
                               None) == sd.SD_ERR_INVALID_ARG
    big = sd.make_select(5000)
    assert lib.sd_hamming_topk(ctypes.byref(shp), P, P, ctypes.byref(big), P, 5000, P, P,
                               1 << 30, None) == sd.SD_ERR_UNSUPPORTED
    assert lib.sd_hamming_topk(ctypes.byref(shp), P, P, ctypes.byref(sel), P, 511, P, P, 1 << 30,
                               None) == sd.SD_ERR_INVALID_ARG
    hw = sd.sd_hamming_topk_workspace_size(shp, sel)
    assert hw > 0
    assert lib.sd_hamming_topk(ctypes.byref(shp), P, P, ctypes.byref(sel), P, 512, P, P, hw - 1,
                               None) == sd.SD_ERR_WORKSPACE
    huge = sd.make_shape(1, 32, 8, 3 << 20)
    assert lib.sd_hamming_topk(ctypes.byref(huge), P, P, ctypes.byref(sel), P, 512, P, P, 1 << 40,
                               None) == sd.SD_ERR_UNSUPPORTED
    # selection + attention: NULL inputs, strides, workspace
    assert lib.sd_select_attend(ctypes.byref(shp), P, P, ctypes.byref(sel), P, None, P, 0.1, P,
                                512, P, 512, P, None, P, 1 << 30, None) == sd.SD_ERR_INVALID_ARG
    assert lib.sd_select_attend(ctypes.byref(shp), P, P, ctypes.byref(sel), P, P, P, 0.1, P,
                                512, P, 511, P, None, P, 1 << 30, None) == sd.SD_ERR_INVALID_ARG
    sw = sd.sd_select_attend_workspace_size(shp, sel, 512)
    assert sw > 0
    assert lib.sd_select_attend(ctypes.byref(shp), P, P, ctypes.byref(sel), P, P, P, 0.1, P,
                                512, P, 512, P, None, P, sw - 1, None) == sd.SD_ERR_WORKSPACE
    assert sd.sd_last_error()


def test_python_binding_raises_with_message(sd):
    shp = sd.make_shape(1, 4, 1, 4096, d=64)
    with pytest.raises(sd.SdError) as ei:
        sd.sd_plan(shp, 16, 16, 0, 56, 16, stream=0)
    assert ei.value.code == sd.SD_ERR_UNSUPPORTED and "d = 64" in str(ei.value)


def test_fallback_switch_is_off_by_default_and_returns_previous(sd):
    assert sd.sd_set_fallback_paths(True) is False
    assert sd.sd_set_fallback_paths(False) is True
    assert sd.sd_set_fallback_paths(False) is False


def test_copy_argument_checks(sd):
    lib = sd.lib()
    A = 1 << 20  # aligned placeholder addresses; never dereferenced
    assert lib.sd_copy(A, A + 64, 0, None) == sd.SD_OK  # nothing to do
    for dst, src, n in [(None, A, 16), (A, None, 16), (A + 8, A, 16), (A, A + 4, 16), (A, A, 24)]:
        assert lib.sd_copy(dst, src, n, None) == sd.SD_ERR_INVALID_ARG
        assert "sd_copy" in sd.sd_last_error()
