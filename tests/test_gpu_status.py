"""sd_device_status: a bounded wait that runs out inside a kernel is reported to
the host (SD_ERR_TIMEOUT) and cleared, instead of passing silently.  The report
is raised from the host (sd_debug_set_device_error), never by making a wait run
out on the GPU."""
import numpy as np
import pytest
import torch

import synth
from _helpers import dev, empty

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


def test_status_reports_once_and_clears(sd):
    sd.sd_device_status()  # whatever came before: read and cleared
    sd.sd_debug_set_device_error()
    with pytest.raises(sd.SdError) as e:
        sd.sd_device_status()
    assert e.value.code == sd.SD_ERR_TIMEOUT
    assert "incomplete" in str(e.value)
    sd.sd_device_status()  # cleared by the report


def test_status_clean_after_scans(sd):
    cfg = synth.config(2, B=1, n=8192)
    inp = synth.make_inputs(cfg, with_v=False)
    shp = sd.make_shape(cfg.B, cfg.Hq, cfg.Hkv, cfg.n)
    K, q, s2 = dev(inp.K), dev(inp.q), dev(inp.sigma2)
    planes = empty((cfg.B, cfg.Hkv, 128, 4, cfg.n // 32), np.uint32)
    scales = empty((cfg.B, cfg.Hkv, 128, cfg.n // 64), np.uint16)
    sd.sd_build_index(sd.SD_IDX_PLANES, shp, K, None, planes, scales)
    plan = empty((cfg.B, cfg.Hkv, 128), np.uint8)
    scores = empty((cfg.B * cfg.Hkv, cfg.n), np.float32)
    for fallback in (False, True):
        prev = sd.sd_set_fallback_paths(fallback)
        try:
            sd.sd_plan_score(shp, planes, scales, q, s2, sd.SD_PLAN_WATERFILL, 56, plan, scores)
            sd.sd_device_status()
        finally:
            sd.sd_set_fallback_paths(prev)
