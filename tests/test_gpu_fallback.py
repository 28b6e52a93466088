"""The kernels libsd takes where its thread-block clusters cannot be co-resident
or bulk copies do not apply -- the split-n gather-attend with workspace partials,
the sampled-threshold sample/filter/finish top-k, the one-CTA word-maxima top-k,
sd_select_attend as its two calls, the cp.async bit-plane scan -- forced on with
sd_set_fallback_paths and held to the same oracle parity as the cluster and
bulk-copy kernels (on a GB300 they would otherwise never run)."""
import pytest

import test_gpu_pipeline as pl
import test_gpu_select_attend as sa
import test_gpu_stages as st
import test_gpu_topk_wmax as tw
from test_gpu_stages import sd  # noqa: F401  (the module's library fixture)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def fallback_paths(sd):  # noqa: F811
    prev = sd.sd_set_fallback_paths(True)
    try:
        yield
    finally:
        sd.sd_set_fallback_paths(prev)


def test_switch_reports_previous_setting(sd):  # noqa: F811
    assert sd.sd_set_fallback_paths(True) is True
    assert sd.sd_set_fallback_paths(True) is True


# stage parity (oracle), now through the fallback kernels
test_plane_scores = st.test_plane_scores
test_plane_scores_long_ranges = st.test_plane_scores_long_ranges
test_topk_bit_exact_on_shared_scores = st.test_topk_bit_exact_on_shared_scores
test_topk_estimate_misses_fall_back_to_exact = st.test_topk_estimate_misses_fall_back_to_exact
test_topk_clustered_winners = st.test_topk_clustered_winners
test_topk_nan_row = st.test_topk_nan_row
test_gather_attend = st.test_gather_attend
test_topk_wmax_equals_oracle = tw.test_topk_wmax_equals_oracle
test_wmax_signed_zeros_and_infinities = tw.test_signed_zeros_and_infinities
test_wmax_nan_rows = tw.test_nan_rows
test_word_maxima_from_plan_score = tw.test_word_maxima_from_plan_score
test_select_attend_against_oracle = sa.test_select_attend_against_oracle


# whole steps against the oracle
def test_step_cfg0_tiny_all_scorers(sd):  # noqa: F811
    pl.test_cfg0_tiny_all_scorers(sd)


@pytest.mark.slow
def test_step_cfg1_hash_32k(sd):  # noqa: F811
    pl.test_cfg1_hash_32k_full(sd)


@pytest.mark.slow
def test_step_cfg3_quest_b64(sd):  # noqa: F811
    pl.test_cfg3_quest_b64_full(sd)
