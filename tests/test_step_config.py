"""Host-side unit arithmetic of a decode step (no GPU): the scored unit of each
index kind, the number of units per row and the top-k output stride, against the
definitions in include/sd.h (sd_topk: units of sel.block tokens, a short last
unit, stride min(n_units, sink + local + k) * block)."""
import pytest

import top_sparse_decode_gb300 as sd
from top_sparse_decode_gb300.pipeline import StepConfig


@pytest.mark.parametrize("kind,block", [(sd.SD_IDX_SIG, 1), (sd.SD_IDX_PLANES, 1),
                                        (sd.SD_IDX_MINMAX, 16), (sd.SD_IDX_LANDMARK, 8)])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 16, 17, 4096, 1000003, 1 << 20])
def test_units_and_stride(kind, block, n):
    c = StepConfig(kind, 2, 32, 8, n, k=64, sink=1, local=2)
    assert c.block == block
    assert c.n_units == -(-n // block)  # a short last unit counts
    assert (c.n_units - 1) * block < n <= c.n_units * block
    assert c.max_count == min(c.n_units, 1 + 2 + 64) * block


def test_degenerate_budget_takes_every_unit():
    c = StepConfig(sd.SD_IDX_LANDMARK, 1, 4, 1, 100, k=50, sink=3, local=3)
    assert c.n_units == 13 and c.max_count == 13 * 8


def test_stage_tracing_wraps_each_stage_in_order():
    """run_stages with trace: every stage runs inside a range of its own name, in
    order, and a range is closed even when its stage raises."""
    from top_sparse_decode_gb300.pipeline import run_stages
    log = []
    stages = [(n, lambda q, s, n=n: log.append(("run", n, q, s))) for n in ("plan_scan", "topk")]
    run_stages(stages, "q", "st", True, push=lambda n: log.append(("push", n)),
               pop=lambda: log.append(("pop",)))
    assert log == [("push", "sd.plan_scan"), ("run", "plan_scan", "q", "st"), ("pop",),
                   ("push", "sd.topk"), ("run", "topk", "q", "st"), ("pop",)]
    log.clear()
    run_stages(stages, "q", None)  # untraced: the calls alone
    assert [e[0] for e in log] == ["run", "run"]

    def boom(q, s):
        raise RuntimeError("stage failed")
    log.clear()
    with pytest.raises(RuntimeError):
        run_stages([("bad", boom)], "q", None, True, push=lambda n: log.append(("push", n)),
                   pop=lambda: log.append(("pop",)))
    assert log == [("push", "sd.bad"), ("pop",)]
