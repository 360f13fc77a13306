"""Failure detection without a GPU fault.

* The bounded waits: a grid barrier that one participant never reaches and an
  mbarrier phase that nothing completes both give up after the wait limit,
  record the timeout in the device status word and return; the same context
  then builds a correct round.
* Host-side fault injection: a failing workspace allocation (an error code
  from a fake of the failing call) makes dt_create report DT_ERR_OOM and leaves
  nothing behind; the next create succeeds.
"""
import time

import pytest

from tests.parity import check_round, to_np, upload_round, upload_weights
from workloads import get_config, make_round_inputs, make_weights

pytestmark = pytest.mark.gpu

DT_ERR_OOM = 4
DT_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def tiny():
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    from oracle.dartree import Oracle
    torch.cuda.set_device(0)
    cfg = get_config("tiny_bf16")
    w = make_weights(cfg)
    b = DraftTreeBuilder(cfg, upload_weights(w))
    yield cfg, w, b, Oracle(w, cfg)
    b.close()


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_times_out_and_context_stays_usable(tiny, which):
    cfg, w, b, orc = tiny
    assert b.device_status() == 0
    t0 = time.time()
    b.check_bounded_waits(which)
    status = b.device_status()  # synchronises
    elapsed = time.time() - t0
    assert status == DT_ERR_TIMEOUT
    assert 1.0 < elapsed < 30.0
    # the context still builds correct rounds
    H, root = make_round_inputs(cfg, 3)
    out = to_np(b.build_round(*upload_round(H, root)))
    assert all(st != "MISMATCH" for st, _ in check_round(orc, out, H, root))
    assert b.device_status() == 0


def test_check_rejects_unknown_kind(tiny):
    from conditional_draft_tree_lm_gb300 import DtreeError
    _, _, b, _ = tiny
    with pytest.raises(DtreeError):
        b.check_bounded_waits(7)


def test_injected_workspace_allocation_failure(monkeypatch):
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder, DtreeError
    torch.cuda.set_device(0)
    cfg = get_config("tiny_bf16")
    wd = upload_weights(make_weights(cfg))
    monkeypatch.setenv("DT_FAULT_INJECT_ALLOC", "1")
    with pytest.raises(DtreeError) as e:
        DraftTreeBuilder(cfg, wd)
    assert e.value.status == DT_ERR_OOM
    monkeypatch.delenv("DT_FAULT_INJECT_ALLOC")
    b = DraftTreeBuilder(cfg, wd)
    try:
        H, root = make_round_inputs(cfg, 0)
        b.build_round(*upload_round(H, root))
        assert b.device_status() == 0
    finally:
        b.close()
