"""Failure detection without a GPU fault: a bounded wait that runs out is
reported through the status word and the kernel returns, leaving the context
usable (the self-test waits on an mbarrier phase that nothing completes)."""
import pytest
import torch

from block_sparse_long_19_b300 import qsa as Q
from block_sparse_long_19_b300 import workloads as W

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    st = Q.selftest_bounded_wait(1_000_000, complete=False)  # 1 ms
    torch.cuda.synchronize()
    assert int(st.item()) == Q.QSA_ERR_TIMEOUT
    with pytest.raises(Q.QsaError):
        Q.check_status(st)
    # the same context keeps working: a small prefill right after
    t = W.prefill_inputs(300, 91, "cuda")
    res = Q.prefill(Q.default_config(budget=16), t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"])
    torch.cuda.synchronize()
    Q.check_status(res.status)
    assert int(res.idx[299, 15]) == 299 // 4  # the current block closes the row


def test_wait_that_completes_reports_nothing():
    st = Q.selftest_bounded_wait(1_000_000, complete=True)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
