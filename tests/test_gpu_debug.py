"""The checked build, libqsa_debug.so (the same kernels compiled with
QSA_DEBUG_CHECKS=1).  Its kernels range-check the selection rows they are
given or write and the TMA tile coordinates they compute, and report a
violation as QSA_ERR_DEVICE_CHECK in the status word, in place of a memory
checker.

* On valid inputs it reports nothing and writes exactly what the normal
  build writes.
* On selection rows that break the indexer's row format, which the normal
  attention tolerates (it ignores entries out of range), it reports the
  violation and still finishes.  The bad entries are in-range integers, so
  every access stays in bounds.
"""
import pytest
import torch

from block_sparse_long_19_b300 import build as B
from block_sparse_long_19_b300 import qsa as Q
from block_sparse_long_19_b300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
QSA_ERR_DEVICE_CHECK = 6


@pytest.fixture(scope="module")
def debug_lib():
    B.build(debug=True)
    return Q.DEBUG_LIB_PATH


def run_prefill(t, budget, tokens=False):
    cfg = Q.default_config(budget=budget)
    if tokens:
        idx, score, st = Q.index_topk_tokens(cfg, t["qi"], t["w"], t["ki"])
        torch.cuda.synchronize()
        return {"idx": idx, "score": score}, int(st.item())
    res = Q.prefill_overlapped(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"], want_score=True)
    torch.cuda.synchronize()
    return {"idx": res.idx, "score": res.score, "out": res.out, "lse": res.lse, "k_rot": res.k_rot}, \
        int(res.status.item())


@pytest.mark.parametrize("L,budget,tokens", [(4133, 512, False), (3001, 32, False), (2500, 64, True)])
def test_debug_build_is_silent_and_identical_on_valid_prefill(debug_lib, L, budget, tokens):
    t = W.prefill_inputs(L, 51, DEV)
    ref, st = run_prefill(t, budget, tokens)
    assert st == 0
    with Q.using_library(debug_lib):
        got, st_d = run_prefill(t, budget, tokens)
    assert st_d == 0
    for k in ref:
        assert torch.equal(ref[k], got[k]), k


def test_debug_build_is_silent_and_identical_on_valid_decode(debug_lib):
    B_, T = 3, 6000
    d = W.decode_inputs(B_, T, 52, DEV, seq_lens=[T, 4097, 9])
    cfg = Q.default_config()
    k_rot = torch.empty_like(d["k"])
    kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=k_rot)

    def step():
        out, lse, idx, st = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], k_rot, d["v"], kblk, d["seq_lens"])
        torch.cuda.synchronize()
        return out, lse, idx, int(st.item())

    ref = step()
    with Q.using_library(debug_lib):
        got = step()
    assert ref[3] == 0 and got[3] == 0
    for a, b in zip(ref[:3], got[:3]):
        assert torch.equal(a, b)


def test_debug_build_flags_malformed_selection_rows(debug_lib):
    """Rows that break the indexer's format (an entry beyond the query's
    block, a descending pair, padding before the end): the normal build
    tolerates them, the checked build reports QSA_ERR_DEVICE_CHECK."""
    L, budget = 4096, 32
    t = W.prefill_inputs(L, 53, DEV)
    cfg = Q.default_config(budget=budget)
    res = Q.prefill_overlapped(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"])
    torch.cuda.synchronize()
    Q.check_status(res.status)
    good = res.idx.clone()
    bad_rows = []
    idx = good.clone()
    r = 3000  # block 750, 31 past blocks + 750
    idx[r, 0] = 751            # beyond the query's block
    bad_rows.append(idx)
    idx = good.clone()
    idx[r, 4], idx[r, 5] = good[r, 5], good[r, 4]  # a descending pair
    bad_rows.append(idx)
    idx = good.clone()
    idx[r, 10] = -1            # padding before the end of the row
    bad_rows.append(idx)
    for bad in bad_rows:
        _, _, st = Q.sparse_attn_prefill(cfg, t["q"], res.k_rot, t["v"], bad)
        torch.cuda.synchronize()
        assert int(st.item()) == 0  # tolerated by the normal build
        with Q.using_library(debug_lib):
            _, _, st_d = Q.sparse_attn_prefill(cfg, t["q"], res.k_rot, t["v"], bad)
            torch.cuda.synchronize()
        assert int(st_d.item()) == QSA_ERR_DEVICE_CHECK
    # and the well-formed rows pass the checked build
    with Q.using_library(debug_lib):
        _, _, st_d = Q.sparse_attn_prefill(cfg, t["q"], res.k_rot, t["v"], good)
        torch.cuda.synchronize()
    assert int(st_d.item()) == 0
