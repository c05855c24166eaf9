"""GPU parity of the token-level indexer variant (one token per selection
unit; the DSA-style indexer the launch post contrasts QSA with, "Attention:
GDN + QSA").

Reference without a second oracle: token-level selection over L tokens is
the oracle's block-level selection over an expanded sequence in which every
token's indexer key fills a whole 4-token block (the mean of four equal bf16
values is that value, exactly) and query t sits at position 4t+3 (its block
is t, its past blocks the tokens before it)."""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_long_19_b300 import qsa as Q
from block_sparse_long_19_b300 import workloads as W

from .parity import check_selection, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def expanded(hb):
    L = hb["qi"].shape[0]
    e = {"qi": np.repeat(hb["qi"], 4, axis=0), "w": np.repeat(hb["w"], 4, axis=0),
         "ki": np.repeat(hb["ki"], 4, axis=0)}
    # attention inputs are unused for the selection; zeros of the right shape
    e["q"] = np.zeros((4 * L, 24, 256), np.uint16)
    e["k"] = np.zeros((4 * L, 2, 256), np.uint16)
    e["v"] = np.zeros((4 * L, 2, 256), np.uint16)
    return {k_: np.ascontiguousarray(v_) for k_, v_ in e.items()}


@pytest.mark.parametrize("L,budget", [(3001, 512), (777, 64), (40, 8)])
def test_token_level_selection_matches_expanded_oracle(L, budget):
    t = W.prefill_inputs(L, 71, DEV)
    hb = W.host_bits(t)
    cfg = Q.default_config(budget=budget)
    idx, score, st = Q.index_topk_tokens(cfg, t["qi"], t["w"], t["ki"])
    torch.cuda.synchronize()
    Q.check_status(st)
    rows = sample_rows(L, 40, 9)
    e = expanded(hb)
    erows = 4 * rows + 3
    ref = O.prefill_rows(e, erows, budget, want_o=False)
    scores = O.prefill_scores(e, erows)
    idx_g = idx.cpu().numpy()[rows]
    check_selection(idx_g, ref["idx"], scores, erows, budget)
    # the current unit of query t is token t; scores of selected tokens
    sc = score.cpu().numpy()[rows]
    for r, t_ in enumerate(rows):
        row = idx_g[r]
        n = min(budget, t_ + 1)
        assert row[n - 1] == t_ and sc[r, n - 1] == np.inf
        past = row[: n - 1]
        ref_s = scores[r, past]
        assert np.all(np.abs(sc[r, : n - 1] - ref_s) <= 1e-2 * np.abs(ref_s) + 1e-3 * np.sqrt(np.nanmean(scores[r, :t_] ** 2)) + 1e-12)
