"""GPU parity of prefill after a cached prefix (prefix-cache serving; launch
post, "Model Architecture / Attention: GDN + QSA for Efficient Memory and
Precise Retrieval", measures prefill at a 90% prefix-cache hit rate).

The query rows of a chunk are the same rows of a full prefill (same
definition): they are checked against the oracle's rows of the full
sequence, and against the full CUDA prefill bit for bit (the per-query
results do not depend on which other queries share a launch)."""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_long_19_b300 import qsa as Q
from block_sparse_long_19_b300 import workloads as W

from .parity import SCORE_ATOL_RMS, SCORE_RTOL, bf16_to_f64, check_outputs, check_selection, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def rows_from(L, lo, n, seed):
    rows = sample_rows(L, n, seed, extra=range(lo, lo + 4))
    return rows[rows >= lo]


def check_selected_scores(score_g, idx_g, scores_ref, rows):
    """The score written beside each selected past block against the oracle's
    score of that block (the current block carries +inf, padding -inf)."""
    for r, t in enumerate(rows):
        c = int(t) // 4
        ref = scores_ref[r, :c]
        rms = np.sqrt(np.mean(ref * ref)) if c > 0 else 0.0
        for j, b in enumerate(idx_g[r]):
            if b < 0:
                assert score_g[r, j] == -np.inf
            elif b == c:
                assert score_g[r, j] == np.inf
            else:
                assert abs(score_g[r, j] - ref[b]) <= SCORE_RTOL * abs(ref[b]) + SCORE_ATOL_RMS * rms


def full_prefill(t, budget):
    cfg = Q.default_config(budget=budget)
    res = Q.prefill(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"], want_score=True)
    torch.cuda.synchronize()
    Q.check_status(res.status)
    return res


def chunked_prefill(t, budget, bounds):
    """Prefill in chunks [bounds[i], bounds[i+1]): each chunk extends the
    cached K-prep (block keys, RoPE'd keys) and runs the cached indexer and
    attention on its own rows only."""
    cfg = Q.default_config(budget=budget)
    L = t["q"].shape[0]
    kblk = torch.zeros((max(L // 4, 1), 128), dtype=torch.bfloat16, device=DEV)
    k_rot = torch.empty_like(t["k"])
    idx = torch.empty((L, budget), dtype=torch.int32, device=DEV)
    score = torch.empty((L, budget), dtype=torch.float32, device=DEV)
    out = torch.empty_like(t["q"])
    lse = torch.empty((L, 24), dtype=torch.float32, device=DEV)
    status = Q.new_status(DEV)
    for a, b in zip(bounds[:-1], bounds[1:]):
        # only the first b rows exist so far: pass views of the prefix
        Q.kprep_range(cfg, t["ki"][:b], kblk, a, b, k=t["k"][:b], k_rot=k_rot[:b])
        Q.index_topk_cached(cfg, t["qi"][a:b], t["w"][a:b], kblk[: b // 4] if b >= 4 else kblk[:1], a,
                            idx=idx[a:b], score=score[a:b], status=status)
        Q.sparse_attn_prefill_cached(cfg, t["q"][a:b], k_rot[:b], t["v"][:b], idx[a:b], a, out=out[a:b],
                                     lse=lse[a:b], status=status)
    torch.cuda.synchronize()
    Q.check_status(status)
    return idx, score, out, lse, k_rot, kblk


@pytest.mark.parametrize("L,bounds,budget", [
    (4133, [0, 3700, 4133], 512),            # one cached prefix, ragged offset
    (9001, [0, 2500, 6001, 9001], 512),      # three chunks
    (777, [0, 1, 2, 5, 6, 777], 32),         # tiny chunks, offsets not multiples of 4
])
def test_chunked_prefill_matches_full_prefill_and_oracle(L, bounds, budget):
    t = W.prefill_inputs(L, 41, DEV)
    hb = W.host_bits(t)
    full = full_prefill(t, budget)
    idx, score, out, lse, k_rot, kblk = chunked_prefill(t, budget, bounds)
    # bit for bit the full prefill's rows
    assert torch.equal(idx, full.idx)
    assert torch.equal(score, full.score)
    assert torch.equal(out, full.out)
    assert torch.equal(lse, full.lse)
    assert np.array_equal(W.to_bits(kblk[: L // 4]), O.block_keys(hb["ki"]))
    # and the oracle on the rows of the last chunk
    rows = rows_from(L, bounds[-2], 48, 5)
    idx_g = idx.cpu().numpy()[rows]
    ref = O.prefill_rows(hb, rows, budget, want_o=False)
    scores = O.prefill_scores(hb, rows)
    check_selection(idx_g, ref["idx"], scores, rows, budget)
    check_selected_scores(score.cpu().numpy()[rows].astype(np.float64), idx_g, scores, rows)
    att = O.prefill_rows(hb, rows, budget, idx_given=idx_g)
    check_outputs(bf16_to_f64(out[torch.as_tensor(rows, device=DEV)]), att["o"], "O")
    check_outputs(lse.cpu().numpy().astype(np.float64)[rows], att["lse"], "LSE")


def test_prefix90_at_128k():
    """The serving setup: the last 10% of a 131,072-token sequence against a
    90% cached prefix, sampled rows against the oracle and all rows against
    the full prefill."""
    L, budget = 131072, 512
    q_off = L - L // 10
    t = W.prefill_inputs(L, 42, DEV)
    hb = W.host_bits(t)
    full = full_prefill(t, budget)
    cfg = Q.default_config(budget=budget)
    kblk, k_rot = Q.kprep(cfg, t["ki"], t["k"])  # the cache: every block and key row
    idx, score, st = Q.index_topk_cached(cfg, t["qi"][q_off:], t["w"][q_off:], kblk, q_off)
    out, lse, st2 = Q.sparse_attn_prefill_cached(cfg, t["q"][q_off:], k_rot, t["v"], idx, q_off)
    torch.cuda.synchronize()
    Q.check_status(st)
    Q.check_status(st2)
    assert torch.equal(idx, full.idx[q_off:])
    assert torch.equal(out, full.out[q_off:])
    rows = rows_from(L, q_off, 24, 6)
    loc = [r - q_off for r in rows]
    idx_g = idx.cpu().numpy()[loc]
    ref = O.prefill_rows(hb, rows, budget, want_o=False)
    scores = O.prefill_scores(hb, rows)
    check_selection(idx_g, ref["idx"], scores, rows, budget)
    att = O.prefill_rows(hb, rows, budget, idx_given=idx_g)
    check_outputs(bf16_to_f64(out[torch.as_tensor(loc, device=DEV)]), att["o"], "O")


@pytest.mark.parametrize("L,chunk", [(9001, 2048), (266277, 65536)])
def test_host_prefill_pipeline_equals_device_prefill(L, chunk):
    """qsa.HostPrefill (inputs in pinned host memory, chunked, copies on their
    own streams; at 266,277 tokens also the indexer beside the attention on
    two compute streams) returns exactly the device prefill's output and LSE."""
    budget = 512
    t = W.prefill_inputs(L, 44, DEV)
    full = full_prefill(t, budget)
    cfg = Q.default_config(budget=budget)
    host = {n: t[n].cpu().pin_memory() for n in Q.HostPrefill.NAMES}
    out_h = torch.empty((L, 24, 256), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((L, 24), dtype=torch.float32).pin_memory()
    hp = Q.HostPrefill(cfg, L, chunk_tokens=chunk)
    assert (hp.ctas is not None) == (L >= 262144)
    st = hp.run(host, out_h, lse_h)
    torch.cuda.synchronize()
    Q.check_status(st)
    assert torch.equal(out_h, full.out.cpu())
    assert torch.equal(lse_h, full.lse.cpu())
    assert torch.equal(hp.idx, full.idx)


@pytest.mark.parametrize("L,budget,yarn", [
    (266277, 512, 1.0),  # 16 chunks, the last one ragged
    (262144, 32, 1.0),   # 16 chunks, small budget
    (262144, 512, 4.0),  # 16 chunks, YaRN on (the model card's factor 4)
    (70001, 512, 1.0),   # short: the two stages one after the other
    (65536, 1, 1.0),     # no indexer work: the current block only
])
def test_overlapped_prefill_equals_serial_prefill(L, budget, yarn):
    """qsa_prefill_overlapped (the indexer of chunk j beside the attention of
    chunk j-1, on two streams) writes exactly what the serial prefill writes:
    selection, scores, RoPE'd keys, output and LSE; sampled rows of the last
    chunk also against the oracle."""
    t = W.prefill_inputs(L, 45, DEV)
    cfg = Q.default_config(budget=budget, yarn_factor=yarn)
    full = Q.prefill(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"], want_score=True)
    torch.cuda.synchronize()
    Q.check_status(full.status)
    res = Q.prefill_overlapped(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"], want_score=True)
    torch.cuda.synchronize()
    Q.check_status(res.status)
    assert torch.equal(res.idx, full.idx)
    assert torch.equal(res.score, full.score)
    assert torch.equal(res.k_rot, full.k_rot)
    assert torch.equal(res.out, full.out)
    assert torch.equal(res.lse, full.lse)
    if budget > 1 and L >= 262144:
        hb = W.host_bits(t)
        begin, _ = Q.prefill_overlap_plan(cfg, L, torch.cuda.get_device_properties(0).multi_processor_count)
        rows = rows_from(L, begin[-2], 16, 7)
        idx_g = res.idx.cpu().numpy()[rows]
        ref = O.prefill_rows(hb, rows, budget, want_o=False)
        check_selection(idx_g, ref["idx"], O.prefill_scores(hb, rows), rows, budget)
        att = O.prefill_rows(hb, rows, budget, idx_given=idx_g, yarn=O.YARN_CARD if yarn > 1 else None)
        check_outputs(bf16_to_f64(res.out[torch.as_tensor(rows, device=DEV)]), att["o"], "O")


def test_overlapped_prefill_under_graph_capture():
    """Captured into a CUDA graph, the overlapped prefill takes its serial
    schedule on the captured stream; a replay writes the serial results."""
    L, budget = 262144, 512
    t = W.prefill_inputs(L, 46, DEV)
    full = full_prefill(t, budget)
    cfg = Q.default_config(budget=budget)
    k_rot = torch.empty_like(t["k"])
    idx = torch.full((L, budget), -7, dtype=torch.int32, device=DEV)
    out = torch.zeros_like(t["q"])
    lse = torch.zeros((L, 24), dtype=torch.float32, device=DEV)
    ws = torch.empty(Q.prefill_overlapped_workspace_bytes(cfg, L), dtype=torch.uint8, device=DEV)
    status = Q.new_status(DEV)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        Q.prefill_overlapped(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"], k_rot=k_rot, idx=idx,
                             out=out, lse=lse, ws=ws, status=status)
    g.replay()
    torch.cuda.synchronize()
    Q.check_status(status)
    assert torch.equal(idx, full.idx)
    assert torch.equal(out, full.out)
    assert torch.equal(lse, full.lse)
