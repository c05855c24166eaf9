"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded inputs.  Rules are in tests/parity.py."""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_long_19_b300 import qsa as Q
from block_sparse_long_19_b300 import workloads as W

from .parity import (bf16_to_f64, check_outputs, check_rope, check_row_format, check_scores,
                     check_selection, sample_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_prefill(t, budget, want_score=True):
    cfg = Q.default_config(budget=budget)
    res = Q.prefill(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"], want_score=want_score)
    torch.cuda.synchronize()
    Q.check_status(res.status)
    return res


def oracle_compare_prefill(t, hb, res, rows, budget, check_attn=True):
    idx_gpu = res.idx.cpu().numpy()[rows]
    ref = O.prefill_rows(hb, rows, budget, want_o=False)
    scores = O.prefill_scores(hb, rows)
    nmis = check_selection(idx_gpu, ref["idx"], scores, rows, budget)
    if check_attn:
        att = O.prefill_rows(hb, rows, budget, idx_given=idx_gpu)
        check_outputs(bf16_to_f64(res.out[torch.as_tensor(rows, device=DEV)]), att["o"], "O")
        check_outputs(res.lse.cpu().numpy().astype(np.float64)[rows], att["lse"], "LSE")
    return nmis


# ------------------------------------------------------------------ K-prep --

@pytest.mark.parametrize("L", [5, 1003, 4096])
def test_kprep_block_keys_bit_exact_and_rope(L):
    t = W.prefill_inputs(L, 21, DEV)
    hb = W.host_bits(t)
    cfg = Q.default_config()
    kblk, k_rot = Q.kprep(cfg, t["ki"], t["k"])
    torch.cuda.synchronize()
    assert np.array_equal(W.to_bits(kblk), O.block_keys(hb["ki"]))
    ref = O.rope_keys(hb["k"])
    got = W.to_bits(k_rot)
    assert np.array_equal(got[:, :, 64:], hb["k"][:, :, 64:])
    check_rope(got, ref, hb["k"])


def test_kprep_batched_in_place():
    B, T = 3, 1024
    d = W.decode_inputs(B, T, 22, DEV)
    hd = W.host_bits(d)
    cfg = Q.default_config()
    kblk, k_rot = Q.kprep(cfg, d["ki"], d["k"], k_rot=d["k"])  # in place
    torch.cuda.synchronize()
    for s in range(B):
        assert np.array_equal(W.to_bits(kblk[s]), O.block_keys(hd["ki"][s]))
        check_rope(W.to_bits(k_rot[s]), O.rope_keys(hd["k"][s]), hd["k"][s])


# ------------------------------------------------------------ block scores --

@pytest.mark.parametrize("L", [512, 1029, 4100])
def test_index_scores_dense(L):
    t = W.prefill_inputs(L, 23, DEV)
    hb = W.host_bits(t)
    cfg = Q.default_config()
    sc, st = Q.index_scores(cfg, t["qi"], t["w"], t["ki"])
    torch.cuda.synchronize()
    Q.check_status(st)
    rows = sample_rows(L, 200, seed=L)
    ref = O.prefill_scores(hb, rows)
    check_scores(sc.cpu().numpy().astype(np.float64)[rows], ref)


# --------------------------------------------------------------- selection --

@pytest.mark.parametrize("L,budget,nrows", [(512, 32, None), (4133, 512, 150), (16384 + 7, 64, 120)])
def test_prefill_selection_and_attention(L, budget, nrows):
    t = W.prefill_inputs(L, 24 + budget, DEV)
    hb = W.host_bits(t)
    res = run_prefill(t, budget)
    rows = np.arange(L) if nrows is None else sample_rows(L, nrows, seed=L)
    nmis = oracle_compare_prefill(t, hb, res, rows, budget)
    assert nmis <= max(2, len(rows) // 20)
    # the score output holds the selected blocks' scores
    sc = res.score.cpu().numpy()
    r = rows[-1]
    row = res.idx.cpu().numpy()[r]
    n = min(budget, r // 4 + 1)
    assert np.isinf(sc[r, n - 1]) and sc[r, n - 1] > 0
    assert np.all(np.isneginf(sc[r, n:]))


def test_selection_ties_take_lowest_blocks():
    """w = 0: every score is 0 and the tie rule keeps blocks 0..budget-2."""
    L, budget = 4096 + 64, 512
    t = W.prefill_inputs(L, 25, DEV)
    t["w"].zero_()
    res = run_prefill(t, budget, want_score=False)
    idx = res.idx.cpu().numpy()
    for tt in [2044, 2047, 2048, 3000, L - 1]:
        c = tt // 4
        want = list(range(min(budget - 1, c))) + [c]
        assert list(idx[tt][: len(want)]) == want
        assert np.all(idx[tt][len(want):] == -1)


def test_selection_with_many_compactions():
    """Scores that grow with the block index make every new block beat the
    running threshold, so the candidate lists overflow and compact many
    times; bf16-quantised keys also create exact ties."""
    L, budget = 16384, 512
    t = W.prefill_inputs(L, 26, DEV)
    u = torch.zeros(128, device=DEV)
    u[0] = 1.0
    ramp = torch.arange(L, device=DEV, dtype=torch.float32) / L
    t["ki"] = (ramp[:, None] * u[None, :] * 4.0 + 0.01 * t["ki"].float()).to(torch.bfloat16)
    t["qi"] = (u[None, None, :].expand(L, 4, 128) + 0.0).to(torch.bfloat16).contiguous()
    hb = W.host_bits(t)
    res = run_prefill(t, budget, want_score=False)
    rows = sample_rows(L, 60, seed=3, extra=[L - 1, L - 2, L - 5])
    nmis = oracle_compare_prefill(t, hb, res, rows, budget, check_attn=False)
    assert nmis <= len(rows)


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 7, 9, 15, 16, 17, 31, 33, 64, 65, 127])
def test_tiny_and_ragged_lengths(L):
    """Every row against the oracle; the lengths also fall on both sides of
    the prefill attention's 16 query rows per CTA (a last CTA with 1, 15 or
    16 rows)."""
    budget = 4
    t = W.prefill_inputs(L, 27 + L, DEV)
    hb = W.host_bits(t)
    res = run_prefill(t, budget)
    rows = np.arange(L)
    oracle_compare_prefill(t, hb, res, rows, budget)


def test_budget_one():
    L = 300
    t = W.prefill_inputs(L, 28, DEV)
    hb = W.host_bits(t)
    res = run_prefill(t, 1)
    idx = res.idx.cpu().numpy()
    assert np.array_equal(idx[:, 0], np.arange(L) // 4)
    oracle_compare_prefill(t, hb, res, np.arange(L), 1)


def test_needles_selected_on_gpu():
    L, budget = 16384, 512
    t = W.prefill_inputs(L, 2, DEV, needle=True)
    res = run_prefill(t, budget, want_score=False)
    idx = res.idx.cpu().numpy()
    needles = [int(b) for b in t["needle_blocks"]]
    for tt in range(0, L, 97):
        sel = set(idx[tt].tolist())
        for b in needles:
            if tt // 4 > b:
                assert b in sel, (tt, b)


# ------------------------------------------------------------------ decode --

@pytest.mark.parametrize("budget", [64, 512])
def test_decode_against_oracle(budget):
    B, Tmax = 3, 8192
    lens = [Tmax, 1001, 4 * 700 + 2]
    d = W.decode_inputs(B, Tmax, 30 + budget, DEV, seq_lens=lens)
    hd = W.host_bits(d)
    cfg = Q.default_config(budget=budget)
    k_rot = torch.empty_like(d["k"])
    kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=k_rot)
    out, lse, idx, st = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], k_rot, d["v"], kblk,
                                             d["seq_lens"])
    torch.cuda.synchronize()
    Q.check_status(st)
    idx_g = idx.cpu().numpy()
    ref = O.decode(hd, budget, want_o=False)
    # oracle scores of each sequence's query over its past blocks
    for s in range(B):
        T = lens[s]
        pre = {k_: np.zeros((T,) + hd[k_].shape[1:], np.uint16) for k_ in ("q", "qi", "w")}
        pre.update({"k": hd["k"][s, :T], "v": hd["v"][s, :T], "ki": hd["ki"][s, :T]})
        pre = {k_: np.ascontiguousarray(v_) for k_, v_ in pre.items()}
        pre["qi"][T - 1], pre["w"][T - 1] = hd["qi"][s], hd["w"][s]
        scores = O.prefill_scores(pre, [T - 1])
        check_selection(idx_g[s:s + 1], ref["idx"][s:s + 1], scores, [T - 1], budget)
    att = O.decode(hd, budget, idx_given=idx_g)
    check_outputs(bf16_to_f64(out), att["o"], "O")
    check_outputs(lse.cpu().numpy().astype(np.float64), att["lse"], "LSE")


def test_decode_all_ties():
    """w = 0 makes every block score 0: the selection is blocks 0..budget-2
    plus the current block (lower block wins a tie).  At 65,536 tokens the
    16,383 tied candidates exceed the decode candidate area, which sends the
    final selection over all of the sequence's scores; at 8,192 tokens the
    2,047 ties fit."""
    B, Tmax, budget = 2, 65536, 512
    lens = [Tmax, 8192]
    d = W.decode_inputs(B, Tmax, 32, DEV, seq_lens=lens)
    d["w"].zero_()
    hd = W.host_bits(d)
    cfg = Q.default_config(budget=budget)
    k_rot = torch.empty_like(d["k"])
    kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=k_rot)
    out, lse, idx, st = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], k_rot, d["v"], kblk,
                                             d["seq_lens"])
    torch.cuda.synchronize()
    Q.check_status(st)
    ref = O.decode(hd, budget, want_o=False)
    idx_g = idx.cpu().numpy()
    assert np.array_equal(idx_g, ref["idx"])
    for s_ in range(B):
        c = (lens[s_] - 1) // 4
        assert np.array_equal(idx_g[s_], np.r_[np.arange(budget - 1), c])


def test_decode_budget_one():
    """Budget 1: only the current block is attended."""
    B, Tmax = 3, 4096
    lens = [Tmax, 9, 1]
    d = W.decode_inputs(B, Tmax, 33, DEV, seq_lens=lens)
    hd = W.host_bits(d)
    cfg = Q.default_config(budget=1)
    k_rot = torch.empty_like(d["k"])
    kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=k_rot)
    out, lse, idx, st = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], k_rot, d["v"], kblk,
                                             d["seq_lens"])
    torch.cuda.synchronize()
    Q.check_status(st)
    ref = O.decode(hd, 1)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.array_equal(idx.cpu().numpy()[:, 0], [(T - 1) // 4 for T in lens])
    check_outputs(bf16_to_f64(out), ref["o"], "O")


def test_decode_short_sequences():
    B, Tmax = 4, 64
    lens = [1, 2, 5, 64]
    budget = 8
    d = W.decode_inputs(B, Tmax, 31, DEV, seq_lens=lens)
    hd = W.host_bits(d)
    cfg = Q.default_config(budget=budget)
    k_rot = torch.empty_like(d["k"])
    kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=k_rot)
    out, lse, idx, st = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], k_rot, d["v"], kblk,
                                             d["seq_lens"])
    torch.cuda.synchronize()
    Q.check_status(st)
    ref = O.decode(hd, budget)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    check_outputs(bf16_to_f64(out), ref["o"], "O")


# ------------------------------------------------------------------ YaRN --

def test_yarn_prefill_and_decode():
    """YaRN on (model card: factor 4 over 262,144): RoPE'd keys, prefill and
    decode attention against the oracle with the same setting; the selection
    does not depend on it (the indexer has no RoPE)."""
    L, budget = 4133, 512
    cfg = Q.default_config(budget=budget, yarn_factor=4.0)
    t = W.prefill_inputs(L, 51, DEV)
    hb = W.host_bits(t)
    res = Q.prefill(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"])
    torch.cuda.synchronize()
    Q.check_status(res.status)
    check_rope(W.to_bits(res.k_rot), O.rope_keys(hb["k"], yarn=O.YARN_CARD), hb["k"])
    rows = sample_rows(L, 24, 7)
    idx_g = res.idx.cpu().numpy()[rows]
    ref = O.prefill_rows(hb, rows, budget, want_o=False)
    check_selection(idx_g, ref["idx"], O.prefill_scores(hb, rows), rows, budget)
    att = O.prefill_rows(hb, rows, budget, idx_given=idx_g, yarn=O.YARN_CARD)
    check_outputs(bf16_to_f64(res.out[torch.as_tensor(rows, device=DEV)]), att["o"], "O")
    check_outputs(res.lse.cpu().numpy().astype(np.float64)[rows], att["lse"], "LSE")
    plain = O.prefill_rows(hb, rows[-3:], budget, idx_given=idx_g[-3:])
    assert not np.allclose(plain["lse"], att["lse"][-3:])  # the setting does reach the kernels

    B, Tmax = 2, 8192
    lens = [Tmax, 3001]
    d = W.decode_inputs(B, Tmax, 52, DEV, seq_lens=lens)
    hd = W.host_bits(d)
    k_rot = torch.empty_like(d["k"])
    kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=k_rot)
    out, lse, idx, st = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], k_rot, d["v"], kblk, d["seq_lens"])
    torch.cuda.synchronize()
    Q.check_status(st)
    att = O.decode(hd, budget, idx_given=idx.cpu().numpy(), yarn=O.YARN_CARD)
    check_outputs(bf16_to_f64(out), att["o"], "O")
    check_outputs(lse.cpu().numpy().astype(np.float64), att["lse"], "LSE")


# ------------------------------------------------ locality-structured input --

def test_locality_workload_selects_own_topic_and_matches_oracle():
    """Topic segments of 2048 tokens: selection and outputs against the
    oracle, and most selected past blocks come from the query's own segment
    (the structure that makes neighbouring selections overlap)."""
    L, budget, seg = 12288, 512, 2048
    t = W.prefill_inputs(L, 61, DEV, locality=seg)
    hb = W.host_bits(t)
    res = run_prefill(t, budget)
    rows = sample_rows(L, 32, 8)
    oracle_compare_prefill(t, hb, res, rows, budget)
    idx = res.idx.cpu().numpy()
    late = [r for r in rows if r % seg >= seg // 2 and r >= seg]  # own segment has >= 256 past blocks
    own = []
    for r in late:
        blocks = idx[r][idx[r] >= 0][:-1]
        own.append(np.mean((blocks * 4) // seg == r // seg))
    assert own and np.mean(own) > 0.45


def test_decode_step_replays_as_cuda_graph():
    """The decode step (scan, filter, merge, split attention, combine, with
    programmatic dependent launches) captures into a CUDA graph; replays give
    the eager result bit for bit, with new queries written into the captured
    input buffers between replays."""
    B, Tmax, budget = 4, 16384, 512
    d = W.decode_inputs(B, Tmax, 81, DEV, seq_lens=[Tmax, 9000, 4097, 600])
    cfg = Q.default_config(budget=budget)
    kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=d["k"])
    ws = torch.empty(Q.decode_workspace_bytes(cfg, B, Tmax), dtype=torch.uint8, device=DEV)
    out = torch.empty((B, 24, 256), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, 24), dtype=torch.float32, device=DEV)
    idx = torch.empty((B, budget), dtype=torch.int32, device=DEV)
    status = Q.new_status(DEV)

    def step():
        Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], d["k"], d["v"], kblk, d["seq_lens"], out=out, lse=lse,
                             idx_out=idx, ws=ws, status=status)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    gen = torch.Generator(device=DEV).manual_seed(82)
    for _ in range(2):
        d["q"].copy_(torch.randn(d["q"].shape, generator=gen, device=DEV).to(torch.bfloat16))
        d["qi"].copy_(torch.randn(d["qi"].shape, generator=gen, device=DEV).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        got = (out.clone(), lse.clone(), idx.clone())
        step()
        torch.cuda.synchronize()
        Q.check_status(status)
        assert torch.equal(got[2], idx)
        assert torch.equal(got[0], out)
        assert torch.equal(got[1], lse)


def test_failed_threshold_prediction_is_redone_exactly():
    """Blocks 0..767 score far above every later block, so the threshold the
    indexer predicts from the first tiles of a long row (the rp-th best of
    the first 768 blocks) overshoots the row's final (budget-1)-th best: the
    exactness check fails, the query tile is redone without prediction, and
    the selection still equals the oracle's.  The per-(query tile, group)
    flags of the predicting launch sit after the candidate lists in the
    workspace; some must be set here, which shows the redo launch had work."""
    L, budget = 32768, 512
    t = W.prefill_inputs(L, 57, DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(58)
    u = torch.randn(128, generator=g, device=DEV)
    u = u / u.norm()
    t["qi"] = (t["qi"].float() + 2.0 * u).to(torch.bfloat16)
    ki = t["ki"].float()
    ki[:3072] += 6.0 * float(np.sqrt(128.0)) * u
    t["ki"] = ki.to(torch.bfloat16)
    hb = W.host_bits(t)
    cfg = Q.default_config(budget=budget)
    ws = torch.zeros(Q.index_topk_workspace_bytes(cfg, L), dtype=torch.uint8, device=DEV)
    idx, _, k_rot, st = Q.index_topk(cfg, t["qi"], t["w"], t["ki"], k=t["k"], ws=ws, want_score=False)
    torch.cuda.synchronize()
    Q.check_status(st)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nq = (L + 63) // 64
    kblk_bytes = -(-((L // 4) * 128 * 2 + 16) // 1024) * 1024
    flags = ws[kblk_bytes + min(nq, sms) * 64 * 2048 * 8:][: nq * 4].cpu().numpy()
    assert flags.sum() > 0  # some predictions failed their check
    assert flags[: 16352 // 64 * 4].sum() == 0  # rows with few blocks never predict
    rows = sample_rows(L, 96, seed=57, extra=[16384, 20000, 32767])
    ref = O.prefill_rows(hb, rows, budget, want_o=False)
    scores = O.prefill_scores(hb, rows)
    check_selection(idx.cpu().numpy()[rows], ref["idx"], scores, rows, budget)
