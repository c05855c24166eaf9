"""Parity at the full workload sizes (512 tokens at budget 32, 32K, 128K with
and without needles, 64 x 256K decode, 1M prefill, 8 x 1M decode), run in
the launch configuration the benchmark times, checked against the oracle on
sampled query rows / sequences that the oracle computes one by one (every
row at 512 tokens).  Rules are in tests/parity.py."""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_long_19_b300 import qsa as Q
from block_sparse_long_19_b300 import workloads as W

from .parity import bf16_to_f64, check_outputs, check_rope, check_selection, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def host_for_rows(t, rows):
    """Host bit patterns the oracle needs for the listed rows: all of K, V,
    Ki (any past key may be attended or scored), and only the listed rows of
    Q and Qi (other rows stay zero and are never read)."""
    L = t["q"].shape[0]
    hb = {n: W.to_bits(t[n]) for n in ("k", "v", "ki", "w")}
    hb["q"] = np.zeros((L, 24, 256), np.uint16)
    hb["qi"] = np.zeros((L, 4, 128), np.uint16)
    ri = torch.as_tensor(rows, device=t["q"].device)
    hb["q"][rows] = W.to_bits(t["q"][ri])
    hb["qi"][rows] = W.to_bits(t["qi"][ri])
    return hb


def check_k_rot_tail(t, res, n):
    """RoPE'd keys of the last n positions (the largest angles of the
    workload) against the oracle's rotation, row by row."""
    L = t["k"].shape[0]
    raw = W.to_bits(t["k"][L - n:])
    got = W.to_bits(res.k_rot[L - n:])
    ref = np.stack([np.stack([O.rope_row_bf16(raw[i, g], L - n + i) for g in range(2)]) for i in range(n)])
    assert np.array_equal(got[:, :, 64:], raw[:, :, 64:])
    check_rope(got, ref, raw)


def prefill_check(name, nrows, needle=False, all_rows=False, k_rot_tail=0):
    spec = W.WORKLOADS[name]
    L, budget, seed = spec["L"], spec["budget"], spec["seed"]
    t = W.prefill_inputs(L, seed, DEV, needle=needle)
    cfg = Q.default_config(budget=budget)
    # the benchmark's prefill call: at 1M the indexer of each chunk runs
    # beside the attention of the previous one; shorter prefills run serially
    res = Q.prefill_overlapped(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"], want_score=False)
    torch.cuda.synchronize()
    Q.check_status(res.status, name)
    if k_rot_tail:
        check_k_rot_tail(t, res, k_rot_tail)
    rows = np.arange(L, dtype=np.int64) if all_rows else sample_rows(L, nrows, seed=seed)
    hb = host_for_rows(t, rows)
    idx_gpu = res.idx[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    ref = O.prefill_rows(hb, rows, budget, want_o=False)
    scores = O.prefill_scores(hb, rows)
    nmis = check_selection(idx_gpu, ref["idx"], scores, rows, budget)
    assert nmis <= max(2, len(rows) // 10)
    att = O.prefill_rows(hb, rows, budget, idx_given=idx_gpu)
    check_outputs(bf16_to_f64(res.out[torch.as_tensor(rows, device=DEV)]), att["o"], "O")
    check_outputs(res.lse[torch.as_tensor(rows, device=DEV)].double().cpu().numpy(), att["lse"], "LSE")
    return t, res


def test_prefill_512_every_row():
    """512 tokens at budget 32 from seed 0, every query row."""
    prefill_check("prefill_512", 0, all_rows=True, k_rot_tail=512)


def test_prefill_32k():
    prefill_check("prefill_32k", 64)


def test_prefill_128k_plain():
    """The 128K input without planted blocks (i.i.d. draws only)."""
    prefill_check("prefill_128k", 32)


def test_prefill_128k_with_needles():
    t, res = prefill_check("prefill_128k", 32, needle=True)
    idx = res.idx.cpu().numpy()
    needles = np.array([int(b) for b in t["needle_blocks"]])
    L = idx.shape[0]
    c = np.arange(L) // 4
    for b in needles:
        rows = np.nonzero(c > b)[0]
        hit = (idx[rows] == b).any(axis=1)
        assert hit.all(), (b, int((~hit).sum()))


def test_prefill_1m():
    prefill_check("prefill_1m", 12, k_rot_tail=2048)


def decode_check(name, nseq, noalloc=False):
    spec = W.WORKLOADS[name]
    B, T, budget, seed = spec["B"], spec["T"], spec["budget"], spec["seed"]
    d = W.decode_inputs(B, T, seed, DEV)
    cfg = Q.default_config(budget=budget)
    rng = np.random.default_rng(seed)
    seqs = sorted(set([0, B - 1] + list(rng.integers(0, B, size=max(0, nseq - 2)))))
    # host copies of the raw caches of the checked sequences, taken before the
    # in-place RoPE below
    hd = {n: [W.to_bits(d[n][s]) for s in seqs] for n in ("k", "v", "ki")}
    kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=d["k"])
    del d["ki"]
    out, lse, idx, st = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], d["k"], d["v"], kblk,
                                             d["seq_lens"])
    torch.cuda.synchronize()
    Q.check_status(st, name)
    if noalloc:
        # the same step through the entry point that uses the library's
        # built-in scratch array: the same kernels, so the same bits
        o2, l2, i2, st2 = Q.sparse_attn_decode_noalloc(cfg, d["q"], d["qi"], d["w"], d["k"], d["v"], kblk,
                                                       d["seq_lens"])
        torch.cuda.synchronize()
        Q.check_status(st2, name + " (no-alloc)")
        assert torch.equal(i2, idx) and torch.equal(o2, out) and torch.equal(l2, lse)
    for j, s in enumerate(seqs):
        one = {
            "q": W.to_bits(d["q"][s:s + 1]), "qi": W.to_bits(d["qi"][s:s + 1]),
            "w": W.to_bits(d["w"][s:s + 1]), "k": hd["k"][j][None], "v": hd["v"][j][None],
            "ki": hd["ki"][j][None], "seq_lens": np.array([T], np.int64),
        }
        idx_g = idx[s:s + 1].cpu().numpy()
        ref = O.decode(one, budget, want_o=False)
        pre = {"qi": np.zeros((T, 4, 128), np.uint16), "w": np.zeros((T, 4), np.uint16),
               "ki": hd["ki"][j]}
        pre["qi"][T - 1], pre["w"][T - 1] = one["qi"][0], one["w"][0]
        scores = O.prefill_scores(pre, [T - 1])
        check_selection(idx_g, ref["idx"], scores, [T - 1], budget)
        att = O.decode(one, budget, idx_given=idx_g)
        check_outputs(bf16_to_f64(out[s:s + 1]), att["o"], "O")
        check_outputs(lse[s:s + 1].double().cpu().numpy(), att["lse"], "LSE")


def test_decode_64x256k():
    decode_check("decode_64x256k", 4)


def test_decode_8x1m():
    decode_check("decode_8x1m", 2, noalloc=True)
