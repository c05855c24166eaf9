"""Pins of the CPU oracle against things other than itself (CPU only).

Every check below rests on the pages' printed constants, on a closed form,
on an invariant, on a library routine in a special case where the method
reduces to it, or on brute force over tiny inputs.  Together they are chosen
so that a dropped term, a wrong sign, a wrong index or head mapping, a
transposed operand or a wrong tie rule in the oracle fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_long_19_b300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(x: torch.Tensor) -> np.ndarray:
    return W.to_bits(x.to(torch.bfloat16))


def from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


# ----------------------------------------------------------- page values --

def test_constants_match_pages():
    """Shapes/constants the oracle uses equal the values printed on the
    model card (fixture cites where each is printed)."""
    g = json.load(open(os.path.join(GOLDEN, "qsa_page_constants.json")))
    assert O.HQ == g["n_q_heads"]["value"]
    assert O.HKV == g["n_kv_heads"]["value"]
    assert O.D == g["head_dim"]["value"]
    assert O.RD == g["rope_dim"]["value"]
    assert O.RD == g["partial_rotary_factor"]["value"] * g["head_dim"]["value"]
    assert O.HI == g["n_idx_heads"]["value"]
    assert O.DI == g["idx_dim"]["value"]
    assert O.THETA == g["rope_theta"]["value"]
    # 512 blocks <-> 2048 tokens fixes the micro-block size
    assert O.BS * g["budget_blocks"]["value"] == g["budget_tokens"]["value"]


# --------------------------------------------------------------- rounding --

def test_bf16_rounding_matches_torch():
    """double -> bf16 equals torch's float32 -> bf16 (round-to-nearest-even)
    on values exactly representable in float32, including exact ties."""
    rng = np.random.default_rng(0)
    x = rng.standard_normal(4000).astype(np.float32) * np.float32(3.0)
    ties = np.array([1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -(1.0 + 2.0**-8), 2.0**-130,
                     3.0 * 2.0**-134, 65280.0, 0.0, -0.0, 1.0e-38], dtype=np.float32)
    x = np.concatenate([x, ties])
    want = bits(torch.from_numpy(x))
    got = O.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_rounding_sticky_beyond_float():
    """A value just above a bf16 tie that float32 cannot hold must still
    round up (direct rounding, no double rounding through float32)."""
    x = 1.0 + 2.0**-8 + 2.0**-40
    assert O.f64_to_bf16_bits(np.array([x]))[0] == 0x3F81
    assert O.f64_to_bf16_bits(np.array([1.0 + 2.0**-8]))[0] == 0x3F80


# ----------------------------------------------------------- block keys --

def test_block_keys_equal_torch_mean():
    """kblk = mean of the 4 keys of each block, rounded to bf16 (RNE):
    torch float64 mean over the view [L/4, 4, 128], converted through
    float32 (exact here, checked) to bf16."""
    g = torch.Generator().manual_seed(1)
    L = 4 * 37 + 3  # ragged tail: 3 tokens form no complete block
    ki = torch.randn(L, 128, generator=g).to(torch.bfloat16)
    got = O.block_keys(bits(ki))
    assert got.shape == (L // 4, 128)
    mean64 = ki[: (L // 4) * 4].double().view(L // 4, 4, 128).mean(dim=1)
    assert torch.equal(mean64.float().double(), mean64)  # float32 holds it exactly
    want = bits(mean64.float())
    assert np.array_equal(got, want)


def test_block_keys_tie_to_even():
    """Mean landing exactly on a bf16 tie rounds to the even neighbour."""
    one = 1.0
    ki = torch.zeros(8, 128, dtype=torch.float32)
    ki[:4, 0] = torch.tensor([one, one, one, one + 2.0**-6])      # mean 1 + 2^-8: tie -> 1.0
    ki[4:, 0] = torch.tensor([one, one, one, one + 3 * 2.0**-6])  # mean 1 + 3*2^-8: tie -> 1 + 2^-6
    got = O.block_keys(bits(ki))
    assert got[0, 0] == 0x3F80
    assert got[1, 0] == 0x3F82


# ------------------------------------------------------------------ RoPE --

@pytest.mark.parametrize("pos", [0, 1, 7, 262143, 1048575])
def test_rope_closed_form_unit_vectors(pos):
    """e_i -> (cos a) e_i + (sin a) e_{i+32};  e_{i+32} -> -(sin a) e_i + (cos a) e_{i+32},
    a = pos * theta^(-2i/64): fixes the pairing, the sign and the frequency."""
    for i in [0, 1, 5, 17, 31]:
        a = pos * O.THETA ** (-2.0 * i / 64.0)
        x = np.zeros(O.D, dtype=np.uint16)
        x[i] = 0x3F80  # 1.0
        r = O.rope_exact(x, pos)
        exp = np.zeros(64)
        exp[i], exp[i + 32] = math.cos(a), math.sin(a)
        assert np.allclose(r, exp, rtol=0, atol=1e-12)
        x = np.zeros(O.D, dtype=np.uint16)
        x[i + 32] = 0x3F80
        r = O.rope_exact(x, pos)
        exp = np.zeros(64)
        exp[i], exp[i + 32] = -math.sin(a), math.cos(a)
        assert np.allclose(r, exp, rtol=0, atol=1e-12)


def test_rope_identity_at_zero_and_passthrough():
    g = torch.Generator().manual_seed(2)
    x = bits(torch.randn(O.D, generator=g))
    assert np.array_equal(O.rope_row_bf16(x, 0), x)
    y = O.rope_row_bf16(x, 12345)
    assert np.array_equal(y[64:], x[64:])
    assert not np.array_equal(y[:64], x[:64])


def test_rope_norm_and_relative_position():
    """Rotation preserves the norm, and q(p+d).k(s+d) = q(p).k(s)."""
    g = torch.Generator().manual_seed(3)
    for _ in range(5):
        q = bits(torch.randn(O.D, generator=g))
        k = bits(torch.randn(O.D, generator=g))
        p, s, d = [int(v) for v in torch.randint(0, 1 << 20, (3,), generator=g)]
        qf = O.bf16_bits_to_f64(q[:64])
        assert abs(np.linalg.norm(O.rope_exact(q, p)) - np.linalg.norm(qf)) < 1e-12 * np.linalg.norm(qf)
        a = O.rope_exact(q, p) @ O.rope_exact(k, s)
        b = O.rope_exact(q, p + d) @ O.rope_exact(k, s + d)
        assert abs(a - b) < 1e-9 * (1 + abs(a))


# ------------------------------------------------------------------ YaRN --
# YaRN (model card "Processing Ultra-Long Texts": factor 4 over 262,144; the
# published method): a frequency whose wavelength fits more than beta = 32
# times into the original context keeps its value; one whose wavelength is
# longer than the original context (r < alpha = 1) is interpolated by the
# factor; in between the two are blended.

def _wavelength_ratio(i):
    return O.YARN_CARD[1] / (2 * math.pi / O.THETA ** (-2.0 * i / 64.0))


def test_yarn_off_is_plain_rope():
    assert np.array_equal(O.rope_inv_freq(O.THETA, None), O.rope_inv_freq(O.THETA, (1.0, 262144.0, 1.0, 32.0)))
    assert O.yarn_logit_factor(1.0) == 1.0


def test_yarn_keeps_fast_dims_and_interpolates_slow_dims():
    """Fast rotary pairs rotate exactly as without YaRN; slow pairs rotate at
    position 4p exactly as without YaRN at p (position interpolation by the
    factor 4).  Checked on the rotation itself, through rope_exact."""
    g = torch.Generator().manual_seed(41)
    fast = [i for i in range(32) if _wavelength_ratio(i) > 32.0]
    slow = [i for i in range(32) if _wavelength_ratio(i) < 1.0]
    assert fast and slow and max(fast) < min(slow)
    for _ in range(4):
        x = bits(torch.randn(O.D, generator=g))
        p = int(torch.randint(0, 1 << 18, (1,), generator=g))
        plain_p = O.rope_exact(x, p)
        yarn_p = O.rope_exact(x, p, yarn=O.YARN_CARD)
        yarn_4p = O.rope_exact(x, 4 * p, yarn=O.YARN_CARD)
        plain_4p = O.rope_exact(x, 4 * p)
        for i in fast:
            assert yarn_p[i] == plain_p[i] and yarn_p[i + 32] == plain_p[i + 32]
            assert yarn_4p[i] == plain_4p[i]
        for i in slow:
            assert yarn_4p[i] == plain_p[i] and yarn_4p[i + 32] == plain_p[i + 32]


def test_yarn_blend_is_between_and_monotone():
    w = O.rope_inv_freq(O.THETA, None)
    wy = O.rope_inv_freq(O.THETA, O.YARN_CARD)
    assert np.all(wy <= w) and np.all(wy >= w / 4.0)
    assert np.all(np.diff(wy) < 0)  # still strictly decreasing frequencies
    mid = [i for i in range(32) if 1.0 < _wavelength_ratio(i) < 32.0]
    assert mid and all(w[i] / 4.0 < wy[i] < w[i] for i in mid)


def test_yarn_temperature_scales_logits_only():
    """With the rotary dims zero, RoPE cannot matter: YaRN attention equals
    plain attention with the softmax scale times the YaRN logit factor."""
    g = torch.Generator().manual_seed(43)
    L = 24
    q = torch.randn(L, 24, 256, generator=g)
    k = torch.randn(L, 2, 256, generator=g)
    q[..., :64] = 0
    k[..., :64] = 0
    hb = {"q": bits(q), "k": bits(k), "v": bits(torch.randn(L, 2, 256, generator=g)),
          "qi": bits(torch.randn(L, 4, 128, generator=g)), "w": bits(torch.rand(L, 4, generator=g)),
          "ki": bits(torch.randn(L, 128, generator=g))}
    rows = [3, 11, 23]
    y = O.prefill_rows(hb, rows, 512, yarn=O.YARN_CARD)
    f = O.yarn_logit_factor(4.0)
    assert f > 1.0
    p = O.prefill_rows(hb, rows, 512, scale=O.SCALE * f)
    assert np.array_equal(y["idx"], p["idx"])
    assert np.allclose(y["o"], p["o"], rtol=0, atol=1e-12)
    assert np.allclose(y["lse"], p["lse"], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- scores --

def _kblk_and_q(seed, nb=50, positive=False):
    g = torch.Generator().manual_seed(seed)
    kblk = torch.randn(nb, 128, generator=g)
    qi = torch.randn(4, 128, generator=g)
    if positive:
        kblk, qi = kblk.abs(), qi.abs()
    return bits(kblk), bits(qi)


@pytest.mark.parametrize("h", [0, 1, 2, 3])
def test_scores_one_head_is_matmul(h):
    """With w = e_h and all dot products positive, the block score is the
    plain matmul qi[h] @ kblk^T (fixes head indexing and operand layout)."""
    kblk, qi = _kblk_and_q(10 + h, positive=True)
    w = np.zeros(4, dtype=np.uint16)
    w[h] = 0x3F80
    got = O.block_scores(qi, w, kblk)
    want = (from_bits(qi).double()[h] @ from_bits(kblk).double().T).numpy()
    assert np.allclose(got, want, rtol=1e-13, atol=0)


def test_scores_relu_and_linearity_in_w():
    """Negative dot products contribute exactly 0 (ReLU); scores are linear
    in the head weights (w is a per-head factor outside the ReLU)."""
    kblk, qi = _kblk_and_q(20, positive=True)
    neg_qi = bits(-from_bits(qi).float())
    w1 = bits(torch.tensor([0.25, 0.5, 0.75, 1.0]))
    assert np.all(O.block_scores(neg_qi, w1, kblk) == 0.0)

    kblk, qi = _kblk_and_q(21)
    wa = bits(torch.tensor([0.5, 0.0, 0.25, 1.0]))
    wb = bits(torch.tensor([0.0, 0.75, 0.5, 0.125]))
    wab = bits(torch.tensor([0.5, 0.75, 0.75, 1.125]))
    w2a = bits(torch.tensor([1.0, 0.0, 0.5, 2.0]))
    sa, sb, sab = (O.block_scores(qi, w, kblk) for w in (wa, wb, wab))
    assert np.allclose(sa + sb, sab, rtol=1e-12, atol=1e-12)
    assert np.allclose(2 * sa, O.block_scores(qi, w2a, kblk), rtol=1e-12, atol=1e-12)
    # relu is applied per head: the score is never below the best single head term
    dots = from_bits(qi).double() @ from_bits(kblk).double().T
    wv = from_bits(wa).double()
    term = (wv[:, None] * dots.clamp(min=0)).numpy()
    assert np.all(sa >= term.max(axis=0) - 1e-12)


# ------------------------------------------------------------- selection --

def test_select_equals_full_sort():
    rng = np.random.default_rng(5)
    for c, budget in [(0, 4), (3, 4), (4, 4), (5, 4), (100, 9), (1000, 512), (600, 512)]:
        s = np.round(rng.standard_normal(max(c, 1)) * 4) / 4  # many exact ties
        sel, ss, n = O.select(s[:c], c, budget)
        ranked = sorted(range(c), key=lambda b: (-s[b], b))[: budget - 1]
        want = sorted(ranked) + [c]
        assert n == len(want)
        assert list(sel[:n]) == want
        assert np.all(sel[n:] == -1)
        assert ss[n - 1] == np.inf and np.all(ss[n:] == -np.inf)
        assert np.array_equal(ss[: n - 1], s[want[:-1]])


def test_select_all_ties_takes_lowest_blocks():
    """w = 0 makes every score 0: the tie rule keeps blocks 0..budget-2."""
    c, budget = 700, 512
    sel, _, n = O.select(np.zeros(c), c, budget)
    assert n == budget
    assert list(sel) == list(range(budget - 1)) + [c]


# ------------------------------------------------------------- attention --

def _tiny(L, seed):
    t = W.prefill_inputs(L, seed, "cpu")
    return t, W.host_bits(t)


def _rope_all(hb, L):
    q = np.stack([[O.rope_row_bf16(hb["q"][t, h], t) for h in range(24)] for t in range(L)])
    k = O.rope_keys(hb["k"])
    return from_bits(q).double(), from_bits(k).double()


def test_dense_budget_equals_causal_sdpa():
    """Budget covering every block: QSA = dense causal GQA attention
    (torch SDPA in fp64, K/V repeated 12x per KV head, scale 1/16)."""
    L = 4 * 9 + 2
    t, hb = _tiny(L, 7)
    rows = np.arange(L)
    res = O.prefill_rows(hb, rows, budget=64)
    q, k = _rope_all(hb, L)
    v = from_bits(hb["v"]).double()
    qh = q.permute(1, 0, 2)                                  # [24, L, 256]
    kh = k.permute(1, 0, 2).repeat_interleave(12, dim=0)     # [24, L, 256]
    vh = v.permute(1, 0, 2).repeat_interleave(12, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, is_causal=True)
    assert np.allclose(res["o"], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    logits = (qh @ kh.transpose(1, 2)) / 16.0
    logits = logits.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool), 1), -math.inf)
    lse = torch.logsumexp(logits, dim=-1).T.numpy()
    assert np.allclose(res["lse"], lse, rtol=1e-12, atol=1e-12)


def test_first_token_returns_its_value():
    """t = 0 attends only to itself: O[0, h] = V[0, h // 12] exactly."""
    t, hb = _tiny(8, 8)
    res = O.prefill_rows(hb, [0], budget=4)
    v = from_bits(hb["v"]).double().numpy()
    for h in range(24):
        assert np.array_equal(res["o"][0, h], v[0, h // 12])


def test_budget_one_block_start_returns_its_value():
    """Budget 1 keeps only the current block; at t = 4c the causal mask
    leaves only key t, so O[t, h] = V[t, h // 12]."""
    L = 64
    t, hb = _tiny(L, 9)
    rows = [4, 8, 40, 60]
    res = O.prefill_rows(hb, rows, budget=1)
    v = from_bits(hb["v"]).double().numpy()
    for r, tt in enumerate(rows):
        assert list(res["idx"][r]) == [tt // 4]
        for h in range(24):
            assert np.array_equal(res["o"][r, h], v[tt, h // 12])


def test_constant_values_pass_through():
    L = 40
    t, hb = _tiny(L, 10)
    row = np.full(256, 0x3FC0, dtype=np.uint16)  # 1.5
    hb["v"] = np.ascontiguousarray(np.broadcast_to(row, hb["v"].shape))
    res = O.prefill_rows(hb, [5, 17, 39], budget=3)
    assert np.allclose(res["o"], 1.5, rtol=0, atol=1e-14)


def test_brute_force_tiny_pipeline():
    """Tiny L, small budget: (1) the selection keeps the current block and
    the budget-1 best past blocks by (score desc, index asc), checked against
    scores from a plain torch matmul; (2) the output equals torch SDPA with an
    explicit mask of the selected, causal keys."""
    L, budget = 4 * 16 + 3, 4
    t, hb = _tiny(L, 11)
    rows = np.arange(L)
    res = O.prefill_rows(hb, rows, budget=budget)
    ki = from_bits(hb["ki"]).double()
    kblk = torch.from_numpy(
        O.bf16_bits_to_f64(bits(ki[: (L // 4) * 4].view(L // 4, 4, 128).mean(1).float()))
    )
    qi = from_bits(hb["qi"]).double()
    w = from_bits(hb["w"]).double()
    q, k = _rope_all(hb, L)
    v = from_bits(hb["v"]).double()
    for r, tt in enumerate(rows):
        c = tt // 4
        s = (w[tt][:, None] * (qi[tt] @ kblk.T).clamp(min=0)).sum(0).numpy()[:c]
        best = sorted(range(c), key=lambda b: (-s[b], b))[: budget - 1]
        want = sorted(best) + [c]
        got = [b for b in res["idx"][r] if b >= 0]
        assert got == want, (tt, got, want)
        mask = torch.zeros(L, dtype=torch.bool)
        for b in want:
            mask[4 * b: 4 * b + 4] = True
        mask[tt + 1:] = False
        qh = q[tt].unsqueeze(1)                                   # [24, 1, 256]
        kh = k.permute(1, 0, 2).repeat_interleave(12, dim=0)      # [24, L, 256]
        vh = v.permute(1, 0, 2).repeat_interleave(12, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask[None, None, :])
        assert np.allclose(res["o"][r], ref[:, 0].numpy(), rtol=1e-10, atol=1e-12)


def test_softmax_weights_sum_to_one_via_lse():
    """sum_j exp(z_j - lse) = 1 for each head (z from torch on RoPE'd bf16)."""
    L = 48
    t, hb = _tiny(L, 12)
    rows = [47]
    res = O.prefill_rows(hb, rows, budget=64)
    q, k = _rope_all(hb, L)
    z = torch.einsum("hd,jhd->hj", q[47], k.repeat_interleave(12, dim=1)[:48]) / 16.0
    tot = torch.exp(z - torch.from_numpy(res["lse"][0])[:, None]).sum(1)
    assert np.allclose(tot.numpy(), 1.0, rtol=0, atol=1e-12)


# ----------------------------------------------------------------- decode --

def test_decode_equals_prefill_last_row():
    """A decode step over a cache filled from a sequence equals that
    sequence's prefill at its last position (selection and output)."""
    B, T, budget = 3, 4 * 20 + 1, 6
    lens = [T, T - 1, 4 * 20]
    d = W.decode_inputs(B, T, 13, "cpu", seq_lens=lens)
    hd = W.host_bits(d)
    got = O.decode(hd, budget)
    for s in range(B):
        Ts = lens[s]
        pre = {
            "q": np.zeros((Ts, 24, 256), np.uint16), "k": hd["k"][s, :Ts], "v": hd["v"][s, :Ts],
            "qi": np.zeros((Ts, 4, 128), np.uint16), "w": np.zeros((Ts, 4), np.uint16), "ki": hd["ki"][s, :Ts],
        }
        pre = {k_: np.ascontiguousarray(v_) for k_, v_ in pre.items()}
        pre["q"][Ts - 1], pre["qi"][Ts - 1], pre["w"][Ts - 1] = hd["q"][s], hd["qi"][s], hd["w"][s]
        ref = O.prefill_rows(pre, [Ts - 1], budget)
        assert np.array_equal(got["idx"][s], ref["idx"][0])
        assert np.array_equal(got["o"][s], ref["o"][0])
        assert np.array_equal(got["lse"][s], ref["lse"][0])


# ----------------------------------------------------------------- needle --

def test_needle_blocks_are_selected():
    """Planted-needle variant: every query whose current block is past a
    needle block selects it."""
    L, budget = 4096, 64
    t = W.prefill_inputs(L, 2, "cpu", needle=True)
    hb = W.host_bits(t)
    needles = [int(b) for b in t["needle_blocks"]]
    rows = np.arange(0, L, 37)
    res = O.prefill_rows(hb, rows, budget, want_o=False)
    for r, tt in enumerate(rows):
        sel = set(int(b) for b in res["idx"][r])
        for b in needles:
            if tt // 4 > b:
                assert b in sel, (tt, b)
