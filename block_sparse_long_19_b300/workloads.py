"""Seeded synthetic inputs for the QSA layer.

This module only draws random tensors of the right shapes and distributions;
it holds none of the attention/indexer arithmetic, so both the CUDA path and
the CPU oracle can be fed from it.

Shapes follow the model card of Qwen3.8-Flash-Next ("Model Overview / Qwen
Sparse Attention"): 24 query heads and 2 KV heads of dim 256, an indexer with
4 query heads and one shared key head of dim 128, per-head indexer weights.
Q, K, V, Qi, Ki ~ N(0, 1) rounded to bf16; w ~ U(0, 1) rounded to bf16.
The pages measure on no dataset; these i.i.d. draws stand in for the 128K-1M
token contexts the pages quote.

The workloads (name -> sizes):
  prefill_512      L=512,     budget 32,  seed 0
  prefill_32k      L=32768,   budget 512, seed 1
  prefill_128k     L=131072,  budget 512, seed 2  (+ planted-needle variant)
  decode_64x256k   64 sequences x 262144 cached tokens, budget 512, seed 3
  prefill_1m       L=1048576, budget 512, seed 4
  decode_8x1m      8 sequences x 1048576 cached tokens, budget 512, seed 4

Locality variant (prefill_inputs(..., locality=S)): neighbouring queries share
a topic, so their selections overlap -- the structure real long contexts
have and i.i.d. draws lack (see locality_plant).
"""
from __future__ import annotations

import math

import torch

HQ, HKV, D = 24, 2, 256
HI, DI = 4, 128

WORKLOADS = {
    "prefill_512": dict(kind="prefill", L=512, budget=32, seed=0),
    "prefill_32k": dict(kind="prefill", L=32768, budget=512, seed=1),
    "prefill_128k": dict(kind="prefill", L=131072, budget=512, seed=2),
    "decode_64x256k": dict(kind="decode", B=64, T=262144, budget=512, seed=3),
    "prefill_1m": dict(kind="prefill", L=1048576, budget=512, seed=4),
    "decode_8x1m": dict(kind="decode", B=8, T=1048576, budget=512, seed=4),
}

# Needle variant of prefill_128k: how many planted blocks and how strong.
NEEDLE_BLOCKS = 8
NEEDLE_Q_GAIN = 3.0


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, g, device, chunk_rows: int = 1 << 16) -> torch.Tensor:
    """N(0,1) in bf16, drawn in row chunks so no large fp32 temporary exists."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                                  dtype=torch.float32).to(torch.bfloat16)
    return out


def _uniform(shape, g, device) -> torch.Tensor:
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def prefill_inputs(L: int, seed: int, device="cpu", needle: bool = False, locality: int = 0) -> dict:
    """One sequence of L tokens: q [L,24,256], k/v [L,2,256] (k before RoPE),
    qi [L,4,128], w [L,4], ki [L,128].  With needle=True, also returns
    'needle_blocks' (int64 [8]) -- see needle_plant.  locality=S > 0 plants
    topic segments of S tokens (see locality_plant)."""
    g = _gen(device, seed)
    t = {
        "q": _normal((L, HQ, D), g, device),
        "k": _normal((L, HKV, D), g, device),
        "v": _normal((L, HKV, D), g, device),
        "qi": _normal((L, HI, DI), g, device),
        "ki": _normal((L, DI), g, device),
        "w": _uniform((L, HI), g, device),
    }
    if needle:
        needle_plant(t, seed, device)
    if locality:
        locality_plant(t, seed, locality, device)
    return t


LOCALITY_GAIN = 3.0


def locality_plant(t: dict, seed: int, seg: int, device, chunk_rows: int = 1 << 16) -> None:
    """Topic segments: tokens [s*seg, (s+1)*seg) share a random unit
    direction u_s in R^128; every indexer query head of those tokens gets
    +3.0*u_s and their indexer keys +3.0*sqrt(128)*u_s.  A query's own
    segment then outscores the rest of the context, so nearby queries select
    mostly the same blocks.  Values are rounded to bf16."""
    L = t["ki"].shape[0]
    g = _gen(device, seed + 2000)
    nseg = (L + seg - 1) // seg
    u = torch.randn(nseg, DI, generator=g, device=device, dtype=torch.float32)
    u = u / u.norm(dim=1, keepdim=True)
    for r0 in range(0, L, chunk_rows):
        r1 = min(L, r0 + chunk_rows)
        us = u[torch.arange(r0, r1, device=device) // seg]          # [rows, 128]
        t["qi"][r0:r1] = (t["qi"][r0:r1].float() + LOCALITY_GAIN * us[:, None, :]).to(torch.bfloat16)
        t["ki"][r0:r1] = (t["ki"][r0:r1].float() + LOCALITY_GAIN * math.sqrt(DI) * us).to(torch.bfloat16)


def needle_plant(t: dict, seed: int, device) -> None:
    """Planted-needle variant: a random unit direction u in R^128; every
    indexer query head gets +3.0*u, and the 4 indexer keys of each of 8
    random blocks get +3.0*sqrt(128)*u, so those blocks should be selected by
    every later query.  Values are rounded to bf16."""
    L = t["ki"].shape[0]
    g = _gen(device, seed + 1000)
    u = torch.randn(DI, generator=g, device=device, dtype=torch.float32)
    u = u / u.norm()
    nb = L // 4
    # needles in the first 3/4 of the sequence so most queries can see them
    blocks = torch.randperm(max(nb * 3 // 4, NEEDLE_BLOCKS), generator=g, device=device)[:NEEDLE_BLOCKS]
    blocks = torch.sort(blocks).values
    t["qi"] = (t["qi"].float() + NEEDLE_Q_GAIN * u).to(torch.bfloat16)
    ki = t["ki"].float()
    for b in blocks.tolist():
        ki[4 * b:4 * b + 4] += NEEDLE_Q_GAIN * math.sqrt(DI) * u
    t["ki"] = ki.to(torch.bfloat16)
    t["needle_blocks"] = blocks.to(torch.int64)


def decode_inputs(B: int, T: int, seed: int, device="cpu", Tmax: int | None = None,
                  seq_lens=None) -> dict:
    """B sequences with caches [B, Tmax, ...] holding raw (pre-RoPE) keys,
    values and per-token indexer keys, plus one new query per sequence.
    seq_lens[s] counts the new token (already in the cache at T-1)."""
    Tmax = T if Tmax is None else Tmax
    g = _gen(device, seed)
    t = {
        "q": _normal((B, HQ, D), g, device),
        "qi": _normal((B, HI, DI), g, device),
        "w": _uniform((B, HI), g, device),
        "k": _normal((B * Tmax, HKV, D), g, device).view(B, Tmax, HKV, D),
        "v": _normal((B * Tmax, HKV, D), g, device).view(B, Tmax, HKV, D),
        "ki": _normal((B * Tmax, DI), g, device).view(B, Tmax, DI),
    }
    if seq_lens is None:
        seq_lens = [T] * B
    t["seq_lens"] = torch.tensor(seq_lens, dtype=torch.int32, device=device)
    return t


def to_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    import numpy as np

    return x.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_bits(t: dict) -> dict:
    """Host numpy copies of a workload dict (bf16 as uint16 bits)."""
    import numpy as np

    out = {}
    for k_, v_ in t.items():
        if v_.dtype == torch.bfloat16:
            out[k_] = to_bits(v_)
        else:
            out[k_] = v_.detach().cpu().numpy().astype(np.int64)
    return out
