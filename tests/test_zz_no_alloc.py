"""The decode entry point that allocates nothing.

qsa_sparse_attn_decode_noalloc serves callers that cannot allocate device
memory when they run a decode step (a host program whose device memory is
owned by another runtime, or a serving loop that must not call
cudaMalloc/cudaFree mid-request); it uses the library's built-in 16 MiB
scratch array instead of a workspace argument.  Here it must give the same
selection and, within the parity tolerance, the same outputs as
qsa_sparse_attn_decode with a caller workspace, on two calls in a row (the
second call finds the first call's data in the shared array).  This file is
collected last so that a failure here cannot hide another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_long_19_b300 import qsa as Q
from block_sparse_long_19_b300 import workloads as W

from .parity import bf16_to_f64, check_outputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_noalloc_decode_matches_workspace_decode():
    B, Tmax, budget = 3, 8192, 512
    lens = [Tmax, 1001, 4 * 700 + 2]
    d = W.decode_inputs(B, Tmax, 77, DEV, seq_lens=lens)
    cfg = Q.default_config(budget=budget)
    kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=d["k"])
    out_ref, lse_ref, idx_ref, st = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], d["k"],
                                                         d["v"], kblk, d["seq_lens"])
    torch.cuda.synchronize()
    Q.check_status(st, "decode with workspace")
    for _ in range(2):
        out, lse, idx, st = Q.sparse_attn_decode_noalloc(cfg, d["q"], d["qi"], d["w"], d["k"],
                                                         d["v"], kblk, d["seq_lens"])
        torch.cuda.synchronize()
        Q.check_status(st, "decode without allocation")
        assert torch.equal(idx, idx_ref)
        check_outputs(bf16_to_f64(out), bf16_to_f64(out_ref), "O")
        check_outputs(lse.double().cpu().numpy(), lse_ref.double().cpu().numpy(), "LSE")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """256 sequences x 1M tokens need more than 16 MiB of decode scratch: the
    call is refused before anything is launched (the pointers are never
    read on this path)."""
    cfg = Q.default_config()
    lib = Q.load()
    A = ctypes.c_void_p(0x10000)
    need = lib.qsa_decode_workspace_bytes(ctypes.byref(cfg), 256, 1 << 20)
    assert need > (16 << 20)
    rc = lib.qsa_sparse_attn_decode_noalloc(ctypes.byref(cfg), 256, A, A, A, A, A, A, 1 << 20, A, A,
                                            None, None, A, None)
    assert rc == 2
    assert b"16 MiB" in lib.qsa_last_error_detail()
