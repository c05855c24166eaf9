"""The decode entry point that allocates nothing.

qsa_sparse_attn_decode_noalloc serves callers that cannot allocate device
memory when they run a decode step (a host program whose device memory is
owned by another runtime, or a serving loop that must not call
cudaMalloc/cudaFree mid-request); it uses the library's built-in 16 MiB
scratch array instead of a workspace argument.  It runs the same kernels on
the same inputs as qsa_sparse_attn_decode with a caller workspace, so its
selection, output and log-sum-exp must be the same bit for bit, on two calls
in a row (the second call finds the first call's data in the shared array).
This file is collected last so that a failure here cannot hide another
test's result.
"""
import ctypes

import pytest
import torch

from block_sparse_long_19_b300 import qsa as Q
from block_sparse_long_19_b300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _decode_both(B, Tmax, lens, seed, budget=512):
    d = W.decode_inputs(B, Tmax, seed, DEV, seq_lens=lens)
    cfg = Q.default_config(budget=budget)
    kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=d["k"])
    ref = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], d["k"], d["v"], kblk, d["seq_lens"])
    torch.cuda.synchronize()
    Q.check_status(ref[3], "decode with workspace")
    for _ in range(2):
        out, lse, idx, st = Q.sparse_attn_decode_noalloc(cfg, d["q"], d["qi"], d["w"], d["k"], d["v"], kblk,
                                                         d["seq_lens"])
        torch.cuda.synchronize()
        Q.check_status(st, "decode without allocation")
        assert torch.equal(idx, ref[2])
        assert torch.equal(out, ref[0])
        assert torch.equal(lse, ref[1])


def test_noalloc_decode_matches_workspace_decode():
    _decode_both(3, 8192, [8192, 1001, 4 * 700 + 2], 77)


def test_noalloc_decode_near_its_scratch_limit():
    """4 sequences of 2M tokens: a workspace of about 12 MB of the 16 MiB
    (the same block-score area as 8 x 1M)."""
    cfg = Q.default_config()
    need = Q.decode_workspace_bytes(cfg, 4, 1 << 21)
    assert (8 << 20) < need <= (16 << 20)
    _decode_both(4, 1 << 21, [1 << 21, (1 << 21) - 3, 1_500_001, 4 * 300_000], 78)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """256 sequences x 1M tokens need more than 16 MiB of decode scratch: the
    call is refused before anything is launched.  The pointers are real (if
    small) device buffers all the same."""
    cfg = Q.default_config()
    lib = Q.load()
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    A = ctypes.c_void_p(buf.data_ptr())
    need = lib.qsa_decode_workspace_bytes(ctypes.byref(cfg), 256, 1 << 20)
    assert need > (16 << 20)
    rc = lib.qsa_sparse_attn_decode_noalloc(ctypes.byref(cfg), 256, A, A, A, A, A, A, 1 << 20, A, A,
                                            None, None, A, None)
    assert rc == 2
    assert b"16 MiB" in lib.qsa_last_error_detail()
    rc = lib.qsa_sparse_attn_decode_noalloc(ctypes.byref(cfg), 0, A, A, A, A, A, A, 1024, A, A,
                                            None, None, A, None)
    assert rc == 1
    torch.cuda.synchronize()
    assert int(buf.count_nonzero()) == 0
