"""The tcgen05 attention kernel (selected with QSA_ATTENTION_KERNEL=tc when
the library is first used in a process) through the same parity tests as the
default kernel, in a child process of its own.

The two kernels compute the same attention in different arithmetic orders:
on one input their outputs agree within the parity tolerance but not bit for
bit, which also shows that the child really ran the other kernel."""
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest
import torch

from block_sparse_long_19_b300 import qsa as Q
from block_sparse_long_19_b300 import workloads as W

from .parity import OUT_ATOL, OUT_RTOL

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
from block_sparse_long_19_b300 import qsa as Q
from block_sparse_long_19_b300 import workloads as W
t = W.prefill_inputs(4100, 31, "cuda")
cfg = Q.default_config(budget=512)
res = Q.prefill(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"])
d = W.decode_inputs(3, 8192, 32, "cuda", seq_lens=[8192, 5001, 2050])
kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=d["k"])
out, lse, idx, st = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], d["k"], d["v"], kblk, d["seq_lens"])
torch.cuda.synchronize()
Q.check_status(res.status); Q.check_status(st)
np.savez({path!r}, o=res.out.float().cpu().numpy(), lse=res.lse.cpu().numpy(), idx=res.idx.cpu().numpy(),
         do=out.float().cpu().numpy(), dlse=lse.cpu().numpy(), didx=idx.cpu().numpy())
"""


def _env():
    env = dict(os.environ)
    env["QSA_ATTENTION_KERNEL"] = "tc"
    return env


def test_parity_suite_with_tc_attention():
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_gpu_parity.py", "tests/test_gpu_cached.py",
                        "tests/test_gpu_fullsize.py::test_prefill_32k", "tests/test_gpu_fullsize.py::test_prefill_128k_plain"],
                       cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]


def test_tc_and_mma_kernels_agree():
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "tc.npz")
        r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT, path=path)], env=_env(),
                           capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
        tc = np.load(path)
        # this process runs the default kernel
        t = W.prefill_inputs(4100, 31, "cuda")
        cfg = Q.default_config(budget=512)
        res = Q.prefill(cfg, t["q"], t["k"], t["v"], t["qi"], t["w"], t["ki"])
        d = W.decode_inputs(3, 8192, 32, "cuda", seq_lens=[8192, 5001, 2050])
        kblk, _ = Q.kprep(cfg, d["ki"], d["k"], k_rot=d["k"])
        out, lse, idx, st = Q.sparse_attn_decode(cfg, d["q"], d["qi"], d["w"], d["k"], d["v"], kblk, d["seq_lens"])
        torch.cuda.synchronize()
        Q.check_status(res.status)
        Q.check_status(st)
        # the selection does not depend on the attention kernel
        assert np.array_equal(tc["idx"], res.idx.cpu().numpy())
        assert np.array_equal(tc["didx"], idx.cpu().numpy())
        for a, b in ((tc["o"], res.out.float().cpu().numpy()), (tc["lse"], res.lse.cpu().numpy()),
                     (tc["do"], out.float().cpu().numpy()), (tc["dlse"], lse.cpu().numpy())):
            assert np.all(np.abs(a - b) <= OUT_ATOL + OUT_RTOL * np.abs(b))
        assert not np.array_equal(tc["o"], res.out.float().cpu().numpy())
