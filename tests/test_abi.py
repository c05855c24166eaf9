"""C-ABI checks that need no GPU: the library loads, exports every symbol
that include/qsa.h declares, and rejects bad arguments synchronously with
the documented status codes (nothing is launched on those paths)."""
import ctypes
import os
import re

import pytest

from block_sparse_long_19_b300 import build as B
from block_sparse_long_19_b300 import qsa as Q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return Q.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "qsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(Q.EXPORTED) == names


def test_status_strings(lib):
    for code, name in Q.STATUS_NAMES.items():
        assert lib.qsa_status_string(code).decode() == name


def test_default_config(lib):
    cfg = Q.default_config()
    assert (cfg.block_size, cfg.budget_blocks, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
            cfg.rope_dim, cfg.n_idx_heads, cfg.idx_dim) == (4, 512, 24, 2, 256, 64, 4, 128)
    assert cfg.rope_theta == 1e7
    assert abs(cfg.softmax_scale - 1 / 16) < 1e-9


P = ctypes.c_void_p


def _pointers():
    """The pointers the rejected calls below are given.  Nothing is launched
    on these paths, but where a GPU is present they still point at a real
    device buffer (64 MiB, covering every size the calls name up to the
    ones that are rejected for size), so that a validation step that ever
    moved behind a launch could not make a kernel read a made-up address.
    Without a GPU nothing can be launched at all, and any aligned value
    serves."""
    try:
        import torch

        if torch.cuda.is_available():
            buf = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
            return buf, P(buf.data_ptr()), P(buf.data_ptr() + 8)
    except Exception:  # pragma: no cover
        pass
    return None, P(0x10000), P(0x10008)


_BUF, A, MIS = _pointers()  # A 256-byte aligned; MIS 8-byte aligned only


def call_topk(lib, cfg, L=64, qi=A, w=A, ki=A, k=None, k_rot=None, idx=A, score=None, ws=A,
              ws_bytes=1 << 40, status=A):
    return lib.qsa_index_topk(ctypes.byref(cfg), qi, w, ki, k, k_rot, L, idx, score, ws, ws_bytes,
                              status, None)


def test_index_topk_rejects(lib):
    cfg = Q.default_config()
    assert call_topk(lib, cfg, qi=None) == 1
    assert call_topk(lib, cfg, w=MIS) == 1
    assert call_topk(lib, cfg, L=0) == 1
    assert call_topk(lib, cfg, L=(1 << 24) + 1) == 2
    assert call_topk(lib, cfg, k=A, k_rot=None) == 1
    assert call_topk(lib, cfg, status=None) == 1
    assert call_topk(lib, cfg, ws_bytes=16) == 3
    assert call_topk(lib, cfg, ws=None) == 3
    bad = Q.default_config()
    bad.head_dim = 128
    assert call_topk(lib, bad) == 2
    bad = Q.default_config(budget=0)
    assert call_topk(lib, bad) == 1
    bad = Q.default_config(budget=513)
    assert call_topk(lib, bad) == 2
    bad = Q.default_config(rope_theta=-1.0)
    assert call_topk(lib, bad) == 1
    assert b"rope_theta" in lib.qsa_last_error_detail()


def test_workspace_sizes(lib):
    cfg = Q.default_config()
    assert lib.qsa_index_topk_workspace_bytes(ctypes.byref(cfg), 1 << 20) > (1 << 20) // 4 * 256
    assert lib.qsa_index_topk_workspace_bytes(ctypes.byref(cfg), 0) == 0
    assert lib.qsa_decode_workspace_bytes(ctypes.byref(cfg), 8, 1 << 20) > 0
    assert lib.qsa_decode_workspace_bytes(ctypes.byref(cfg), 8, 1 << 23) == 0


def test_prefill_attn_rejects(lib):
    cfg = Q.default_config()
    f = lib.qsa_sparse_attn_prefill
    assert f(ctypes.byref(cfg), A, A, A, A, 0, A, None, A, None) == 1
    assert f(ctypes.byref(cfg), A, A, MIS, A, 16, A, None, A, None) == 1
    assert f(ctypes.byref(cfg), A, A, A, None, 16, A, None, A, None) == 1
    assert f(None, A, A, A, A, 16, A, None, A, None) == 1


def test_decode_rejects(lib):
    cfg = Q.default_config()
    f = lib.qsa_sparse_attn_decode

    def call(batch=2, max_ctx=1024, ws_bytes=1 << 40, **kw):
        args = dict(q=A, qi=A, w=A, kc=A, vc=A, kb=A, sl=A, out=A, lse=None, idx=None, ws=A, st=A)
        args.update(kw)
        return f(ctypes.byref(cfg), batch, args["q"], args["qi"], args["w"], args["kc"], args["vc"],
                 args["kb"], max_ctx, args["sl"], args["out"], args["lse"], args["idx"], args["ws"],
                 ws_bytes, args["st"], None)

    assert call(batch=0) == 1
    assert call(max_ctx=1022) == 1
    assert call(max_ctx=1 << 23) == 2
    assert call(sl=None) == 1
    assert call(ws_bytes=64) == 3
    assert call(kb=MIS) == 1


def test_decode_noalloc_rejects(lib):
    """The decode without a workspace argument reports argument errors with
    the statuses of the decode with one, and refuses sizes whose workspace
    exceeds its built-in scratch; nothing is launched on these paths."""
    cfg = Q.default_config()
    f = lib.qsa_sparse_attn_decode_noalloc

    def call(batch=2, max_ctx=1024, cfgp=ctypes.byref(cfg), **kw):
        a = dict(q=A, qi=A, w=A, kc=A, vc=A, kb=A, sl=A, out=A, lse=None, idx=None, st=A)
        a.update(kw)
        return f(cfgp, batch, a["q"], a["qi"], a["w"], a["kc"], a["vc"], a["kb"], max_ctx, a["sl"], a["out"],
                 a["lse"], a["idx"], a["st"], None)

    assert call(batch=0) == 1
    assert call(batch=-3) == 1
    assert call(max_ctx=0) == 1
    assert call(max_ctx=3_080_192 + 4) == 2
    assert call(cfgp=None) == 1
    bad = Q.default_config()
    bad.head_dim = 128
    assert call(cfgp=ctypes.byref(bad)) == 2
    assert call(batch=256, max_ctx=1 << 20) == 2  # workspace beyond the 16 MiB scratch
    assert b"16 MiB" in lib.qsa_last_error_detail()
    assert call(max_ctx=1022) == 1
    assert call(sl=None) == 1
    assert call(kb=MIS) == 1


def test_kprep_rejects(lib):
    cfg = Q.default_config()
    f = lib.qsa_kprep
    assert f(ctypes.byref(cfg), 1, 0, 16, A, None, None, A, None) == 1
    assert f(ctypes.byref(cfg), 1, 32, 16, A, None, None, A, None) == 1
    assert f(ctypes.byref(cfg), 1, 16, 16, None, None, None, A, None) == 1
    assert f(ctypes.byref(cfg), 1, 16, 16, A, A, None, A, None) == 1
    assert f(ctypes.byref(cfg), 0, 16, 16, A, None, None, A, None) == 1


def test_cached_prefix_calls_reject(lib):
    """The cached-prefix calls validate before launching anything."""
    cfg = Q.default_config()
    kr = lib.qsa_kprep_range
    assert kr(ctypes.byref(cfg), A, None, None, A, 8, 8, None) == 1      # empty range
    assert kr(ctypes.byref(cfg), A, None, None, A, -1, 8, None) == 1     # negative start
    assert kr(ctypes.byref(cfg), None, None, None, A, 0, 8, None) == 1   # no ki
    assert kr(ctypes.byref(cfg), A, A, None, A, 0, 8, None) == 1         # k without k_rot
    assert kr(ctypes.byref(cfg), A, None, None, A, 0, (1 << 24) + 4, None) == 2
    assert lib.qsa_index_topk_cached_workspace_bytes(ctypes.byref(cfg), 0) == 0
    need = lib.qsa_index_topk_cached_workspace_bytes(ctypes.byref(cfg), 1 << 16)
    assert need > 0
    ix = lib.qsa_index_topk_cached

    def call(q_off=64, Lq=64, ws_bytes=1 << 40, **kw):
        a = dict(qi=A, w=A, kb=A, idx=A, sc=None, ws=A, st=A)
        a.update(kw)
        return ix(ctypes.byref(cfg), a["qi"], a["w"], a["kb"], q_off, Lq, a["idx"], a["sc"], a["ws"],
                  ws_bytes, a["st"], None)

    assert call(q_off=-4) == 1
    assert call(Lq=0) == 1
    assert call(q_off=1 << 24) == 2
    assert call(kb=None) == 1
    assert call(kb=MIS) == 1
    assert call(ws_bytes=16) == 3
    ixc = lib.qsa_index_topk_cached_ctas
    assert ixc(ctypes.byref(cfg), A, A, A, 64, 64, A, None, -1, A, 1 << 40, A, None) == 1  # negative grid
    assert ixc(ctypes.byref(cfg), A, A, A, 64, 0, A, None, 8, A, 1 << 40, A, None) == 1
    at = lib.qsa_sparse_attn_prefill_cached
    assert at(ctypes.byref(cfg), A, A, A, A, -1, 16, A, None, A, None) == 1
    assert at(ctypes.byref(cfg), A, A, A, A, 16, 0, A, None, A, None) == 1
    assert at(ctypes.byref(cfg), A, A, A, None, 16, 16, A, None, A, None) == 1


def test_yarn_config_checked(lib):
    cfg = Q.default_config(yarn_factor=4.0)
    cfg.yarn_beta = cfg.yarn_alpha  # empty ramp
    f = lib.qsa_sparse_attn_prefill
    assert f(ctypes.byref(cfg), A, A, A, A, 16, A, None, A, None) == 1
    cfg = Q.default_config(yarn_factor=float("nan"))
    assert f(ctypes.byref(cfg), A, A, A, A, 16, A, None, A, None) == 1
    cfg = Q.default_config(yarn_factor=4.0)
    cfg.yarn_original_max_pos = 0
    assert f(ctypes.byref(cfg), A, A, A, A, 16, A, None, A, None) == 1


def test_selftest_rejects(lib):
    assert lib.qsa_selftest_bounded_wait(1000, 0, None, None) == 1
    assert lib.qsa_selftest_bounded_wait(0, 0, A, None) == 1
    assert lib.qsa_selftest_bounded_wait(200_000_000, 0, A, None) == 1


def test_overlapped_prefill_rejects(lib):
    """The overlapped prefill validates before it creates a stream or
    launches anything."""
    cfg = Q.default_config()
    f = lib.qsa_prefill_overlapped
    need = lib.qsa_prefill_overlapped_workspace_bytes(ctypes.byref(cfg), 1 << 16)
    assert need == lib.qsa_index_topk_workspace_bytes(ctypes.byref(cfg), 1 << 16) > 0

    def call(L=1 << 16, ws_bytes=1 << 40, **kw):
        a = dict(q=A, qi=A, w=A, ki=A, k=A, kr=A, v=A, idx=A, sc=None, out=A, lse=None, ws=A, st=A)
        a.update(kw)
        return f(ctypes.byref(cfg), a["q"], a["qi"], a["w"], a["ki"], a["k"], a["kr"], a["v"], L, a["idx"],
                 a["sc"], a["out"], a["lse"], a["ws"], ws_bytes, a["st"], None)

    assert call(L=0) == 1
    assert call(L=(1 << 24) + 4) == 2
    for name in ("q", "qi", "w", "ki", "k", "kr", "v", "idx", "out", "st"):
        assert call(**{name: None}) == 1, name
    assert call(q=MIS) == 1
    assert call(ws_bytes=16) == 3
    assert call(ws=MIS) == 1


@pytest.mark.parametrize("L", [1, 1000, 16384, 70001, 262143, 262144, 266277, 1 << 20, 3_000_001, 1 << 24])
@pytest.mark.parametrize("sms", [148, 132, 8])
def test_overlap_plan_invariants(L, sms):
    """Chunks tile [0, L) in order with inner starts on 64-row tiles; the
    first indexer grid has every SM and the others leave SMs to the
    attention; long prefills are cut into several chunks."""
    cfg = Q.default_config()
    begin, ctas = Q.prefill_overlap_plan(cfg, L, sms)
    n = len(ctas)
    assert 1 <= n <= 64 and len(begin) == n + 1
    assert begin[0] == 0 and begin[-1] == L
    assert all(a < b for a, b in zip(begin[:-1], begin[1:]))
    assert all(b % 64 == 0 for b in begin[1:-1])
    assert ctas[0] == sms
    assert all(1 <= c < sms for c in ctas[1:])
    if L >= 262144:
        assert n >= 4
    else:
        assert n == 1  # short prefills: nothing to overlap
    if n > 1:
        # the first and the last chunk come in four parts on 64-row tiles
        sizes = [b - a for a, b in zip(begin[:-1], begin[1:])]
        assert n >= 10 and all(4 * s_ <= sizes[4] + 16 * 64 for s_ in sizes[:4])
        assert all(4 * s_ <= 2 * sizes[4] for s_ in sizes[-4:])
        # between them a later chunk's indexer has more past blocks per query
        # and the attention beside it the same work: never fewer SMs
        mid = ctas[5:-5]
        assert all(a <= b for a, b in zip(mid[:-1], mid[1:]))
        # no stub of a part at the end
        assert sizes[-1] >= sizes[-2] // 2


def test_overlap_plan_rejects_and_small_budget():
    cfg = Q.default_config()
    with pytest.raises(Q.QsaError):
        Q.prefill_overlap_plan(cfg, 0, 148)
    with pytest.raises(Q.QsaError):
        Q.prefill_overlap_plan(cfg, 1 << 20, 1)
    begin, ctas = Q.prefill_overlap_plan(Q.default_config(budget=1), 1 << 20, 148)
    assert begin == [0, 1 << 20] and ctas == [148]  # nothing to overlap without an indexer
    begin, ctas = Q.prefill_overlap_plan(cfg, 1 << 20, 148, max_chunks=3)
    assert len(ctas) <= 3 and begin[-1] == 1 << 20


def test_debug_library_builds_and_exports_every_symbol():
    """libqsa_debug.so (QSA_DEBUG_CHECKS=1) is the same ABI."""
    path = B.build(debug=True)
    assert path == Q.DEBUG_LIB_PATH
    dbg = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(dbg, n), n
    with Q.using_library(path) as L:
        cfg = Q.default_config()
        assert L.qsa_index_topk_workspace_bytes(ctypes.byref(cfg), 1 << 16) == \
            Q.load().qsa_index_topk_workspace_bytes(ctypes.byref(cfg), 1 << 16)
