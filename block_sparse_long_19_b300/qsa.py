"""Thin Python binding of libqsa.so (ctypes).

Argument marshalling only: torch tensors are checked for device, dtype,
shape and contiguity and passed as raw pointers together with the current
CUDA stream; every step of the computation runs in the library's kernels.
The binding never falls back to anything else: if libqsa.so is missing or a
call fails, it raises.

Function names follow the C ABI in include/qsa.h (without the qsa_ prefix).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqsa.so")
# the same kernels built with QSA_DEBUG_CHECKS=1 (python -m block_sparse_long_19_b300.build --debug)
DEBUG_LIB_PATH = os.path.join(_HERE, "libqsa_debug.so")

QSA_OK = 0
QSA_ERR_TIMEOUT = 5
STATUS_NAMES = {
    0: "QSA_OK", 1: "QSA_ERR_INVALID_ARG", 2: "QSA_ERR_UNSUPPORTED", 3: "QSA_ERR_WORKSPACE",
    4: "QSA_ERR_CUDA", 5: "QSA_ERR_TIMEOUT", 6: "QSA_ERR_DEVICE_CHECK",
}

# Every function the header declares.
EXPORTED = [
    "qsa_default_config", "qsa_status_string", "qsa_last_error_detail", "qsa_kprep",
    "qsa_index_topk_workspace_bytes", "qsa_index_topk", "qsa_index_scores",
    "qsa_sparse_attn_prefill", "qsa_decode_workspace_bytes", "qsa_sparse_attn_decode",
    "qsa_sparse_attn_decode_noalloc", "qsa_kprep_range", "qsa_index_topk_cached_workspace_bytes",
    "qsa_index_topk_cached", "qsa_sparse_attn_prefill_cached", "qsa_index_topk_tokens_workspace_bytes",
    "qsa_index_topk_tokens", "qsa_selftest_bounded_wait", "qsa_prefill_overlapped_workspace_bytes",
    "qsa_prefill_overlapped", "qsa_prefill_overlap_plan", "qsa_index_topk_cached_ctas",
]


class QsaError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({detail})")


class Config(ctypes.Structure):
    _fields_ = [
        ("block_size", ctypes.c_int), ("budget_blocks", ctypes.c_int),
        ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("rope_dim", ctypes.c_int), ("n_idx_heads", ctypes.c_int), ("idx_dim", ctypes.c_int),
        ("rope_theta", ctypes.c_double), ("softmax_scale", ctypes.c_float),
        ("yarn_factor", ctypes.c_float), ("yarn_original_max_pos", ctypes.c_int),
        ("yarn_alpha", ctypes.c_float), ("yarn_beta", ctypes.c_float),
    ]


_lib = None


def load(path: str = LIB_PATH):
    """Load libqsa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = _open(path)
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Route every call of this module to another build of the library (e.g.
    DEBUG_LIB_PATH) inside the `with` block."""
    global _lib
    saved = _lib
    _lib = _open(path)
    try:
        yield _lib
    finally:
        _lib = saved


def _open(path: str):
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m block_sparse_long_19_b300.build` "
            "(there is no fallback implementation)")
    L = ctypes.CDLL(path)
    c = ctypes
    P = c.c_void_p
    cfgp = c.POINTER(Config)
    L.qsa_default_config.argtypes = [cfgp]
    L.qsa_default_config.restype = None
    L.qsa_status_string.argtypes = [c.c_int]
    L.qsa_status_string.restype = c.c_char_p
    L.qsa_last_error_detail.argtypes = []
    L.qsa_last_error_detail.restype = c.c_char_p
    L.qsa_kprep.argtypes = [cfgp, c.c_int, c.c_int64, c.c_int64, P, P, P, P, P]
    L.qsa_kprep.restype = c.c_int
    L.qsa_index_topk_workspace_bytes.argtypes = [cfgp, c.c_int64]
    L.qsa_index_topk_workspace_bytes.restype = c.c_size_t
    L.qsa_index_topk.argtypes = [cfgp, P, P, P, P, P, c.c_int64, P, P, P, c.c_size_t, P, P]
    L.qsa_index_topk.restype = c.c_int
    L.qsa_index_scores.argtypes = [cfgp, P, P, P, c.c_int64, P, P, c.c_size_t, P, P]
    L.qsa_index_scores.restype = c.c_int
    L.qsa_sparse_attn_prefill.argtypes = [cfgp, P, P, P, P, c.c_int64, P, P, P, P]
    L.qsa_sparse_attn_prefill.restype = c.c_int
    L.qsa_decode_workspace_bytes.argtypes = [cfgp, c.c_int, c.c_int64]
    L.qsa_decode_workspace_bytes.restype = c.c_size_t
    L.qsa_sparse_attn_decode.argtypes = [cfgp, c.c_int, P, P, P, P, P, P, c.c_int64, P, P, P, P,
                                         P, c.c_size_t, P, P]
    L.qsa_sparse_attn_decode.restype = c.c_int
    L.qsa_sparse_attn_decode_noalloc.argtypes = [cfgp, c.c_int, P, P, P, P, P, P, c.c_int64, P, P,
                                                 P, P, P, P]
    L.qsa_sparse_attn_decode_noalloc.restype = c.c_int
    L.qsa_kprep_range.argtypes = [cfgp, P, P, P, P, c.c_int64, c.c_int64, P]
    L.qsa_kprep_range.restype = c.c_int
    L.qsa_index_topk_cached_workspace_bytes.argtypes = [cfgp, c.c_int64]
    L.qsa_index_topk_cached_workspace_bytes.restype = c.c_size_t
    L.qsa_index_topk_cached.argtypes = [cfgp, P, P, P, c.c_int64, c.c_int64, P, P, P, c.c_size_t, P, P]
    L.qsa_index_topk_cached.restype = c.c_int
    L.qsa_index_topk_cached_ctas.argtypes = [cfgp, P, P, P, c.c_int64, c.c_int64, P, P, c.c_int, P, c.c_size_t,
                                             P, P]
    L.qsa_index_topk_cached_ctas.restype = c.c_int
    L.qsa_sparse_attn_prefill_cached.argtypes = [cfgp, P, P, P, P, c.c_int64, c.c_int64, P, P, P, P]
    L.qsa_sparse_attn_prefill_cached.restype = c.c_int
    L.qsa_index_topk_tokens_workspace_bytes.argtypes = [cfgp, c.c_int64]
    L.qsa_index_topk_tokens_workspace_bytes.restype = c.c_size_t
    L.qsa_index_topk_tokens.argtypes = [cfgp, P, P, P, c.c_int64, P, P, P, c.c_size_t, P, P]
    L.qsa_index_topk_tokens.restype = c.c_int
    L.qsa_selftest_bounded_wait.argtypes = [c.c_int64, c.c_int, P, P]
    L.qsa_selftest_bounded_wait.restype = c.c_int
    L.qsa_prefill_overlapped_workspace_bytes.argtypes = [cfgp, c.c_int64]
    L.qsa_prefill_overlapped_workspace_bytes.restype = c.c_size_t
    L.qsa_prefill_overlapped.argtypes = [cfgp, P, P, P, P, P, P, P, c.c_int64, P, P, P, P, P, c.c_size_t, P, P]
    L.qsa_prefill_overlapped.restype = c.c_int
    L.qsa_prefill_overlap_plan.argtypes = [cfgp, c.c_int64, c.c_int, c.c_int, c.POINTER(c.c_int64),
                                           c.POINTER(c.c_int)]
    L.qsa_prefill_overlap_plan.restype = c.c_int
    return L


def default_config(budget: int = 512, rope_theta: float = 1.0e7, softmax_scale: float = 1.0 / 16,
                   yarn_factor: float = 1.0) -> Config:
    """The model card's configuration; yarn_factor > 1 turns YaRN on (the card
    uses 4 over an original context of 262,144)."""
    cfg = Config()
    load().qsa_default_config(ctypes.byref(cfg))
    cfg.budget_blocks = budget
    cfg.rope_theta = rope_theta
    cfg.softmax_scale = softmax_scale
    cfg.yarn_factor = yarn_factor
    return cfg


def _check(code: int, where: str):
    if code != QSA_OK:
        detail = load().qsa_last_error_detail().decode()
        raise QsaError(code, where, detail)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, shape=None, cuda: bool = True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_status(status: torch.Tensor, where: str = "device"):
    """Synchronise and raise if a kernel reported a problem."""
    v = int(status.item())
    if v != 0:
        raise QsaError(v, where, "reported by a kernel")


# --------------------------------------------------------------- entries --

def kprep(cfg: Config, ki, k=None, k_rot=None, kblk=None, L: int | None = None, stream=None):
    """Block keys (and RoPE'd keys) for caches [B, max_ctx, ...] or a single
    sequence [L, ...].  Returns kblk."""
    batched = ki.dim() == 3
    B = ki.shape[0] if batched else 1
    max_ctx = ki.shape[1] if batched else ki.shape[0]
    L = max_ctx if L is None else L
    _need(ki, "ki", torch.bfloat16, (B, max_ctx, 128) if batched else (max_ctx, 128))
    if kblk is None:
        shape = (B, max_ctx // 4, 128) if batched else (max_ctx // 4, 128)
        kblk = torch.empty(shape, dtype=torch.bfloat16, device=ki.device)
    if k is not None:
        _need(k, "k", torch.bfloat16, (B, max_ctx, 2, 256) if batched else (max_ctx, 2, 256))
        if k_rot is None:
            k_rot = torch.empty_like(k)
        _need(k_rot, "k_rot", torch.bfloat16, k.shape)
    _check(load().qsa_kprep(ctypes.byref(cfg), B, L, max_ctx, _ptr(ki), _ptr(k), _ptr(k_rot),
                            _ptr(kblk), _stream(stream)), "qsa_kprep")
    return kblk, k_rot


def index_topk_workspace_bytes(cfg: Config, L: int) -> int:
    return int(load().qsa_index_topk_workspace_bytes(ctypes.byref(cfg), L))


def index_topk(cfg: Config, qi, w, ki, k=None, k_rot=None, idx=None, score=None, ws=None,
               status=None, want_score: bool = True, stream=None):
    """Prefill indexer + selection.  Returns (idx, score, k_rot, status)."""
    L = qi.shape[0]
    dev = qi.device
    _need(qi, "qi", torch.bfloat16, (L, 4, 128))
    _need(w, "w", torch.bfloat16, (L, 4))
    _need(ki, "ki", torch.bfloat16, (L, 128))
    if k is not None:
        _need(k, "k", torch.bfloat16, (L, 2, 256))
        if k_rot is None:
            k_rot = torch.empty_like(k)
    B = cfg.budget_blocks
    if idx is None:
        idx = torch.empty((L, B), dtype=torch.int32, device=dev)
    if score is None and want_score:
        score = torch.empty((L, B), dtype=torch.float32, device=dev)
    need = index_topk_workspace_bytes(cfg, L)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if status is None:
        status = new_status(dev)
    _check(load().qsa_index_topk(ctypes.byref(cfg), _ptr(qi), _ptr(w), _ptr(ki), _ptr(k), _ptr(k_rot),
                                 L, _ptr(idx), _ptr(score), _ptr(ws), ws.numel(), _ptr(status),
                                 _stream(stream)), "qsa_index_topk")
    return idx, score, k_rot, status


def index_scores(cfg: Config, qi, w, ki, scores=None, ws=None, status=None, stream=None):
    """Dense block-score matrix [L, L/4] (NaN where b >= floor(t/4))."""
    L = qi.shape[0]
    dev = qi.device
    _need(qi, "qi", torch.bfloat16, (L, 4, 128))
    _need(w, "w", torch.bfloat16, (L, 4))
    _need(ki, "ki", torch.bfloat16, (L, 128))
    if scores is None:
        scores = torch.full((L, L // 4), float("nan"), dtype=torch.float32, device=dev)
    need = index_topk_workspace_bytes(cfg, L)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if status is None:
        status = new_status(dev)
    _check(load().qsa_index_scores(ctypes.byref(cfg), _ptr(qi), _ptr(w), _ptr(ki), L, _ptr(scores),
                                   _ptr(ws), ws.numel(), _ptr(status), _stream(stream)),
           "qsa_index_scores")
    return scores, status


def sparse_attn_prefill(cfg: Config, q, k_rot, v, idx, out=None, lse=None, status=None,
                        want_lse: bool = True, stream=None):
    L = q.shape[0]
    dev = q.device
    _need(q, "q", torch.bfloat16, (L, 24, 256))
    _need(k_rot, "k_rot", torch.bfloat16, (L, 2, 256))
    _need(v, "v", torch.bfloat16, (L, 2, 256))
    _need(idx, "idx", torch.int32, (L, cfg.budget_blocks))
    if out is None:
        out = torch.empty((L, 24, 256), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((L, 24), dtype=torch.float32, device=dev)
    if status is None:
        status = new_status(dev)
    _check(load().qsa_sparse_attn_prefill(ctypes.byref(cfg), _ptr(q), _ptr(k_rot), _ptr(v), _ptr(idx),
                                          L, _ptr(out), _ptr(lse), _ptr(status), _stream(stream)),
           "qsa_sparse_attn_prefill")
    return out, lse, status


def kprep_range(cfg: Config, ki, kblk, t_begin: int, t_end: int, k=None, k_rot=None, stream=None):
    """Block keys of blocks t_begin//4 .. t_end//4-1 into kblk and RoPE'd key
    rows t_begin .. t_end-1 (a new chunk after a cached prefix)."""
    _need(ki, "ki", torch.bfloat16)
    _need(kblk, "kblk", torch.bfloat16)
    if ki.shape[0] < t_end or kblk.shape[0] < t_end // 4:
        raise ValueError("ki must hold t_end rows and kblk t_end // 4 rows")
    if (k is None) != (k_rot is None):
        raise ValueError("k and k_rot must both be given or both be None")
    _check(load().qsa_kprep_range(ctypes.byref(cfg), _ptr(ki), _ptr(k), _ptr(k_rot), _ptr(kblk), t_begin,
                                  t_end, _stream(stream)), "qsa_kprep_range")


def index_topk_cached(cfg: Config, qi, w, kblk, q_offset: int, idx=None, score=None, ws=None, status=None,
                      want_score: bool = True, stream=None, max_ctas: int = 0):
    """Indexer + selection for the query rows q_offset .. q_offset+Lq-1 of a
    sequence whose block keys so far are kblk.  max_ctas > 0 limits the
    persistent grid to that many SMs.  Returns (idx, score, status)."""
    Lq = qi.shape[0]
    dev = qi.device
    _need(qi, "qi", torch.bfloat16, (Lq, 4, 128))
    _need(w, "w", torch.bfloat16, (Lq, 4))
    _need(kblk, "kblk", torch.bfloat16)
    if kblk.shape[0] < (q_offset + Lq) // 4:
        raise ValueError("kblk must hold (q_offset + Lq) // 4 block keys")
    B = cfg.budget_blocks
    if idx is None:
        idx = torch.empty((Lq, B), dtype=torch.int32, device=dev)
    if score is None and want_score:
        score = torch.empty((Lq, B), dtype=torch.float32, device=dev)
    need = load().qsa_index_topk_cached_workspace_bytes(ctypes.byref(cfg), Lq)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if status is None:
        status = new_status(dev)
    _check(load().qsa_index_topk_cached_ctas(ctypes.byref(cfg), _ptr(qi), _ptr(w), _ptr(kblk), q_offset, Lq,
                                             _ptr(idx), _ptr(score), max_ctas, _ptr(ws), ws.numel(), _ptr(status),
                                             _stream(stream)), "qsa_index_topk_cached_ctas")
    return idx, score, status


def sparse_attn_prefill_cached(cfg: Config, q, k_rot, v, idx, q_offset: int, out=None, lse=None, status=None,
                               want_lse: bool = True, stream=None):
    """Attention for the query rows q_offset .. q_offset+Lq-1 over the whole
    prefix k_rot / v [q_offset+Lq, 2, 256]."""
    Lq = q.shape[0]
    dev = q.device
    _need(q, "q", torch.bfloat16, (Lq, 24, 256))
    _need(k_rot, "k_rot", torch.bfloat16, (q_offset + Lq, 2, 256))
    _need(v, "v", torch.bfloat16, (q_offset + Lq, 2, 256))
    _need(idx, "idx", torch.int32, (Lq, cfg.budget_blocks))
    if out is None:
        out = torch.empty((Lq, 24, 256), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((Lq, 24), dtype=torch.float32, device=dev)
    if status is None:
        status = new_status(dev)
    _check(load().qsa_sparse_attn_prefill_cached(ctypes.byref(cfg), _ptr(q), _ptr(k_rot), _ptr(v), _ptr(idx),
                                                 q_offset, Lq, _ptr(out), _ptr(lse), _ptr(status),
                                                 _stream(stream)), "qsa_sparse_attn_prefill_cached")
    return out, lse, status


def index_topk_tokens(cfg: Config, qi, w, ki, idx=None, score=None, ws=None, status=None,
                      want_score: bool = True, stream=None):
    """Token-level indexer (one token per selection unit; cfg.budget_blocks
    counts tokens).  Returns (idx, score, status)."""
    L = qi.shape[0]
    dev = qi.device
    _need(qi, "qi", torch.bfloat16, (L, 4, 128))
    _need(w, "w", torch.bfloat16, (L, 4))
    _need(ki, "ki", torch.bfloat16, (L, 128))
    B = cfg.budget_blocks
    if idx is None:
        idx = torch.empty((L, B), dtype=torch.int32, device=dev)
    if score is None and want_score:
        score = torch.empty((L, B), dtype=torch.float32, device=dev)
    need = load().qsa_index_topk_tokens_workspace_bytes(ctypes.byref(cfg), L)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if status is None:
        status = new_status(dev)
    _check(load().qsa_index_topk_tokens(ctypes.byref(cfg), _ptr(qi), _ptr(w), _ptr(ki), L, _ptr(idx), _ptr(score),
                                        _ptr(ws), ws.numel(), _ptr(status), _stream(stream)),
           "qsa_index_topk_tokens")
    return idx, score, status


def selftest_bounded_wait(limit_ns: int, complete: bool, status=None, stream=None):
    """Run the bounded-wait self-test kernel; returns the status tensor (its
    value is QSA_ERR_TIMEOUT after the wait ran out)."""
    if status is None:
        status = new_status("cuda")
    _check(load().qsa_selftest_bounded_wait(int(limit_ns), 1 if complete else 0, _ptr(status), _stream(stream)),
           "qsa_selftest_bounded_wait")
    return status


def decode_workspace_bytes(cfg: Config, batch: int, max_ctx: int) -> int:
    return int(load().qsa_decode_workspace_bytes(ctypes.byref(cfg), batch, max_ctx))


def sparse_attn_decode(cfg: Config, q, qi, w, k_cache, v_cache, kblk_cache, seq_lens, out=None,
                       lse=None, idx_out=None, ws=None, status=None, want_idx: bool = True,
                       want_lse: bool = True, stream=None):
    B, Tmax = k_cache.shape[0], k_cache.shape[1]
    dev = q.device
    _need(q, "q", torch.bfloat16, (B, 24, 256))
    _need(qi, "qi", torch.bfloat16, (B, 4, 128))
    _need(w, "w", torch.bfloat16, (B, 4))
    _need(k_cache, "k_cache", torch.bfloat16, (B, Tmax, 2, 256))
    _need(v_cache, "v_cache", torch.bfloat16, (B, Tmax, 2, 256))
    _need(kblk_cache, "kblk_cache", torch.bfloat16, (B, Tmax // 4, 128))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, 24, 256), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, 24), dtype=torch.float32, device=dev)
    if idx_out is None and want_idx:
        idx_out = torch.empty((B, cfg.budget_blocks), dtype=torch.int32, device=dev)
    need = decode_workspace_bytes(cfg, B, Tmax)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if status is None:
        status = new_status(dev)
    _check(load().qsa_sparse_attn_decode(
        ctypes.byref(cfg), B, _ptr(q), _ptr(qi), _ptr(w), _ptr(k_cache), _ptr(v_cache),
        _ptr(kblk_cache), Tmax, _ptr(seq_lens), _ptr(out), _ptr(lse), _ptr(idx_out), _ptr(ws),
        ws.numel(), _ptr(status), _stream(stream)), "qsa_sparse_attn_decode")
    return out, lse, idx_out, status


def sparse_attn_decode_noalloc(cfg: Config, q, qi, w, k_cache, v_cache, kblk_cache, seq_lens,
                               out=None, lse=None, idx_out=None, status=None, want_idx: bool = True,
                               want_lse: bool = True, stream=None):
    """Decode through qsa_sparse_attn_decode_noalloc: no workspace argument,
    the library's built-in 16 MiB device scratch is used instead (for callers
    that cannot allocate device memory; see include/qsa.h)."""
    B, Tmax = k_cache.shape[0], k_cache.shape[1]
    dev = q.device
    _need(q, "q", torch.bfloat16, (B, 24, 256))
    _need(qi, "qi", torch.bfloat16, (B, 4, 128))
    _need(w, "w", torch.bfloat16, (B, 4))
    _need(k_cache, "k_cache", torch.bfloat16, (B, Tmax, 2, 256))
    _need(v_cache, "v_cache", torch.bfloat16, (B, Tmax, 2, 256))
    _need(kblk_cache, "kblk_cache", torch.bfloat16, (B, Tmax // 4, 128))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, 24, 256), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, 24), dtype=torch.float32, device=dev)
    if idx_out is None and want_idx:
        idx_out = torch.empty((B, cfg.budget_blocks), dtype=torch.int32, device=dev)
    if status is None:
        status = new_status(dev)
    _check(load().qsa_sparse_attn_decode_noalloc(
        ctypes.byref(cfg), B, _ptr(q), _ptr(qi), _ptr(w), _ptr(k_cache), _ptr(v_cache),
        _ptr(kblk_cache), Tmax, _ptr(seq_lens), _ptr(out), _ptr(lse), _ptr(idx_out), _ptr(status),
        _stream(stream)), "qsa_sparse_attn_decode_noalloc")
    return out, lse, idx_out, status


@dataclass
class PrefillResult:
    idx: torch.Tensor
    score: torch.Tensor | None
    k_rot: torch.Tensor
    out: torch.Tensor
    lse: torch.Tensor | None
    status: torch.Tensor


def prefill(cfg: Config, q, k, v, qi, w, ki, want_score: bool = False, want_lse: bool = True,
            ws=None, stream=None) -> PrefillResult:
    """The whole QSA prefill layer: indexer + selection, then sparse attention."""
    idx, score, k_rot, status = index_topk(cfg, qi, w, ki, k=k, want_score=want_score, ws=ws,
                                           stream=stream)
    out, lse, _ = sparse_attn_prefill(cfg, q, k_rot, v, idx, status=status, want_lse=want_lse,
                                      stream=stream)
    return PrefillResult(idx, score, k_rot, out, lse, status)


def prefill_overlapped_workspace_bytes(cfg: Config, L: int) -> int:
    return int(load().qsa_prefill_overlapped_workspace_bytes(ctypes.byref(cfg), L))


def prefill_overlap_plan(cfg: Config, L: int, sms: int, max_chunks: int = 64):
    """Chunk starts (n+1 values, the last = L) and indexer grid sizes (n
    values) that prefill_overlapped uses on a GPU with `sms` SMs."""
    begin = (ctypes.c_int64 * (max_chunks + 1))()
    ctas = (ctypes.c_int * max_chunks)()
    n = load().qsa_prefill_overlap_plan(ctypes.byref(cfg), L, sms, max_chunks, begin, ctas)
    if n < 1:
        raise QsaError(1, "qsa_prefill_overlap_plan: invalid arguments")
    return [int(begin[i]) for i in range(n + 1)], [int(ctas[i]) for i in range(n)]


def prefill_overlapped(cfg: Config, q, k, v, qi, w, ki, k_rot=None, idx=None, score=None, out=None, lse=None,
                       ws=None, status=None, want_score: bool = False, want_lse: bool = True,
                       stream=None) -> PrefillResult:
    """The whole prefill layer with the indexer of one chunk of query rows
    running beside the attention of the previous chunk (same results as
    prefill())."""
    L = q.shape[0]
    dev = q.device
    _need(q, "q", torch.bfloat16, (L, 24, 256))
    _need(k, "k", torch.bfloat16, (L, 2, 256))
    _need(v, "v", torch.bfloat16, (L, 2, 256))
    _need(qi, "qi", torch.bfloat16, (L, 4, 128))
    _need(w, "w", torch.bfloat16, (L, 4))
    _need(ki, "ki", torch.bfloat16, (L, 128))
    B = cfg.budget_blocks
    if k_rot is None:
        k_rot = torch.empty_like(k)
    if idx is None:
        idx = torch.empty((L, B), dtype=torch.int32, device=dev)
    if score is None and want_score:
        score = torch.empty((L, B), dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty((L, 24, 256), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((L, 24), dtype=torch.float32, device=dev)
    need = prefill_overlapped_workspace_bytes(cfg, L)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if status is None:
        status = new_status(dev)
    _check(load().qsa_prefill_overlapped(ctypes.byref(cfg), _ptr(q), _ptr(qi), _ptr(w), _ptr(ki), _ptr(k),
                                         _ptr(k_rot), _ptr(v), L, _ptr(idx), _ptr(score), _ptr(out), _ptr(lse),
                                         _ptr(ws), ws.numel(), _ptr(status), _stream(stream)),
           "qsa_prefill_overlapped")
    return PrefillResult(idx, score, k_rot, out, lse, status)


class HostPrefill:
    """Prefill of one sequence whose inputs live in pinned host memory.

    The sequence is processed in chunks of query rows with the cached-prefix
    calls (each chunk's rows against every earlier token), so the host->device
    copies of chunk c+1 and the device->host copy of chunk c-1's output run on
    their own streams while chunk c computes.  For long prefills the chunks
    and indexer grid sizes are those of prefill_overlapped() (whose first and
    last chunk come in four parts, a short pipeline fill and drain): the
    indexer of a chunk runs on a higher-priority stream on a share of the SMs
    while the attention of the previous chunk runs on the rest, and each
    chunk's K-prep on a third stream once its inputs are in (the plan's
    starting split is used throughout; prefill_overlapped() also adapts it).
    The results equal those of prefill() on the whole sequence (the
    per-query computation does not depend on the chunking).  Device buffers
    are allocated once, here."""

    NAMES = ("q", "k", "v", "qi", "w", "ki")

    def __init__(self, cfg: Config, L: int, chunk_tokens: int = 65536, device="cuda"):
        self.cfg, self.L, self.dev = cfg, L, device
        self.chunk = max(64, (chunk_tokens // 64) * 64)
        shapes = {"q": (L, 24, 256), "k": (L, 2, 256), "v": (L, 2, 256), "qi": (L, 4, 128), "w": (L, 4),
                  "ki": (L, 128)}
        self.dev_in = {n: torch.empty(shapes[n], dtype=torch.bfloat16, device=device) for n in self.NAMES}
        self.k_rot = torch.empty((L, 2, 256), dtype=torch.bfloat16, device=device)
        self.kblk = torch.zeros((max(L // 4, 1), 128), dtype=torch.bfloat16, device=device)
        self.idx = torch.empty((L, cfg.budget_blocks), dtype=torch.int32, device=device)
        self.out = torch.empty((L, 24, 256), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((L, 24), dtype=torch.float32, device=device)
        self.status = new_status(device)
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        begin, ctas = prefill_overlap_plan(cfg, L, sms)
        if len(ctas) > 1:
            self.bounds, self.ctas = list(begin), list(ctas)
        else:
            self.bounds = list(range(0, L, self.chunk)) + [L]
            self.ctas = None
        longest = max(b - a for a, b in zip(self.bounds[:-1], self.bounds[1:]))
        need = load().qsa_index_topk_cached_workspace_bytes(ctypes.byref(cfg), longest)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        self.h2d = torch.cuda.Stream(device=device)
        self.d2h = torch.cuda.Stream(device=device)
        self.side = torch.cuda.Stream(device=device, priority=-8) if self.ctas else None
        self.kps = torch.cuda.Stream(device=device, priority=-8) if self.ctas else None  # K-prep

    def run(self, host: dict, out_host: torch.Tensor, lse_host: torch.Tensor | None = None):
        """host: pinned CPU tensors q, k, v, qi, w, ki of the whole sequence;
        out_host [L, 24, 256] (and lse_host [L, 24]) receive the outputs.
        Enqueues everything; the caller's current stream waits for the last
        copy back."""
        cfg, comp = self.cfg, torch.cuda.current_stream(self.dev)
        ixs = self.side if self.ctas else comp  # stream of K-prep + indexer
        start = torch.cuda.Event()
        start.record(comp)
        for st in (self.h2d, self.d2h) + ((self.side, self.kps) if self.side else ()):
            st.wait_event(start)
        chunks = list(zip(self.bounds[:-1], self.bounds[1:]))
        ins = []
        for a, b in chunks:
            ev = torch.cuda.Event()
            with torch.cuda.stream(self.h2d):
                for n in self.NAMES:
                    self.dev_in[n][a:b].copy_(host[n][a:b], non_blocking=True)
                ev.record(self.h2d)
            ins.append(ev)
        d = self.dev_in
        # With the indexer on its own stream, each chunk's K-prep runs on a
        # third stream as soon as the chunk's inputs are in, so the indexer
        # stream goes from one indexer chunk straight to the next: a K-prep
        # between them would let the attention's CTAs take the SMs freed by
        # the indexer before the next indexer chunk is launched (1M: 706 vs
        # 708 ms end to end).
        kp_done = []
        if self.ctas:
            for (a, b), ev in zip(chunks, ins):
                self.kps.wait_event(ev)
                kprep_range(cfg, d["ki"][:b], self.kblk, a, b, k=d["k"][:b], k_rot=self.k_rot[:b], stream=self.kps)
                e_kp = torch.cuda.Event()
                e_kp.record(self.kps)
                kp_done.append(e_kp)
        for j, ((a, b), ev) in enumerate(zip(chunks, ins)):
            if kp_done:
                ixs.wait_event(kp_done[j])
            else:
                ixs.wait_event(ev)
                kprep_range(cfg, d["ki"][:b], self.kblk, a, b, k=d["k"][:b], k_rot=self.k_rot[:b], stream=ixs)
            index_topk_cached(cfg, d["qi"][a:b], d["w"][a:b], self.kblk[: max(b // 4, 1)], a, idx=self.idx[a:b],
                              score=None, ws=self.ws, status=self.status, want_score=False, stream=ixs,
                              max_ctas=self.ctas[j] if self.ctas else 0)
            if self.ctas:
                sel = torch.cuda.Event()
                sel.record(ixs)
                comp.wait_event(sel)
            sparse_attn_prefill_cached(cfg, d["q"][a:b], self.k_rot[:b], d["v"][:b], self.idx[a:b], a,
                                       out=self.out[a:b], lse=self.lse[a:b], status=self.status, stream=comp)
            done = torch.cuda.Event()
            done.record(comp)
            self.d2h.wait_event(done)
            with torch.cuda.stream(self.d2h):
                out_host[a:b].copy_(self.out[a:b], non_blocking=True)
                if lse_host is not None:
                    lse_host[a:b].copy_(self.lse[a:b], non_blocking=True)
        comp.wait_stream(self.d2h)
        return self.status
