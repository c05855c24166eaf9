"""ctypes wrapper of the C oracle (``qsa_oracle.c``) -- test infrastructure only.

Arrays are numpy; bf16 tensors travel as ``np.uint16`` bit patterns.  The
library is compiled with gcc on first use if it is missing or older than its
source (``build_oracle`` does it explicitly).

Sources: Qwen3.8-Flash-Next launch post, "Model Architecture / Attention:
GDN + QSA"; Qwen3.8-Flash-Next model card, "Model Overview / Qwen Sparse
Attention" and "Processing Ultra-Long Texts" (rope_parameters).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

__all__ = [
    "BS", "HQ", "HKV", "D", "RD", "HI", "DI", "THETA", "SCALE", "YARN_CARD",
    "rope_inv_freq", "yarn_logit_factor",
    "build_oracle", "lib", "max_threads",
    "bf16_bits_to_f64", "f64_to_bf16_bits", "block_keys", "rope_exact",
    "rope_row_bf16", "rope_keys", "block_scores", "select", "attend",
    "prefill_rows", "prefill_scores", "decode",
]

# Shapes and constants restated from the model card (the CUDA side has its own).
BS = 4          # tokens per micro-block: 512 blocks <-> 2048 tokens
HQ, HKV, D = 24, 2, 256
RD = 64         # rotary dims = 0.25 * 256
HI, DI = 4, 128
THETA = 1.0e7
SCALE = 1.0 / 16.0   # 1/sqrt(256)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_LIB = os.path.join(_HERE, "libqsa_oracle.so")
_lock = threading.Lock()
_lib = None

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build_oracle(force: bool = False) -> str:
    """Compile ``libqsa_oracle.so`` (gcc, -O2, OpenMP).  Returns its path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _opt(ptr_type):
    """ndpointer that also accepts None (NULL)."""

    def from_param(obj):
        if obj is None:
            return None
        return ptr_type.from_param(obj)

    return type("Opt" + ptr_type.__name__, (), {"from_param": staticmethod(from_param)})


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build_oracle())
            c = ctypes
            L.qo_bf16_to_f64.argtypes = [c.c_uint16]
            L.qo_bf16_to_f64.restype = c.c_double
            L.qo_f64_to_bf16.argtypes = [c.c_double]
            L.qo_f64_to_bf16.restype = c.c_uint16
            L.qo_block_keys.argtypes = [c.c_int64, _u16p, _u16p]
            L.qo_rope_inv_freq.argtypes = [c.c_double, c.c_double, c.c_double, c.c_double, c.c_double, _f64p]
            L.qo_yarn_logit_factor.argtypes = [c.c_double]
            L.qo_yarn_logit_factor.restype = c.c_double
            L.qo_rope_exact.argtypes = [_u16p, _f64p, c.c_int64, _f64p]
            L.qo_rope_row_bf16.argtypes = [_u16p, _f64p, c.c_int64, _u16p]
            L.qo_rope_keys.argtypes = [c.c_int64, _f64p, _u16p, _u16p]
            L.qo_block_scores.argtypes = [_u16p, _u16p, _u16p, c.c_int64, _f64p]
            L.qo_select.argtypes = [_f64p, c.c_int64, c.c_int, _i32p, _opt(_f64p)]
            L.qo_select.restype = c.c_int
            L.qo_attend.argtypes = [_u16p, c.c_int64, _u16p, _u16p, _i32p, c.c_int,
                                    _f64p, c.c_double, _f64p, _f64p]
            L.qo_prefill_rows.argtypes = [
                c.c_int64, c.c_int, _f64p, c.c_double,
                _u16p, _u16p, _u16p, _u16p, _u16p, _u16p,
                _i64p, c.c_int64, _opt(_i32p),
                _opt(_i32p), _opt(_f64p), _opt(_f64p), _opt(_f64p), c.c_int]
            L.qo_prefill_scores.argtypes = [c.c_int64, _u16p, _u16p, _u16p, _i64p, c.c_int64,
                                            _f64p, c.c_int]
            L.qo_decode.argtypes = [
                c.c_int, c.c_int64, _i64p, c.c_int, _f64p, c.c_double,
                _u16p, _u16p, _u16p, _u16p, _u16p, _u16p, _opt(_i32p),
                _opt(_i32p), _opt(_f64p), _opt(_f64p), _opt(_f64p), c.c_int]
            L.qo_max_threads.restype = c.c_int
            _lib = L
    return _lib


def max_threads() -> int:
    return int(lib().qo_max_threads())


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return np.ascontiguousarray(a)


# ------------------------------------------------------------------ pieces --

def bf16_bits_to_f64(bits) -> np.ndarray:
    L = lib()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([L.qo_bf16_to_f64(int(x)) for x in b], dtype=np.float64).reshape(np.shape(bits))


def f64_to_bf16_bits(x) -> np.ndarray:
    L = lib()
    a = np.asarray(x, dtype=np.float64).ravel()
    return np.array([L.qo_f64_to_bf16(float(v)) for v in a], dtype=np.uint16).reshape(np.shape(x))


def block_keys(ki) -> np.ndarray:
    """kblk [L//4, 128] (bf16 bits) from indexer keys ki [L, 128]."""
    ki = _u16(ki)
    L = ki.shape[0]
    out = np.zeros((L // BS, DI), dtype=np.uint16)
    if L // BS:
        lib().qo_block_keys(L, ki, out)
    return out


# YaRN settings (factor s, original context, ramp alpha, ramp beta) or None:
# the model card's "Processing Ultra-Long Texts" enables factor 4 over
# 262,144 positions; alpha = 1, beta = 32 are the published method's values.
YARN_CARD = (4.0, 262144.0, 1.0, 32.0)


def rope_inv_freq(theta: float = THETA, yarn=None) -> np.ndarray:
    """The 32 rotary frequencies (fp64), YaRN-rescaled when yarn is given."""
    s, l_orig, alpha, beta = yarn if yarn is not None else (1.0, 1.0, 1.0, 32.0)
    out = np.zeros(RD // 2, dtype=np.float64)
    lib().qo_rope_inv_freq(float(theta), float(s), float(l_orig), float(alpha), float(beta), out)
    return out


def yarn_logit_factor(s: float) -> float:
    """YaRN's attention temperature 1/t = (0.1 ln s + 1)^2 (1 for s <= 1)."""
    return float(lib().qo_yarn_logit_factor(float(s)))


def _attn_scale(scale: float, yarn) -> float:
    return scale * (yarn_logit_factor(yarn[0]) if yarn is not None else 1.0)


def rope_exact(x, pos: int, theta: float = THETA, yarn=None) -> np.ndarray:
    """The 64 rotated dims of one head row, fp64, before rounding."""
    x = _u16(x)
    out = np.zeros(RD, dtype=np.float64)
    lib().qo_rope_exact(x, rope_inv_freq(theta, yarn), int(pos), out)
    return out


def rope_row_bf16(x, pos: int, theta: float = THETA, yarn=None) -> np.ndarray:
    x = _u16(x)
    out = np.zeros(D, dtype=np.uint16)
    lib().qo_rope_row_bf16(x, rope_inv_freq(theta, yarn), int(pos), out)
    return out


def rope_keys(k, theta: float = THETA, yarn=None) -> np.ndarray:
    """K' [rows, 2, 256] bf16 bits for keys at positions 0..rows-1."""
    k = _u16(k)
    out = np.zeros_like(k)
    lib().qo_rope_keys(k.shape[0], rope_inv_freq(theta, yarn), k, out)
    return out


def block_scores(qi_t, w_t, kblk, nb: int | None = None) -> np.ndarray:
    qi_t, w_t, kblk = _u16(qi_t), _u16(w_t), _u16(kblk)
    nb = kblk.shape[0] if nb is None else nb
    out = np.zeros(max(nb, 0), dtype=np.float64)
    if nb > 0:
        lib().qo_block_scores(qi_t, w_t, kblk, nb, out)
    return out


def select(s, c: int, budget: int):
    """(idx [budget] int32, scores [budget] f64, count)."""
    s = np.ascontiguousarray(np.asarray(s, dtype=np.float64))
    if s.size == 0:
        s = np.zeros(1)
    sel = np.zeros(budget, dtype=np.int32)
    ss = np.zeros(budget, dtype=np.float64)
    n = lib().qo_select(s, int(c), int(budget), sel, ss)
    return sel, ss, n


def attend(q_t, pos: int, k, v, sel, theta: float = THETA, scale: float = SCALE, yarn=None):
    q_t, k, v = _u16(q_t), _u16(k), _u16(v)
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32))
    o = np.zeros((HQ, D), dtype=np.float64)
    lse = np.zeros(HQ, dtype=np.float64)
    lib().qo_attend(q_t, int(pos), k, v, sel, int(sel.size), rope_inv_freq(theta, yarn),
                    _attn_scale(scale, yarn), o, lse)
    return o, lse


# ----------------------------------------------------------- whole layer --

def prefill_rows(inputs: dict, rows, budget: int, *, idx_given=None, want_o: bool = True,
                 theta: float = THETA, scale: float = SCALE, yarn=None, nthreads: int = 0):
    """QSA prefill for the listed query rows.

    inputs: dict of uint16 arrays q [L,24,256], k [L,2,256], v [L,2,256],
    qi [L,4,128], w [L,4], ki [L,128].  Returns dict idx, score, o, lse
    (per listed row)."""
    q, k, v = _u16(inputs["q"]), _u16(inputs["k"]), _u16(inputs["v"])
    qi, w, ki = _u16(inputs["qi"]), _u16(inputs["w"]), _u16(inputs["ki"])
    L = q.shape[0]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.size
    if n and (rows.min() < 0 or rows.max() >= L):
        raise ValueError("row out of range")
    idx = np.zeros((n, budget), dtype=np.int32)
    sc = np.zeros((n, budget), dtype=np.float64)
    o = np.zeros((n, HQ, D), dtype=np.float64) if want_o else None
    lse = np.zeros((n, HQ), dtype=np.float64) if want_o else None
    given = None if idx_given is None else np.ascontiguousarray(np.asarray(idx_given, dtype=np.int32))
    if given is not None and given.shape != (n, budget):
        raise ValueError("idx_given must be [nrows, budget]")
    lib().qo_prefill_rows(L, int(budget), rope_inv_freq(theta, yarn), _attn_scale(scale, yarn), q, k, v, qi, w,
                          ki, rows, n, given,
                          idx, sc, o, lse, int(nthreads))
    return {"idx": idx, "score": sc, "o": o, "lse": lse}


def prefill_scores(inputs: dict, rows, nthreads: int = 0) -> np.ndarray:
    """Dense block scores [nrows, L//4] (NaN where b >= c(t))."""
    qi, w, ki = _u16(inputs["qi"]), _u16(inputs["w"]), _u16(inputs["ki"])
    L = qi.shape[0]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((rows.size, L // BS), dtype=np.float64)
    if rows.size and L // BS:
        lib().qo_prefill_scores(L, qi, w, ki, rows, rows.size, out, int(nthreads))
    return out


def decode(inputs: dict, budget: int, *, idx_given=None, want_o: bool = True,
           theta: float = THETA, scale: float = SCALE, yarn=None, nthreads: int = 0):
    """QSA decode, one new token per sequence.

    inputs: q [B,24,256], qi [B,4,128], w [B,4], k [B,Tmax,2,256] (pre-RoPE),
    v [B,Tmax,2,256], ki [B,Tmax,128], seq_lens [B] (int64, the new token
    included)."""
    q, qi, w = _u16(inputs["q"]), _u16(inputs["qi"]), _u16(inputs["w"])
    k, v, ki = _u16(inputs["k"]), _u16(inputs["v"]), _u16(inputs["ki"])
    seq = np.ascontiguousarray(np.asarray(inputs["seq_lens"], dtype=np.int64))
    B, Tmax = k.shape[0], k.shape[1]
    if seq.min() < 1 or seq.max() > Tmax:
        raise ValueError("seq_lens out of range")
    idx = np.zeros((B, budget), dtype=np.int32)
    sc = np.zeros((B, budget), dtype=np.float64)
    o = np.zeros((B, HQ, D), dtype=np.float64) if want_o else None
    lse = np.zeros((B, HQ), dtype=np.float64) if want_o else None
    given = None if idx_given is None else np.ascontiguousarray(np.asarray(idx_given, dtype=np.int32))
    lib().qo_decode(B, Tmax, seq, int(budget), rope_inv_freq(theta, yarn), _attn_scale(scale, yarn), q, qi, w,
                    k, v, ki, given,
                    idx, sc, o, lse, int(nthreads))
    return {"idx": idx, "score": sc, "o": o, "lse": lse}
