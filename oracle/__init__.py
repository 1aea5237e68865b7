"""CPU oracle for the paged-attention hot path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  The product path
(``paged_kv_cache_198_gb300``) never imports it.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this module
builds it with gcc and marshals numpy / torch CPU arrays into it.  bf16 arrays
are passed as their 16-bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {
    -1: "bad argument",
    -2: "slot out of range",
    -3: "block id out of range",
    -4: "context length out of range",
    -5: "query length larger than context length",
    -6: "out of memory",
}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile liboracle.so next to oracle.c (OpenMP when gcc supports it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            LL = ctypes.c_longlong
            lib.oracle_kv_write.argtypes = [P, P, P, P, P, LL, LL, LL]
            lib.oracle_kv_write.restype = LL
            lib.oracle_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_double, P]
            lib.oracle_decode.restype = I
            lib.oracle_prefill.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I,
                                           ctypes.c_double, P]
            lib.oracle_prefill.restype = I
            lib.oracle_rope_double.argtypes = [P, P, I, LL, ctypes.c_double]
            lib.oracle_rope_double.restype = None
            lib.oracle_rope_kv_write.argtypes = [P, P, P, P, P, P, P, LL, I, I, I, LL,
                                                 ctypes.c_double]
            lib.oracle_rope_kv_write.restype = LL
            lib.oracle_round_bf16.argtypes = [P, P, LL]
            lib.oracle_round_bf16.restype = None
            lib.oracle_set_threads.argtypes = [I]
            lib.oracle_set_threads.restype = None
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = I
            _lib = lib
    return _lib


def _bits(x) -> np.ndarray:
    """bf16 torch tensor or uint16 numpy array -> contiguous uint16 numpy."""
    if hasattr(x, "view") and hasattr(x, "numpy") and not isinstance(x, np.ndarray):
        import torch

        assert x.dtype == torch.bfloat16, x.dtype
        x = x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, x.dtype
    return x


def _i32(x) -> np.ndarray:
    if hasattr(x, "numpy") and not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    x = np.ascontiguousarray(x, dtype=np.int32)
    return x


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def kv_write(k_cache, v_cache, k_new, v_new, slot_mapping):
    """Returns (k_cache', v_cache') as new uint16 arrays with the rows written."""
    kc = _bits(k_cache).copy()
    vc = _bits(v_cache).copy()
    kn = _bits(k_new)
    vn = _bits(v_new)
    sm = _i32(slot_mapping)
    nb, bs = kc.shape[0], kc.shape[1]
    row = int(np.prod(kc.shape[2:]))
    assert kn.shape[0] == sm.shape[0] and int(np.prod(kn.shape[1:])) == row
    rc = _load().oracle_kv_write(_ptr(kc), _ptr(vc), _ptr(kn), _ptr(vn), _ptr(sm),
                                 sm.shape[0], row, nb * bs)
    if rc < 0:
        raise OracleError(ERRORS.get(int(rc), str(rc)))
    return kc, vc


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, seq_mask=None):
    """float64 [S, Hq, D]; rows of sequences outside seq_mask are NaN."""
    qb = _bits(q)
    kc = _bits(k_cache)
    vc = _bits(v_cache)
    bt = _i32(block_tables)
    cl = _i32(context_lens)
    s, hq, d = qb.shape
    nb, bs, hkv, d2 = kc.shape
    assert d2 == d and vc.shape == kc.shape and cl.shape == (s,)
    mb = bt.shape[1] if bt.ndim == 2 else 0
    out = np.full((s, hq, d), np.nan, dtype=np.float64)
    mask = None
    if seq_mask is not None:
        mask = np.ascontiguousarray(seq_mask, dtype=np.uint8)
        assert mask.shape == (s,)
    rc = _load().oracle_decode(_ptr(out), _ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl),
                               s, hq, hkv, d, bs, nb, mb, float(scale),
                               _ptr(mask) if mask is not None else None)
    if rc != 0:
        raise OracleError(ERRORS.get(int(rc), str(rc)))
    return out


def prefill(q, query_start_loc, k_cache, v_cache, block_tables, context_lens, scale,
            row_mask=None):
    """float64 [Tq, Hq, D]; rows outside row_mask are NaN."""
    qb = _bits(q)
    qsl = _i32(query_start_loc)
    kc = _bits(k_cache)
    vc = _bits(v_cache)
    bt = _i32(block_tables)
    cl = _i32(context_lens)
    tq, hq, d = qb.shape
    nb, bs, hkv, d2 = kc.shape
    s = cl.shape[0]
    assert d2 == d and qsl.shape == (s + 1,)
    mb = bt.shape[1] if bt.ndim == 2 else 0
    out = np.full((tq, hq, d), np.nan, dtype=np.float64)
    mask = None
    if row_mask is not None:
        mask = np.ascontiguousarray(row_mask, dtype=np.uint8)
        assert mask.shape == (tq,)
    rc = _load().oracle_prefill(_ptr(out), _ptr(qb), _ptr(qsl), _ptr(kc), _ptr(vc), _ptr(bt),
                                _ptr(cl), s, tq, hq, hkv, d, bs, nb, mb, float(scale),
                                _ptr(mask) if mask is not None else None)
    if rc != 0:
        raise OracleError(ERRORS.get(int(rc), str(rc)))
    return out


def rope_double(x, pos: int, theta: float) -> np.ndarray:
    """Rotary embedding of one float64 head vector (no rounding)."""
    xv = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(xv)
    _load().oracle_rope_double(_ptr(y), _ptr(xv), xv.shape[0], int(pos), float(theta))
    return y


def rope_kv_write(q, k_cache, v_cache, k_new, v_new, slot_mapping, positions, theta):
    """Returns (q', k_cache', v_cache') as new uint16 arrays: q and the new K
    rotated at their positions (rounded to bf16), K/V rows written."""
    qb = _bits(q).copy() if q is not None else None
    kc = _bits(k_cache).copy()
    vc = _bits(v_cache).copy()
    kn = _bits(k_new)
    vn = _bits(v_new)
    sm = _i32(slot_mapping)
    pos = _i32(positions)
    nb, bs, hkv, d = kc.shape
    hq = qb.shape[1] if qb is not None else 0
    rc = _load().oracle_rope_kv_write(_ptr(qb) if qb is not None else None, _ptr(kc), _ptr(vc),
                                      _ptr(kn), _ptr(vn), _ptr(sm), _ptr(pos), sm.shape[0], hq,
                                      hkv, d, nb * bs, float(theta))
    if rc < 0:
        raise OracleError(ERRORS.get(int(rc), str(rc)))
    return qb, kc, vc


def round_bf16(values) -> np.ndarray:
    """float64 values -> bf16 bit patterns (round to nearest, ties to even)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_round_bf16(_ptr(out), _ptr(v), v.size)
    return out
