"""fp64 CPU oracle for exact softmax attention -- TEST INFRASTRUCTURE ONLY.

This package is the checker, not the product.  Only ``tests/``, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it.  It shares no code with the GPU library: the arithmetic lives in
``attn_oracle.c`` (plain C, double precision, OpenMP over query rows), which
this module compiles with gcc and calls through ctypes.  Inputs are numpy
float64 arrays holding the already-rounded 16-bit values; nothing here knows
about bf16/fp16 encodings.

Definitions follow the pages: the attention output softmax(scale * Q K^T) V
and its naive three-pass evaluation ("FlashAttention: Why Tiling Attention
Makes Transformers Fast Without Changing the Result", section "The problem is
memory, not arithmetic"), the per-row logsumexp output ("FlashAttention:
IO-aware attention kernels", table "What goes in, what comes out"), and the
blocked online softmax ("Flash attention and memory-efficient attention
variants", sections "Tiling and the running (online) softmax" and "Worked
example: tracing the running statistics by hand").  Pins for every function
are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_WINDOW = 2
_MASKS = {"none": MASK_NONE, "causal": MASK_CAUSAL, "window": MASK_WINDOW,
          "sliding_window": MASK_WINDOW}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_default = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def compile_source(src: str, out: str) -> str:
    """Compile one oracle C source into a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so if out of date."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _mask(mask) -> int:
    if isinstance(mask, str):
        return _MASKS[mask]
    return int(mask)


def _shapes(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """(B, H, Sq, d, Hkv, Sk) of q [B,H,Sq,d] and k, v [B,Hkv,Sk,d]."""
    if q.ndim != 4 or k.ndim != 4:
        raise ValueError("q, k, v must be 4-D [B,heads,S,d]")
    B, H, Sq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if k.shape != (B, Hkv, Sk, d) or v.shape != (B, Hkv, Sk, d):
        raise ValueError("k and v must be [B,Hkv,Sk,d] matching q")
    if Hkv < 1 or H % Hkv != 0:
        raise ValueError("the K/V head count must divide the query head count")
    return B, H, Sq, d, Hkv, Sk


class OracleLib:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_attn_naive.restype = ctypes.c_int
        lib.oracle_attn_naive.argtypes = [
            _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
            _i64p, ctypes.c_int64, _dp, _dp]
        lib.oracle_attn_blocked.restype = ctypes.c_int
        lib.oracle_attn_blocked.argtypes = [
            _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, _dp, _dp]
        lib.oracle_online_trace.restype = ctypes.c_int
        lib.oracle_online_trace.argtypes = [
            _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
            _dp, _dp, _dp, _dp, _dp]
        lib.oracle_probs.restype = ctypes.c_int
        lib.oracle_probs.argtypes = [
            _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            ctypes.c_int, ctypes.c_int, _dp]
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_attn_bwd.argtypes = [
            _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
            _dp, _dp, _dp]
        _i32p = ctypes.POINTER(ctypes.c_int32)
        lib.oracle_attn_paged.restype = ctypes.c_int
        lib.oracle_attn_paged.argtypes = [
            _dp, _dp, _dp, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
            _dp, _dp]
        lib.oracle_set_threads.restype = None
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        self.lib = lib
        self.path = path

    def set_threads(self, n: int) -> None:
        self.lib.oracle_set_threads(int(n))

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def attention(self, q, k, v, scale: float, mask="none", window: int = 0, rows=None):
        """Naive fp64 attention.

        q: [B,H,Sq,d], k, v: [B,Hkv,Sk,d] with Hkv dividing H (grouped-query
        attention: query head h reads K/V head h // (H // Hkv); Hkv == H is
        plain multi-head attention).  Returns (o, lse): o is [B,H,Sq,d]
        and lse [B,H,Sq] when ``rows`` is None; otherwise ``rows`` lists flat
        query-row indices (b*H + h)*Sq + i and o is [len(rows), d], lse
        [len(rows)].
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, Sq, d, Hkv, Sk = _shapes(q, k, v)
        if rows is None:
            o = np.empty((B, H, Sq, d), np.float64)
            lse = np.empty((B, H, Sq), np.float64)
            rc = self.lib.oracle_attn_naive(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, Sq, Sk, d,
                                            float(scale), _mask(mask), int(window), None, 0,
                                            _ptr(o), _ptr(lse))
        else:
            r = np.ascontiguousarray(rows, dtype=np.int64)
            o = np.empty((r.size, d), np.float64)
            lse = np.empty((r.size,), np.float64)
            rc = self.lib.oracle_attn_naive(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, Sq, Sk, d,
                                            float(scale), _mask(mask), int(window),
                                            r.ctypes.data_as(_i64p), r.size, _ptr(o), _ptr(lse))
        if rc != 0:
            raise ValueError("oracle_attn_naive rejected its arguments")
        return o, lse

    def attention_blocked(self, q, k, v, scale: float, mask="none", window: int = 0,
                          block_size: int = 2):
        """Blocked online-softmax fp64 attention (second, independent form).

        Shapes as in ``attention`` (K/V may have fewer heads than Q)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, Sq, d, Hkv, Sk = _shapes(q, k, v)
        o = np.empty((B, H, Sq, d), np.float64)
        lse = np.empty((B, H, Sq), np.float64)
        rc = self.lib.oracle_attn_blocked(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, Sq, Sk, d,
                                          float(scale), _mask(mask), int(window),
                                          int(block_size), _ptr(o), _ptr(lse))
        if rc != 0:
            raise ValueError("oracle_attn_blocked rejected its arguments")
        return o, lse

    def attention_bwd(self, q, k, v, dout, scale: float, mask="none", window: int = 0):
        """Gradients (dq, dk, dv) of sum(O * dout) for O = attention(q, k, v).

        Shapes as in ``attention``; dout like q.  dk, dv have k's shape (with
        shared K/V heads they sum over the query heads that read them).
        """
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        B, H, Sq, d, Hkv, Sk = _shapes(q, k, v)
        if dout.shape != q.shape:
            raise ValueError("dout must have q's shape")
        dq = np.empty_like(q)
        dk = np.empty_like(k)
        dv = np.empty_like(v)
        rc = self.lib.oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, H, Hkv, Sq, Sk,
                                      d, float(scale), _mask(mask), int(window), _ptr(dq),
                                      _ptr(dk), _ptr(dv))
        if rc != 0:
            raise ValueError("oracle_attn_bwd rejected its arguments")
        return dq, dk, dv

    def attention_paged(self, q, k_cache, v_cache, block_table, seq_lens, scale: float,
                        mask="none"):
        """Attention of the Sq new rows of each request over its paged K/V cache.

        q: [B, H, Sq, d]; k_cache, v_cache: [num_blocks, Hkv, block_size, d];
        block_table: int [B, max_blocks]; seq_lens: int [B] (cached tokens,
        the last Sq being the new rows').  mask: "none" or "causal" (row i at
        position seq_lens[b] - Sq + i).  Returns (o [B,H,Sq,d], lse [B,H,Sq]).
        """
        q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, H, Sq, d = q.shape
        nb, Hkv, bs, d2 = kc.shape
        if vc.shape != kc.shape or d2 != d or bt.ndim != 2 or bt.shape[0] != B or sl.shape != (B,):
            raise ValueError("shapes: q [B,H,Sq,d]; caches [blocks,Hkv,bs,d]; table [B,n]; lens [B]")
        o = np.empty((B, H, Sq, d), np.float64)
        lse = np.empty((B, H, Sq), np.float64)
        i32 = ctypes.POINTER(ctypes.c_int32)
        rc = self.lib.oracle_attn_paged(_ptr(q), _ptr(kc), _ptr(vc), bt.ctypes.data_as(i32),
                                        sl.ctypes.data_as(i32), B, H, Hkv, Sq, d, bs, bt.shape[1],
                                        nb, float(scale), _mask(mask), _ptr(o), _ptr(lse))
        if rc != 0:
            raise ValueError("oracle_attn_paged rejected its arguments")
        return o, lse

    def online_trace(self, q_row, K, V, scale: float, block_size: int):
        """Running (m, l, unnormalised O) after each key block for one query row.

        Returns dict with m [nblk], l [nblk], o_unnorm [nblk, d], o [d], lse.
        """
        q_row, K, V = _f64(q_row), _f64(K), _f64(V)
        Sk, d = K.shape
        nblk = -(-Sk // block_size)
        tm = np.empty(nblk, np.float64)
        tl = np.empty(nblk, np.float64)
        to = np.empty((nblk, d), np.float64)
        o = np.empty(d, np.float64)
        lse = np.empty(1, np.float64)
        rc = self.lib.oracle_online_trace(_ptr(q_row), _ptr(K), _ptr(V), Sk, d, float(scale),
                                          int(block_size), _ptr(tm), _ptr(tl), _ptr(to),
                                          _ptr(o), _ptr(lse))
        if rc != 0:
            raise ValueError("oracle_online_trace rejected its arguments")
        return {"m": tm, "l": tl, "o_unnorm": to, "o": o, "lse": float(lse[0])}

    def probs(self, q_head, k_head, scale: float, mask="none", window: int = 0):
        """Normalised probability matrix P [Sq, Sk] of one head."""
        q_head, k_head = _f64(q_head), _f64(k_head)
        Sq, d = q_head.shape
        Sk = k_head.shape[0]
        P = np.empty((Sq, Sk), np.float64)
        rc = self.lib.oracle_probs(_ptr(q_head), _ptr(k_head), Sq, Sk, d, float(scale),
                                   _mask(mask), int(window), _ptr(P))
        if rc != 0:
            raise ValueError("oracle_probs rejected its arguments")
        return P


def default() -> OracleLib:
    """The oracle built from attn_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default


def set_threads(n: int) -> None:
    default().set_threads(n)


def max_threads() -> int:
    return default().max_threads()


def attention(*args, **kwargs):
    return default().attention(*args, **kwargs)


def attention_blocked(*args, **kwargs):
    return default().attention_blocked(*args, **kwargs)


def attention_bwd(*args, **kwargs):
    return default().attention_bwd(*args, **kwargs)


def attention_paged(*args, **kwargs):
    return default().attention_paged(*args, **kwargs)


def online_trace(*args, **kwargs):
    return default().online_trace(*args, **kwargs)


def probs(*args, **kwargs):
    return default().probs(*args, **kwargs)


def visible_pairs(Sq: int, Sk: int, mask="none", window: int = 0) -> int:
    """Number of (query, key) pairs that the mask leaves visible in one head.

    Counting by the same visibility rule as attn_oracle.c: none -> all keys;
    causal -> keys j <= i; window W -> i - W < j <= i; always j < Sk.
    """
    mk = _mask(mask)
    total = 0
    for i in range(Sq):
        if mk == MASK_NONE:
            total += Sk
            continue
        hi = min(i, Sk - 1)
        lo = 0 if mk == MASK_CAUSAL else max(0, i - int(window) + 1)
        total += max(0, hi - lo + 1)
    return total
