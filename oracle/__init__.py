"""CPU FP64 oracle for exact attention forward, chunk partials and the LSE merge.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package; the library in ``exact_long_context_tcgen05_gb300`` never does, and
shares no code with it. The arithmetic is in ``oracle.c`` (plain C, double precision, OpenMP over
rows), which states the definition it follows and where the pages state the problem.

The backward (``attn_bwd``, ``attn_bwd_f64``; at listed rows or columns ``attn_bwd_rows`` and
``attn_bwd_cols``, which agree with ``attn_bwd`` wherever both run) is the chain rule through the softmax, pinned in
``tests/test_oracle_bwd.py`` by central finite differences of the loss sum(dO * O), by sympy's symbolic
gradient of the written-out loss on a 3-token problem, by the forward
part agreeing with ``attn_full``, by the key-shift invariance sum_j dK_j = 0 and by the uniform-score
closed form of dV.

Pins (``tests/test_oracle.py``): normalisation (V = 1 gives O = 1), causal row 0 (O_0 = v_0,
LSE_0 = s_00), uniform scores (Q = 0 gives the mean of the allowed V rows and LSE = ln|A_i|),
affinity in V, permutation equivariance, the two-key closed form, hand-derived fixtures under
``tests/golden/``, a separately written long-double brute force without max subtraction, and
chunk-plus-merge equal to the monolithic result over many partitions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1
LAYOUT_BHND, LAYOUT_BNHD = 0, 1

_p = ctypes.c_void_p
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c (gcc, OpenMP; no fast-math and no FMA contraction, so x86 and Arm agree)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_attn_rows.restype = ctypes.c_int
            lib.oracle_attn_rows.argtypes = [_p, _p, _p, ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, _i64,
                                             _i64, _i64, _i64, ctypes.c_int, ctypes.c_double, _p, _i64, _p, _p]
            lib.oracle_merge.restype = ctypes.c_int
            lib.oracle_merge.argtypes = [_p, _p, ctypes.c_int, _i64, _i64, _p, _p]
            lib.oracle_attn_bruteforce_ld.restype = ctypes.c_int
            lib.oracle_attn_bruteforce_ld.argtypes = [_p, _p, _p, ctypes.c_int, _i64, _i64, _i64, _i64,
                                                      ctypes.c_int, ctypes.c_double, _p, _p]
            lib.oracle_widen.restype = None
            lib.oracle_widen.argtypes = [_p, _i64, ctypes.c_int, _p]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_double,
                                            _p, _p, _p, _p, _p]
            lib.oracle_attn_bwd_rows.restype = ctypes.c_int
            lib.oracle_attn_bwd_rows.argtypes = [_p, _p, _p, _p, ctypes.c_int, _i64, _i64, _i64, _i64, ctypes.c_int,
                                                 ctypes.c_double, _p, _i64, _p]
            lib.oracle_attn_bwd_cols.restype = ctypes.c_int
            lib.oracle_attn_bwd_cols.argtypes = [_p, _p, _p, _p, ctypes.c_int, _i64, _i64, _i64, _i64, ctypes.c_int,
                                                 ctypes.c_double, _p, _i64, _p, _p]
            _lib = lib
    return _lib


def _u16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are fp16/bf16 storage bits (numpy uint16)")
    return x


def default_scale(d: int) -> float:
    """SDPA's default 1/sqrt(d), as the fp32 value the GPU receives, widened to double."""
    return float(np.float32(1.0 / np.sqrt(d)))


def attn_rows(q, k, v, *, B, H, Nq, Nkv=None, d, causal, scale=None, dtype=F16, layout=LAYOUT_BHND,
              q_off=0, kv_off=0, rows=None):
    """Oracle output and LSE (float64) of the given (b, h, i) rows; all rows if ``rows`` is None.

    Returns (out [nrows, d], lse [nrows]) and the rows array used.
    """
    Nkv = Nq if Nkv is None else Nkv
    scale = default_scale(d) if scale is None else float(np.float32(scale))
    if rows is None:
        bb, hh, ii = np.meshgrid(np.arange(B), np.arange(H), np.arange(Nq), indexing="ij")
        rows = np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    q, k, v = _u16(q), _u16(k), _u16(v)
    if q.size != B * H * Nq * d or k.size != B * H * Nkv * d or v.size != B * H * Nkv * d:
        raise ValueError("tensor sizes do not match B, H, N, d")
    out = np.empty((len(rows), d), dtype=np.float64)
    lse = np.empty(len(rows), dtype=np.float64)
    rc = _load().oracle_attn_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, layout, dtype, B, H, Nq, Nkv, d,
                                  q_off, kv_off, int(bool(causal)), scale, rows.ctypes.data, len(rows),
                                  out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_attn_rows rejected its arguments")
    return out, lse, rows


def attn_full(q, k, v, *, B, H, N, d, causal, scale=None, dtype=F16):
    """Whole-problem oracle in [B,H,N,d] / [B,H,N] shape (float64)."""
    out, lse, _ = attn_rows(q, k, v, B=B, H=H, Nq=N, d=d, causal=causal, scale=scale, dtype=dtype)
    return out.reshape(B, H, N, d), lse.reshape(B, H, N)


def merge(O_parts, LSE_parts):
    """Exact FP64 merge of partials. O_parts: list of [..., d] arrays; LSE_parts: list of [...] arrays."""
    n = len(O_parts)
    if n < 1 or len(LSE_parts) != n:
        raise ValueError("need n >= 1 matching partials")
    shape = np.shape(LSE_parts[0])
    d = np.shape(O_parts[0])[-1]
    Os = [np.ascontiguousarray(o, dtype=np.float64).reshape(-1, d) for o in O_parts]
    Ls = [np.ascontiguousarray(l_, dtype=np.float64).ravel() for l_ in LSE_parts]
    rows = Ls[0].size
    if any(o.shape[0] != rows for o in Os) or any(l_.size != rows for l_ in Ls):
        raise ValueError("partials disagree in shape")
    po = (ctypes.c_void_p * n)(*[o.ctypes.data for o in Os])
    pl = (ctypes.c_void_p * n)(*[l_.ctypes.data for l_ in Ls])
    out = np.empty((rows, d), dtype=np.float64)
    lse = np.empty(rows, dtype=np.float64)
    rc = _load().oracle_merge(ctypes.cast(po, ctypes.c_void_p), ctypes.cast(pl, ctypes.c_void_p), n, rows, d,
                              out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_merge rejected its arguments")
    return out.reshape(*shape, d), lse.reshape(shape)


def bruteforce_ld(q, k, v, *, B, H, N, d, causal, scale=None, dtype=F16):
    """Separately written long-double brute force (no max subtraction) for tiny problems."""
    scale = default_scale(d) if scale is None else float(np.float32(scale))
    q, k, v = _u16(q), _u16(k), _u16(v)
    out = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().oracle_attn_bruteforce_ld(q.ctypes.data, k.ctypes.data, v.ctypes.data, dtype, B, H, N, d,
                                           int(bool(causal)), scale, out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_attn_bruteforce_ld rejected its arguments")
    return out, lse


def widen(bits, dtype=F16) -> np.ndarray:
    """fp16/bf16 storage bits -> exact float64 values."""
    bits = _u16(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_widen(bits.ctypes.data, bits.size, dtype, out.ctypes.data)
    return out


def attn_bwd_f64(q, k, v, dout, *, causal, scale):
    """Backward from double inputs [B,H,N,d]: returns dict(out, lse, dq, dk, dv) in float64."""
    q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, dout))
    if q.ndim != 4 or any(x.shape != q.shape for x in (k, v, dout)):
        raise ValueError("q, k, v, dout must share one [B,H,N,d] shape")
    B, H, N, d = q.shape
    res = {n: np.empty(q.shape, dtype=np.float64) for n in ("out", "dq", "dk", "dv")}
    res["lse"] = np.empty((B, H, N), dtype=np.float64)
    rc = _load().oracle_attn_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, B, H, N, d,
                                 int(bool(causal)), float(scale), res["out"].ctypes.data, res["lse"].ctypes.data,
                                 res["dq"].ctypes.data, res["dk"].ctypes.data, res["dv"].ctypes.data)
    if rc != 0:
        raise ValueError("oracle_attn_bwd rejected its arguments")
    return res


def attn_bwd(q, k, v, dout, *, B, H, N, d, causal, scale=None, dtype=F16):
    """Backward of [B,H,N,d] fp16/bf16 storage bits (q, k, v, dout), widened exactly; scale defaults to
    the fp32 1/sqrt(d). Returns dict(out, lse, dq, dk, dv) in float64."""
    scale = default_scale(d) if scale is None else float(np.float32(scale))
    shape = (B, H, N, d)
    ws = [widen(x, dtype).reshape(shape) for x in (q, k, v, dout)]
    return attn_bwd_f64(*ws, causal=causal, scale=scale)


def _triples(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.int64)
    if x.ndim != 2 or x.shape[1] != 3:
        raise ValueError("expected an array of (b, h, index) triples")
    return x


def attn_bwd_rows(q, k, v, dout, *, B, H, N, d, causal, rows, scale=None, dtype=F16):
    """dq (float64, [nrows, d]) of the listed (b, h, i) query rows of a [B,H,N,d] problem (16-bit bits)."""
    scale = default_scale(d) if scale is None else float(np.float32(scale))
    q, k, v, dout = (_u16(x) for x in (q, k, v, dout))
    if any(x.size != B * H * N * d for x in (q, k, v, dout)):
        raise ValueError("tensor sizes do not match B, H, N, d")
    rows = _triples(rows)
    dq = np.empty((len(rows), d), dtype=np.float64)
    rc = _load().oracle_attn_bwd_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, dtype, B, H, N,
                                      d, int(bool(causal)), scale, rows.ctypes.data, len(rows), dq.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_attn_bwd_rows rejected its arguments")
    return dq


def attn_bwd_cols(q, k, v, dout, *, B, H, N, d, causal, cols, scale=None, dtype=F16):
    """dk, dv (float64, [ncols, d] each) of the listed (b, h, j) key columns of a [B,H,N,d] problem."""
    scale = default_scale(d) if scale is None else float(np.float32(scale))
    q, k, v, dout = (_u16(x) for x in (q, k, v, dout))
    if any(x.size != B * H * N * d for x in (q, k, v, dout)):
        raise ValueError("tensor sizes do not match B, H, N, d")
    cols = _triples(cols)
    dk = np.empty((len(cols), d), dtype=np.float64)
    dv = np.empty((len(cols), d), dtype=np.float64)
    rc = _load().oracle_attn_bwd_cols(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, dtype, B, H, N,
                                      d, int(bool(causal)), scale, cols.ctypes.data, len(cols), dk.ctypes.data,
                                      dv.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_attn_bwd_cols rejected its arguments")
    return dk, dv
