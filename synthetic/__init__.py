"""Seeded synthetic inputs (counter-based SplitMix64 + Box-Muller), shared by tests and bench.

This module holds no attention arithmetic. It generates Q/K/V tensors as raw fp16/bf16 bit
patterns (numpy ``uint16``) from ``(seed, tensor_id, logical element index)``, and draws the seeded
sets of query rows that large problems are checked on. The C source ``gen.c`` documents the exact
definition of every value. Note: these are not torch's random streams.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None

F16, BF16, F32 = 0, 1, 2
LAYOUT_BHND, LAYOUT_BNHD = 0, 1
# tensor ids of the Q/K/V streams and of the upstream output gradient dO of the backward
TID_Q, TID_K, TID_V, TID_DO = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile gen.c into a shared library next to it (gcc, OpenMP, no fast-math)."""
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
            lib.synth_sm64_at.restype = ctypes.c_uint64
            lib.synth_sm64_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_f32_to_f16.restype = ctypes.c_uint16
            lib.synth_f32_to_f16.argtypes = [ctypes.c_float]
            lib.synth_f32_to_bf16.restype = ctypes.c_uint16
            lib.synth_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.synth_normal.restype = None
            lib.synth_normal.argtypes = [ctypes.c_void_p] + [ctypes.c_int64] * 6 + [
                ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float]
            lib.synth_words.restype = None
            lib.synth_words.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                        ctypes.c_uint64, ctypes.c_uint64]
            _lib = lib
    return _lib


def sm64_at(state: int, n: int) -> int:
    """n-th SplitMix64 output of the sequence whose state starts at ``state``."""
    return int(_load().synth_sm64_at(state, n))


def words(n: int, seed: int, stream_id: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_words(out.ctypes.data, n, seed, stream_id, first)
    return out


def normal(B: int, H: int, N: int, d: int, *, seed: int = 0, tensor_id: int = 0, dtype: int = F16,
           layout: int = LAYOUT_BHND, mul: float = 1.0, n0: int = 0, n_cnt: int | None = None,
           out: np.ndarray | None = None) -> np.ndarray:
    """Tokens [n0, n0+n_cnt) of tensor ``tensor_id`` (logical shape [B,H,N,d]) as storage bits.

    Returns a uint16 array shaped [B,H,n_cnt,d] (layout 0) or [B,n_cnt,H,d] (layout 1), or float32
    for ``dtype=F32``. ``out`` may be any C-contiguous buffer of the right size (e.g. a numpy view
    of pinned host memory).
    """
    n_cnt = N - n0 if n_cnt is None else n_cnt
    if not (0 <= n0 and n0 + n_cnt <= N) or d < 1:
        raise ValueError("bad token range or head dim")
    shape = (B, H, n_cnt, d) if layout == LAYOUT_BHND else (B, n_cnt, H, d)
    np_dtype = np.float32 if dtype == F32 else np.uint16
    if out is None:
        out = np.empty(shape, dtype=np_dtype)
    if out.dtype != np_dtype or out.size != B * H * n_cnt * d or not out.flags.c_contiguous:
        raise ValueError("out buffer has the wrong dtype, size or strides")
    _load().synth_normal(out.ctypes.data, B, H, N, d, n0, n_cnt, layout, dtype, seed, tensor_id, mul)
    return out


def qkv(B: int, H: int, N: int, d: int, *, seed: int = 0, dtype: int = F16, k_mul: float = 1.0,
        layout: int = LAYOUT_BHND):
    """The Q, K, V of one workload: tensor ids 0, 1, 2 under ``seed``; K optionally scaled."""
    q = normal(B, H, N, d, seed=seed, tensor_id=TID_Q, dtype=dtype, layout=layout)
    k = normal(B, H, N, d, seed=seed, tensor_id=TID_K, dtype=dtype, layout=layout, mul=k_mul)
    v = normal(B, H, N, d, seed=seed, tensor_id=TID_V, dtype=dtype, layout=layout)
    return q, k, v


def f32_to_f16_bits(x) -> np.ndarray:
    lib = _load()
    flat = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.synth_f32_to_f16(float(v)) for v in flat], dtype=np.uint16)


def f32_to_bf16_bits(x) -> np.ndarray:
    lib = _load()
    flat = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.synth_f32_to_bf16(float(v)) for v in flat], dtype=np.uint16)


def sample_rows(B: int, H: int, N: int, count: int, *, seed: int = 1, must_i=(),
                chunk: int | None = None, causal_tile: int | None = None) -> np.ndarray:
    """Seeded (b, h, i) query rows to check a large problem on, as an int64 [n, 3] array.

    ``count`` rows are drawn uniformly (stream 7 of ``seed``): b, h, i each from one 64-bit draw
    reduced modulo its range. Always included, for every (b, h) = (0, 0) and (B-1, H-1): rows
    0, 1, 127, 128, N-1, the given ``must_i``, every chunk boundary (c*chunk-1, c*chunk) and,
    with ``causal_tile``, the last row of each tile if there are at most 64 tiles.
    """
    w = words(3 * count, seed, 7)
    b = (w[0::3] % np.uint64(B)).astype(np.int64)
    h = (w[1::3] % np.uint64(H)).astype(np.int64)
    i = (w[2::3] % np.uint64(N)).astype(np.int64)
    fixed = {0, 1, 127, 128, N - 1, *must_i}
    if chunk:
        for c in range(1, (N + chunk - 1) // chunk + 1):
            fixed.update({c * chunk - 1, c * chunk})
    if causal_tile and (N + causal_tile - 1) // causal_tile <= 64:
        fixed.update(t * causal_tile - 1 for t in range(1, (N + causal_tile - 1) // causal_tile + 1))
    fixed = sorted(x for x in fixed if 0 <= x < N)
    extra = [(bb, hh, ii) for (bb, hh) in {(0, 0), (B - 1, H - 1)} for ii in fixed]
    rows = np.concatenate([np.stack([b, h, i], axis=1), np.array(extra, dtype=np.int64).reshape(-1, 3)])
    # unique, keeping a deterministic order
    _, idx = np.unique(rows, axis=0, return_index=True)
    return rows[np.sort(idx)]
