"""Exact long-context attention forward on one GB300 (sm_103a): thin Python binding of libcqsa_gb300.

The functions below carry the C ABI's names (``include/cqsa.h``) and only marshal arguments:
torch tensors or integer addresses become pointers, the current torch CUDA stream becomes the
``cudaStream_t``, and a non-OK status raises :class:`CqsaError` with the library's message. Every
step of the computation runs in the library's CUDA kernels. If the compiled library is missing the
import of the binding fails loudly (there is no fallback of any kind).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libcqsa_gb300.so")

CQSA_OK, CQSA_ERR_INVALID, CQSA_ERR_UNSUPPORTED, CQSA_ERR_CUDA, CQSA_ERR_OOM, CQSA_ERR_TIMEOUT, CQSA_ERR_DEVICE = (
    0, -1, -2, -3, -4, -5, -6)
CQSA_F16, CQSA_BF16, CQSA_F32 = 0, 1, 2
CQSA_LAYOUT_BHND, CQSA_LAYOUT_BNHD = 0, 1
CQSA_ENGINE_CLASSIC, CQSA_ENGINE_WAVE = 0, 1

EXPORTED = ("cqsa_attn_fwd", "cqsa_attn_fwd_chunk", "cqsa_merge_partials", "cqsa_stream_attn_fwd",
            "cqsa_attn_fwd_chunked_static", "cqsa_quorum_check", "cqsa_quorum_schedule", "cqsa_quorum_attn_fwd",
            "cqsa_quorum_attn_fwd_ex", "cqsa_release_cache", "cqsa_attn_bwd_workspace_size", "cqsa_attn_bwd", "cqsa_attn_bwd_dvec",
            "cqsa_attn_bwd_chunk", "cqsa_attn_bwd_cast", "cqsa_stream_attn_bwd", "cqsa_stream_attn_bwd_ex",
            "cqsa_status_string", "cqsa_last_error", "cqsa_device_error", "cqsa_set_timeout_ms",
            "cqsa_debug_set_fault", "cqsa_version", "cqsa_set_stream_kv_resident_bytes")
CQSA_STATIC_SCRATCH_BYTES = 32 << 20


class CqsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_name(status)}: {message}")
        self.status = status


class cqsa_stream_stats(ctypes.Structure):
    _fields_ = [("wall_ms", ctypes.c_double), ("compute_ms", ctypes.c_double), ("h2d_ms", ctypes.c_double),
                ("stall_ms", ctypes.c_double), ("h2d_bytes", ctypes.c_longlong), ("d2h_bytes", ctypes.c_longlong),
                ("peak_device_bytes", ctypes.c_longlong), ("n_chunks", ctypes.c_int), ("n_launches", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class cqsa_quorum_stats(ctypes.Structure):
    _fields_ = [("wall_ms", ctypes.c_double), ("compute_ms", ctypes.c_double), ("copy_ms", ctypes.c_double),
                ("copy_bytes", ctypes.c_longlong), ("peak_device_bytes", ctypes.c_longlong),
                ("chunk_tokens", ctypes.c_longlong), ("acc_host_bytes", ctypes.c_longlong),
                ("n_subproblems", ctypes.c_int), ("n_pairs", ctypes.c_int),
                ("n_chunk_loads", ctypes.c_int), ("n_launches", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


_vp, _i, _ll, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libcqsa_gb300.so is not built ({LIB_PATH}); run "
                          "`python -m exact_long_context_tcgen05_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    lib.cqsa_attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]
    lib.cqsa_attn_fwd_chunk.argtypes = [_vp, _vp, _vp, _ll, _ll, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _vp, _i, _vp]
    lib.cqsa_merge_partials.argtypes = [_vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _vp]
    lib.cqsa_stream_attn_fwd.argtypes = [_vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _ll, _i, _i, _f, _i, _ll,
                                         ctypes.POINTER(cqsa_stream_stats), _vp]
    lib.cqsa_attn_fwd_chunked_static.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp]
    lib.cqsa_quorum_check.argtypes = [_i, _vp, _i]
    lib.cqsa_quorum_schedule.argtypes = [_i, _vp, _i, _i, _i, _i, _vp, _ll]
    lib.cqsa_quorum_schedule.restype = _ll
    lib.cqsa_quorum_attn_fwd.argtypes = [_vp, _vp, _vp, _i, _i, _vp, _vp, _i, _i, _i, _ll, _i, _i, _f, _i, _i, _vp,
                                         _i, _i, _i, _i, ctypes.POINTER(cqsa_quorum_stats), _vp]
    lib.cqsa_quorum_attn_fwd_ex.argtypes = [_vp, _vp, _vp, _i, _i, _vp, _vp, _i, _i, _i, _ll, _i, _i, _f, _i, _i,
                                            _vp, _i, _i, _i, _i, _i, _ll, ctypes.POINTER(cqsa_quorum_stats), _vp]
    lib.cqsa_attn_bwd_workspace_size.argtypes = [_i, _i, _i, _i]
    lib.cqsa_attn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.cqsa_attn_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _i, _i, _i, _i,
                                  _i, _f, _i, _vp]
    lib.cqsa_attn_bwd_dvec.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]
    lib.cqsa_attn_bwd_chunk.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _ll, _ll, _i, _i, _i, _i, _i, _i, _f, _i, _vp,
                                        _vp, _vp, _vp]
    lib.cqsa_attn_bwd_cast.argtypes = [_vp, _vp, _ll, _i, _vp]
    lib.cqsa_stream_attn_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _ll, _i, _i, _f, _i,
                                         _ll, _vp]
    lib.cqsa_stream_attn_bwd_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _ll, _i, _i, _f, _i,
                                            _ll, ctypes.POINTER(cqsa_stream_stats), _vp]
    lib.cqsa_set_stream_kv_resident_bytes.argtypes = [_ll]
    lib.cqsa_set_stream_kv_resident_bytes.restype = None
    lib.cqsa_release_cache.argtypes = []
    lib.cqsa_release_cache.restype = _i
    lib.cqsa_status_string.argtypes = [_i]
    lib.cqsa_status_string.restype = ctypes.c_char_p
    lib.cqsa_last_error.argtypes = []
    lib.cqsa_last_error.restype = ctypes.c_char_p
    lib.cqsa_device_error.argtypes = [ctypes.POINTER(_i), ctypes.POINTER(_i), _i]
    lib.cqsa_set_timeout_ms.argtypes = [ctypes.c_uint]
    lib.cqsa_set_timeout_ms.restype = None
    lib.cqsa_debug_set_fault.argtypes = [_i]
    lib.cqsa_debug_set_fault.restype = _i
    lib.cqsa_version.argtypes = []
    lib.cqsa_version.restype = ctypes.c_char_p
    for name in ("cqsa_attn_fwd", "cqsa_attn_fwd_chunk", "cqsa_merge_partials", "cqsa_stream_attn_fwd",
                 "cqsa_attn_fwd_chunked_static", "cqsa_device_error", "cqsa_quorum_check", "cqsa_quorum_attn_fwd",
                 "cqsa_quorum_attn_fwd_ex"):
        getattr(lib, name).restype = _i
    return lib


lib = _load()


def status_name(status: int) -> str:
    return lib.cqsa_status_string(status).decode()


def last_error() -> str:
    return lib.cqsa_last_error().decode()


def _check(rc: int) -> int:
    if rc != CQSA_OK:
        raise CqsaError(rc, last_error())
    return rc


def _ptr(x) -> int | None:
    """Address of a torch tensor / numpy array / int (None and 0 stay NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    if hasattr(x, "data_ptr"):
        return x.data_ptr() or None
    if hasattr(x, "ctypes"):
        return x.ctypes.data or None
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def dtype_code(torch_dtype) -> int:
    import torch
    if torch_dtype == torch.float16:
        return CQSA_F16
    if torch_dtype == torch.bfloat16:
        return CQSA_BF16
    if torch_dtype == torch.float32:
        return CQSA_F32
    raise ValueError(f"unsupported dtype {torch_dtype}")


def cqsa_attn_fwd(q, k, v, out, lse, B, H, N, d, causal, scale, dtype, stream=None) -> int:
    return _check(lib.cqsa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, int(bool(causal)),
                                    float(scale), dtype, _stream(stream)))


def cqsa_attn_fwd_chunk(q_blk, k_blk, v_blk, q_off, kv_off, B, H, Nq, Nkv, d, causal, scale, dtype, O_part, LSE_part,
                        accumulate, stream=None) -> int:
    return _check(lib.cqsa_attn_fwd_chunk(_ptr(q_blk), _ptr(k_blk), _ptr(v_blk), q_off, kv_off, B, H, Nq, Nkv, d,
                                          int(bool(causal)), float(scale), dtype, _ptr(O_part), _ptr(LSE_part),
                                          int(bool(accumulate)), _stream(stream)))


def cqsa_merge_partials(O_parts, LSE_parts, n, out, lse, B, H, Nq, d, out_dtype, stream=None) -> int:
    po = (ctypes.c_void_p * max(n, 1))(*[_ptr(o) for o in O_parts][:n])
    pl = (ctypes.c_void_p * max(n, 1))(*[_ptr(x) for x in LSE_parts][:n])
    return _check(lib.cqsa_merge_partials(ctypes.cast(po, _vp), ctypes.cast(pl, _vp), n, _ptr(out), _ptr(lse), B, H,
                                          Nq, d, out_dtype, _stream(stream)))


def cqsa_stream_attn_fwd(q_host, k_host, v_host, layout, out, lse, out_on_host, B, H, N, d, causal, scale, dtype,
                         chunk_tokens, stats=None, stream=None) -> int:
    st = stats if stats is not None else cqsa_stream_stats()
    return _check(lib.cqsa_stream_attn_fwd(_ptr(q_host), _ptr(k_host), _ptr(v_host), layout, _ptr(out), _ptr(lse),
                                           int(bool(out_on_host)), B, H, N, d, int(bool(causal)), float(scale), dtype,
                                           chunk_tokens, ctypes.byref(st), _stream(stream)))


def cqsa_attn_fwd_chunked_static(q, k, v, out, lse, B, H, N, d, causal, scale, dtype, chunk_tokens,
                                 stream=None) -> int:
    """No-allocation chunked forward (scratch in the library's static device array)."""
    return _check(lib.cqsa_attn_fwd_chunked_static(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                                                   int(bool(causal)), float(scale), dtype, chunk_tokens,
                                                   _stream(stream)))


def _int_array(values):
    vals = [int(x) for x in values]
    return (ctypes.c_int * max(len(vals), 1))(*vals), len(vals)


def cqsa_quorum_check(c, interest_set) -> int:
    """CQSA_OK if interest_set is a perfect difference set modulo c (raises CqsaError otherwise)."""
    arr, l = _int_array(interest_set)
    return _check(lib.cqsa_quorum_check(c, ctypes.cast(arr, _vp), l))


def cqsa_quorum_schedule(c, interest_set, itr, n_chunks, causal):
    """The quorum schedule as a list of (subproblem, query chunk, key chunk) triples (host only)."""
    arr, l = _int_array(interest_set)
    n = lib.cqsa_quorum_schedule(c, ctypes.cast(arr, _vp), l, itr, n_chunks, int(bool(causal)), None, 0)
    if n < 0:
        raise CqsaError(int(n), last_error())
    buf = (ctypes.c_int * max(3 * n, 1))()
    m = lib.cqsa_quorum_schedule(c, ctypes.cast(arr, _vp), l, itr, n_chunks, int(bool(causal)),
                                 ctypes.cast(buf, _vp), n)
    if m != n:
        raise CqsaError(int(m) if m < 0 else CQSA_ERR_INVALID, last_error())
    return [(buf[3 * i], buf[3 * i + 1], buf[3 * i + 2]) for i in range(n)]


def cqsa_quorum_attn_fwd(q, k, v, layout, inputs_on_host, out, lse, out_on_host, B, H, N, d, causal, scale, dtype,
                         c, interest_set, itr, acc_on_host=False, max_parallel=1, stats=None, stream=None) -> int:
    st = stats if stats is not None else cqsa_quorum_stats()
    arr, l = _int_array(interest_set)
    return _check(lib.cqsa_quorum_attn_fwd(_ptr(q), _ptr(k), _ptr(v), layout, int(bool(inputs_on_host)), _ptr(out),
                                           _ptr(lse), int(bool(out_on_host)), B, H, N, d, int(bool(causal)),
                                           float(scale), dtype, c, ctypes.cast(arr, _vp), l, itr,
                                           int(bool(acc_on_host)), int(max_parallel), ctypes.byref(st),
                                           _stream(stream)))


def cqsa_quorum_attn_fwd_ex(q, k, v, layout, inputs_on_host, out, lse, out_on_host, B, H, N, d, causal, scale,
                            dtype, c, interest_set, itr, acc_on_host=False, max_parallel=1, engine=CQSA_ENGINE_WAVE,
                            wave_tokens=0, stats=None, stream=None) -> int:
    st = stats if stats is not None else cqsa_quorum_stats()
    arr, l = _int_array(interest_set)
    return _check(lib.cqsa_quorum_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), layout, int(bool(inputs_on_host)),
                                              _ptr(out), _ptr(lse), int(bool(out_on_host)), B, H, N, d,
                                              int(bool(causal)), float(scale), dtype, c, ctypes.cast(arr, _vp), l,
                                              itr, int(bool(acc_on_host)), int(max_parallel), int(engine),
                                              int(wave_tokens), ctypes.byref(st), _stream(stream)))


def cqsa_attn_bwd_workspace_size(B, H, N, d) -> int:
    return int(lib.cqsa_attn_bwd_workspace_size(B, H, N, d))


def cqsa_attn_bwd(q, k, v, out, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, causal, scale, dtype,
                  stream=None) -> int:
    return _check(lib.cqsa_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                    _ptr(dv), _ptr(workspace), int(workspace_bytes), B, H, N, d, int(bool(causal)),
                                    float(scale), dtype, _stream(stream)))


def cqsa_attn_bwd_dvec(out_blk, dout_blk, dvec_blk, B, H, Nq, d, dtype, stream=None) -> int:
    return _check(lib.cqsa_attn_bwd_dvec(_ptr(out_blk), _ptr(dout_blk), _ptr(dvec_blk), B, H, Nq, d, dtype,
                                         _stream(stream)))


def cqsa_attn_bwd_chunk(q_blk, k_blk, v_blk, dout_blk, lse_blk, dvec_blk, q_off, kv_off, B, H, Nq, Nkv, d, causal,
                        scale, dtype, dq_acc, dk_acc, dv_acc, stream=None) -> int:
    return _check(lib.cqsa_attn_bwd_chunk(_ptr(q_blk), _ptr(k_blk), _ptr(v_blk), _ptr(dout_blk), _ptr(lse_blk),
                                          _ptr(dvec_blk), q_off, kv_off, B, H, Nq, Nkv, d, int(bool(causal)),
                                          float(scale), dtype, _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc),
                                          _stream(stream)))


def cqsa_attn_bwd_cast(acc, out, n, dtype, stream=None) -> int:
    return _check(lib.cqsa_attn_bwd_cast(_ptr(acc), _ptr(out), n, dtype, _stream(stream)))


def cqsa_stream_attn_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, dtype, chunk_tokens,
                         stream=None) -> int:
    """Host-resident backward (all tensors in host memory, pinned for speed)."""
    return _check(lib.cqsa_stream_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq),
                                           _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), float(scale), dtype,
                                           chunk_tokens, _stream(stream)))


def cqsa_stream_attn_bwd_ex(q, k, v, out, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, dtype, chunk_tokens,
                            stats=None, stream=None):
    """cqsa_stream_attn_bwd that also fills a cqsa_stream_stats (kernel, copy and stall times); returns it."""
    st = stats if stats is not None else cqsa_stream_stats()
    _check(lib.cqsa_stream_attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq),
                                       _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), float(scale), dtype,
                                       chunk_tokens, ctypes.byref(st), _stream(stream)))
    return st


def cqsa_set_stream_kv_resident_bytes(nbytes: int) -> None:
    """K/V of cqsa_stream_attn_fwd stay on the device when they take at most nbytes (< 0: half of the free
    device memory, the default; 0: never, every pair through the fp32 accumulator)."""
    lib.cqsa_set_stream_kv_resident_bytes(int(nbytes))


def cqsa_release_cache() -> int:
    """Free the device buffers, events and streams the host-driven entry points keep between calls."""
    return _check(lib.cqsa_release_cache())


def cqsa_device_error(clear: bool = True):
    """(status, code, block) of the device error word after synchronising the device."""
    code, block = _i(0), _i(0)
    rc = lib.cqsa_device_error(ctypes.byref(code), ctypes.byref(block), int(bool(clear)))
    return rc, code.value, block.value


def cqsa_set_timeout_ms(ms: int) -> None:
    lib.cqsa_set_timeout_ms(ms)


def cqsa_debug_set_fault(kind: int) -> int:
    return _check(lib.cqsa_debug_set_fault(kind))


def cqsa_version() -> str:
    return lib.cqsa_version().decode()


# ---- torch conveniences (marshalling only) --------------------------------------------------------

def attention(q, k, v, *, causal=False, scale=None, return_lse=False, stream=None):
    """SDPA-shaped call on device tensors [B,H,N,d] (fp16/bf16): returns out (and lse [B,H,N] fp32)."""
    import torch
    B, H, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors of one shape [B,H,N,d]")
    q, k, v = (t.contiguous() for t in (q, k, v))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    cqsa_attn_fwd(q, k, v, out, lse, B, H, N, d, causal, 0.0 if scale is None else scale, dtype_code(q.dtype),
                  stream)
    return (out, lse) if return_lse else out


def attention_backward(q, k, v, out, dout, lse, *, causal=False, scale=None, stream=None):
    """Gradients (dq, dk, dv) of attention on device tensors [B,H,N,d], d = 64 or 128 (fp16/bf16), from
    the forward's out and lse ([B,H,N] fp32) and the upstream gradient dout."""
    import torch
    B, H, N, d = q.shape
    for t in (k, v, out, dout):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_cuda:
            raise ValueError("q, k, v, out, dout must be CUDA tensors of one shape and dtype [B,H,N,d]")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32:
        raise ValueError("lse must be a float32 tensor [B,H,N]")
    q, k, v, out, dout, lse = (t.contiguous() for t in (q, k, v, out, dout, lse))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = cqsa_attn_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    cqsa_attn_bwd(q, k, v, out, dout, lse, dq, dk, dv, ws, ws.numel(), B, H, N, d, causal,
                  0.0 if scale is None else scale, dtype_code(q.dtype), stream)
    return dq, dk, dv
