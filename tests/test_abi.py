"""The C-ABI library loads and exports every symbol include/cqsa.h declares; arguments are validated
before anything is launched (these calls return errors without touching a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cq():
    import __graft_entry__
    __graft_entry__._builder().build()
    import exact_long_context_tcgen05_gb300 as m
    return m


def _declared():
    with open(os.path.join(ROOT, "include", "cqsa.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(cqsa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(cq):
    lib = ctypes.CDLL(cq.LIB_PATH)
    declared = _declared()
    assert {"cqsa_attn_fwd", "cqsa_attn_fwd_chunk", "cqsa_merge_partials", "cqsa_stream_attn_fwd"} <= set(declared)
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(cq.EXPORTED)


def test_status_strings(cq):
    assert cq.status_name(cq.CQSA_OK) == "CQSA_OK"
    assert cq.status_name(cq.CQSA_ERR_OOM) == "CQSA_ERR_OOM"
    assert cq.status_name(12345) == "CQSA_UNKNOWN_STATUS"
    assert cq.cqsa_version() == "0.1.0"


def test_release_cache_without_device(cq):
    """Freeing the (empty) resource cache is a no-op that succeeds on a machine without a GPU."""
    assert cq.cqsa_release_cache() == cq.CQSA_OK


def test_quorum_validation(cq):
    st, msg = _rc(lambda: cq.cqsa_quorum_attn_fwd(FAKE, FAKE, FAKE, 0, False, FAKE, None, False, 1, 1, 256, 64, True,
                                                  0.0, cq.CQSA_F16, 7, (0, 1, 3), 1, max_parallel=0, stream=0))
    assert st == cq.CQSA_ERR_INVALID and "max_parallel" in msg
    st, msg = _rc(lambda: cq.cqsa_quorum_attn_fwd(FAKE, FAKE, FAKE, 0, False, FAKE, None, False, 1, 1, 256, 96, True,
                                                  0.0, cq.CQSA_F16, 7, (0, 1, 3), 1, stream=0))
    assert st == cq.CQSA_ERR_UNSUPPORTED
    st, msg = _rc(lambda: cq.cqsa_quorum_attn_fwd(FAKE, FAKE, FAKE, 0, False, FAKE, None, False, 1, 1, 256, 64, True,
                                                  0.0, cq.CQSA_F16, 7, (0, 1, 2), 1, stream=0))
    assert st == cq.CQSA_ERR_INVALID and "difference" in msg
    # the engine-selecting entry: unknown engine and negative budget are rejected before any launch
    st, msg = _rc(lambda: cq.cqsa_quorum_attn_fwd_ex(FAKE, FAKE, FAKE, 0, False, FAKE, None, False, 1, 1, 256, 64,
                                                     True, 0.0, cq.CQSA_F16, 7, (0, 1, 3), 1, engine=9, stream=0))
    assert st == cq.CQSA_ERR_INVALID and "engine" in msg
    st, msg = _rc(lambda: cq.cqsa_quorum_attn_fwd_ex(FAKE, FAKE, FAKE, 0, False, FAKE, None, False, 1, 1, 256, 64,
                                                     True, 0.0, cq.CQSA_F16, 7, (0, 1, 3), 1, wave_tokens=-1, stream=0))
    assert st == cq.CQSA_ERR_INVALID and "wave_tokens" in msg


def _rc(fn):
    try:
        fn()
    except Exception as e:  # noqa: BLE001
        return getattr(e, "status", None), str(e)
    return 0, ""


FAKE = 0x10000  # aligned, never dereferenced: validation fails before any launch


def test_attn_fwd_validation(cq):
    L = cq.lib
    assert L.cqsa_attn_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 128, 96, 1, 0.0, cq.CQSA_F16, None) == cq.CQSA_ERR_UNSUPPORTED
    assert "head dim 96" in cq.last_error()
    assert L.cqsa_attn_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 128, 64, 1, 0.0, cq.CQSA_F32, None) == cq.CQSA_ERR_UNSUPPORTED
    assert L.cqsa_attn_fwd(FAKE, FAKE, FAKE, FAKE, None, 0, 1, 128, 64, 1, 0.0, cq.CQSA_F16, None) == cq.CQSA_ERR_INVALID
    assert L.cqsa_attn_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 0, 64, 1, 0.0, cq.CQSA_F16, None) == cq.CQSA_ERR_INVALID
    assert L.cqsa_attn_fwd(None, FAKE, FAKE, FAKE, None, 1, 1, 128, 64, 1, 0.0, cq.CQSA_F16, None) == cq.CQSA_ERR_INVALID
    assert L.cqsa_attn_fwd(FAKE + 2, FAKE, FAKE, FAKE, None, 1, 1, 128, 64, 1, 0.0, cq.CQSA_F16, None) == cq.CQSA_ERR_INVALID
    assert "aligned" in cq.last_error()
    assert L.cqsa_attn_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 128, 64, 1, float("nan"), cq.CQSA_F16, None) == cq.CQSA_ERR_INVALID
    assert L.cqsa_attn_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 128, 64, 1, float("inf"), cq.CQSA_F16, None) == cq.CQSA_ERR_INVALID


def test_chunk_validation(cq):
    L = cq.lib
    args = dict(q=FAKE, k=FAKE, v=FAKE, qo=0, ko=0, B=1, H=1, Nq=128, Nkv=128, d=64, c=1, s=0.0, dt=cq.CQSA_F16,
                O=FAKE, Lp=FAKE, acc=0)

    def call(**kw):
        a = {**args, **kw}
        return L.cqsa_attn_fwd_chunk(a["q"], a["k"], a["v"], a["qo"], a["ko"], a["B"], a["H"], a["Nq"], a["Nkv"],
                                     a["d"], a["c"], a["s"], a["dt"], a["O"], a["Lp"], a["acc"], None)
    assert call(qo=-1) == cq.CQSA_ERR_INVALID
    assert call(O=None) == cq.CQSA_ERR_INVALID
    assert call(Nkv=-1) == cq.CQSA_ERR_INVALID
    assert call(k=None) == cq.CQSA_ERR_INVALID
    assert call(d=32) == cq.CQSA_ERR_UNSUPPORTED
    assert call(Lp=FAKE + 1) == cq.CQSA_ERR_INVALID


def test_merge_validation(cq):
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    bad = (ctypes.c_void_p * 2)(FAKE, FAKE + 8)
    L = cq.lib
    v = ctypes.cast(arr, ctypes.c_void_p)
    assert L.cqsa_merge_partials(v, v, 0, FAKE, None, 1, 1, 1, 64, 0, None) == cq.CQSA_ERR_INVALID
    assert L.cqsa_merge_partials(v, v, 1025, FAKE, None, 1, 1, 1, 64, 0, None) == cq.CQSA_ERR_INVALID
    assert L.cqsa_merge_partials(v, v, 2, FAKE, None, 1, 1, 1, 48, 0, None) == cq.CQSA_ERR_UNSUPPORTED
    assert L.cqsa_merge_partials(v, v, 2, FAKE, None, 1, 1, 1, 64, 7, None) == cq.CQSA_ERR_UNSUPPORTED
    assert L.cqsa_merge_partials(ctypes.cast(bad, ctypes.c_void_p), v, 2, FAKE, None, 1, 1, 1, 64, 0, None) == cq.CQSA_ERR_INVALID
    assert "part 1" in cq.last_error()


def test_stream_validation(cq):
    L = cq.lib
    st = cq.cqsa_stream_stats()
    f = lambda **kw: L.cqsa_stream_attn_fwd(  # noqa: E731
        kw.get("q", FAKE), FAKE, FAKE, kw.get("layout", 1), FAKE, None, 1, 1, 1, kw.get("N", 1000), 64, 1, 0.0,
        cq.CQSA_F16, kw.get("C", 256), ctypes.byref(st), None)
    assert f(C=100) == cq.CQSA_ERR_INVALID
    assert f(C=0) == cq.CQSA_ERR_INVALID
    assert f(layout=5) == cq.CQSA_ERR_UNSUPPORTED
    assert f(q=None) == cq.CQSA_ERR_INVALID
    assert f(N=0) == cq.CQSA_ERR_INVALID


def test_bwd_validation(cq):
    """The backward validates before launching: head dim, workspace size, pointers, alignment."""
    L = cq.lib
    need = cq.cqsa_attn_bwd_workspace_size(1, 2, 256, 64)
    assert need == ((2 * 256 * 64 * 4 + 255) // 256) * 256 + 2 * 256 * 4
    assert cq.cqsa_attn_bwd_workspace_size(0, 2, 256, 64) == 0

    def call(d=64, ws_bytes=need, q=FAKE, lse=FAKE, dtype=cq.CQSA_F16):
        return L.cqsa_attn_bwd(q, FAKE, FAKE, FAKE, FAKE, lse, FAKE, FAKE, FAKE, FAKE, ws_bytes, 1, 2, 256, d, 1, 0.0,
                               dtype, None)
    assert call(d=96) == cq.CQSA_ERR_UNSUPPORTED and "head dim" in cq.last_error()
    assert call(ws_bytes=need - 16) == cq.CQSA_ERR_INVALID and "workspace" in cq.last_error()
    assert call(q=None) == cq.CQSA_ERR_INVALID
    assert call(q=FAKE + 8) == cq.CQSA_ERR_INVALID and "aligned" in cq.last_error()
    assert call(lse=FAKE + 2) == cq.CQSA_ERR_INVALID
    assert call(dtype=cq.CQSA_F32) == cq.CQSA_ERR_UNSUPPORTED


def test_bwd_chunk_validation(cq):
    L = cq.lib
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, lse=FAKE, dvec=FAKE, qo=0, ko=0, B=1, H=1, Nq=256, Nkv=256, d=64, c=1,
                s=0.0, dt=cq.CQSA_F16, dq=FAKE, dk=FAKE, dv=FAKE)

    def call(**kw):
        a = {**args, **kw}
        return L.cqsa_attn_bwd_chunk(a["q"], a["k"], a["v"], a["g"], a["lse"], a["dvec"], a["qo"], a["ko"], a["B"],
                                     a["H"], a["Nq"], a["Nkv"], a["d"], a["c"], a["s"], a["dt"], a["dq"], a["dk"],
                                     a["dv"], None)
    assert call(d=96) == cq.CQSA_ERR_UNSUPPORTED
    assert call(qo=-1) == cq.CQSA_ERR_INVALID
    assert call(dk=None) == cq.CQSA_ERR_INVALID
    assert call(dv=FAKE + 4) == cq.CQSA_ERR_INVALID
    assert call(Nkv=0) == cq.CQSA_ERR_INVALID
    assert L.cqsa_attn_bwd_dvec(FAKE, FAKE, FAKE, 1, 1, 128, 96, cq.CQSA_F16, None) == cq.CQSA_ERR_UNSUPPORTED
    assert L.cqsa_attn_bwd_dvec(FAKE, FAKE + 8, FAKE, 1, 1, 128, 64, cq.CQSA_F16, None) == cq.CQSA_ERR_INVALID
    assert L.cqsa_attn_bwd_cast(FAKE, FAKE, 6, cq.CQSA_F16, None) == cq.CQSA_ERR_INVALID
    assert L.cqsa_attn_bwd_cast(FAKE, FAKE, 8, cq.CQSA_F32, None) == cq.CQSA_ERR_UNSUPPORTED
    assert L.cqsa_attn_bwd_cast(FAKE, FAKE, 0, cq.CQSA_F16, None) == cq.CQSA_OK


def test_stream_bwd_validation(cq):
    L = cq.lib
    f = lambda **kw: L.cqsa_stream_attn_bwd(  # noqa: E731
        kw.get("q", FAKE), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, kw.get("N", 1000), kw.get("d", 64), 1,
        0.0, cq.CQSA_F16, kw.get("C", 256), None)
    assert f(C=100) == cq.CQSA_ERR_INVALID
    assert f(d=96) == cq.CQSA_ERR_UNSUPPORTED and "head dim" in cq.last_error()
    assert f(q=None) == cq.CQSA_ERR_INVALID
    assert f(N=0) == cq.CQSA_ERR_INVALID
