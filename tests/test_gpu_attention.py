"""GPU parity: the CUDA path through the C ABI against the FP64 oracle on the same seeded inputs.

Tolerances (stated by the workload definition for fp16/bf16 outputs): max abs <= 4e-3, mean abs
<= 2e-4, LSE within 1e-3 absolute; chunked vs monolithic fp32 results within 1e-5 relative (per
row, relative to the row's largest |O|). For bf16 the stated output tolerance is below bf16's own
rounding of the result, so it is applied to the fp32 result of the same computation, and the bf16
output must equal that fp32 result rounded to nearest even and lie within one bf16 ulp of the
rounded oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._gpu import assert_close, chunk, errs, mono, to_dev, to_np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cq():
    import exact_long_context_tcgen05_gb300 as m
    return m


def _inputs(B, H, N, d, dtype, seed=0, k_mul=1.0):
    qn, kn, vn = syn.qkv(B, H, N, d, seed=seed, dtype=dtype, k_mul=k_mul)
    return (qn, kn, vn), tuple(to_dev(x, dtype) for x in (qn, kn, vn))


def _bf16_rne(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def _bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def test_config_small_all_rows(cq):
    """B=1, H=2, N=1024, d=64, fp16 N(0,1) seed 0, causal, scale 1/sqrt(64): every row."""
    B, H, N, d = 1, 2, 1024, 64
    (qn, kn, vn), (q, k, v) = _inputs(B, H, N, d, syn.F16)
    out, lse = mono(cq, q, k, v, B, H, N, d, True, syn.F16)
    ref_o, ref_l = oracle.attn_full(qn, kn, vn, B=B, H=H, N=N, d=d, causal=True)
    mx, mn = assert_close(to_np64(out), ref_o, to_np64(lse), ref_l, what="config small")
    print(f"\nconfig small: max abs {mx:.3e} mean abs {mn:.3e}")


@pytest.mark.parametrize("N", [1, 127, 129, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [syn.F16, syn.BF16])
@pytest.mark.parametrize("causal", [True, False])
def test_shapes_and_tails(cq, N, d, dtype, causal):
    B, H = 1, 2
    (qn, kn, vn), (q, k, v) = _inputs(B, H, N, d, dtype, seed=N + d)
    out, lse = mono(cq, q, k, v, B, H, N, d, causal, dtype)
    ref_o, ref_l = oracle.attn_full(qn, kn, vn, B=B, H=H, N=N, d=d, causal=causal, dtype=dtype)
    if dtype == syn.F16:
        assert_close(to_np64(out), ref_o, to_np64(lse), ref_l, what="fp16 out")
        return
    # bf16: fp32 result of the same computation (chunk over the whole range) against the oracle
    O, L = chunk(cq, q, k, v, 0, 0, B, H, N, N, d, causal, dtype)
    o32 = to_np64(O)
    assert_close(o32, ref_o, to_np64(L), ref_l, what="bf16 fp32 result")
    got = to_np64(out)
    assert np.array_equal(got, _bf16_rne(O.cpu().numpy())), "bf16 output is not RNE of the fp32 result"
    # hence |out - oracle| <= half a bf16 ulp of out + the fp32 result's own error (a plain "one ulp of
    # the rounded oracle" cannot hold for outputs near zero, where the fp32 error exceeds a bf16 ulp)
    assert np.all(np.abs(got - ref_o) <= 0.5 * _bf16_ulp(got) + np.abs(o32 - ref_o) + 1e-12)
    assert np.array_equal(to_np64(lse), to_np64(L))


def test_causal_row0_and_uniform_scores(cq):
    B, H, N, d = 1, 2, 700, 64
    (qn, kn, vn), (q, k, v) = _inputs(B, H, N, d, syn.F16, seed=3)
    out, lse = mono(cq, q, k, v, B, H, N, d, True, syn.F16)
    # causal row 0 attends to key 0 only: O_0 = v_0 bit for bit
    assert torch.equal(out[:, :, 0], v[:, :, 0])
    # Q = 0: every allowed key has weight 1/(i+1): O_i = mean of v_0..v_i, LSE_i = ln(i+1)
    qz = torch.zeros_like(q)
    out, lse = mono(cq, qz, k, v, B, H, N, d, True, syn.F16)
    vd = oracle.widen(vn)
    ref = np.cumsum(vd, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    assert_close(to_np64(out), ref, what="uniform scores")
    assert np.max(np.abs(to_np64(lse) - np.log(np.arange(1, N + 1))[None, None, :])) < 1e-5


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("q_off,kv_off", [(0, 0), (500, 0), (0, 500), (256, 128), (100, 37), (131, 300)])
def test_chunk_pairs_vs_oracle(cq, d, causal, q_off, kv_off):
    B, H = 1, 2
    Nq, Nkv = 300, 200
    qn = syn.normal(B, H, Nq, d, seed=5, tensor_id=0)
    kn = syn.normal(B, H, Nkv, d, seed=5, tensor_id=1)
    vn = syn.normal(B, H, Nkv, d, seed=5, tensor_id=2)
    q, k, v = (to_dev(x, syn.F16) for x in (qn, kn, vn))
    O, L = chunk(cq, q, k, v, q_off, kv_off, B, H, Nq, Nkv, d, causal, syn.F16)
    ro, rl, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=Nq, Nkv=Nkv, d=d, causal=causal, q_off=q_off, kv_off=kv_off)
    ro, rl = ro.reshape(B, H, Nq, d), rl.reshape(B, H, Nq)
    o, l_ = to_np64(O), to_np64(L)
    empty = ~np.isfinite(rl)
    assert np.all(o[empty] == 0.0) and np.all(l_[empty] == -np.inf)
    assert_close(o, ro, l_, rl, what=f"chunk pair ({q_off},{kv_off})")


@pytest.mark.parametrize("d,dtype", [(64, syn.F16), (128, syn.F16), (128, syn.BF16)])
def test_accumulate_modes(cq, d, dtype):
    """Accumulate onto an empty accumulator equals the partial result bit for bit; accumulating a
    second key block gives the oracle result over the union of the two blocks."""
    B, H, Nq, Nkv = 1, 2, 260, 200
    qn = syn.normal(B, H, Nq, d, seed=6, tensor_id=0, dtype=dtype)
    kn = syn.normal(B, H, 2 * Nkv, d, seed=6, tensor_id=1, dtype=dtype)
    vn = syn.normal(B, H, 2 * Nkv, d, seed=6, tensor_id=2, dtype=dtype)
    q, k, v = (to_dev(x, dtype) for x in (qn, kn, vn))
    k1, k2 = k[:, :, :Nkv].contiguous(), k[:, :, Nkv:].contiguous()
    v1, v2 = v[:, :, :Nkv].contiguous(), v[:, :, Nkv:].contiguous()
    for causal, q_off in ((False, 0), (True, 150)):
        Op, Lp = chunk(cq, q, k1, v1, q_off, 0, B, H, Nq, Nkv, d, causal, dtype)
        Oa = torch.full((B, H, Nq, d), float("nan"), device="cuda")
        La = torch.full((B, H, Nq), -float("inf"), device="cuda")
        chunk(cq, q, k1, v1, q_off, 0, B, H, Nq, Nkv, d, causal, dtype, O=Oa, L=La, accumulate=True)
        fin = torch.isfinite(Lp)
        assert torch.equal(La, Lp)
        assert torch.equal(Oa[fin], Op[fin])
        chunk(cq, q, k2, v2, q_off, Nkv, B, H, Nq, Nkv, d, causal, dtype, O=Oa, L=La, accumulate=True)
        ro, rl, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=Nq, Nkv=2 * Nkv, d=d, causal=causal, q_off=q_off,
                                     kv_off=0, dtype=dtype)
        ro, rl = ro.reshape(B, H, Nq, d), rl.reshape(B, H, Nq)
        o = to_np64(Oa)
        o[~np.isfinite(rl)] = 0.0
        assert_close(o, ro, to_np64(La), rl, what=f"accumulate d={d} causal={causal}")


def test_empty_kv_block(cq):
    B, H, Nq, d = 1, 1, 130, 64
    q = to_dev(syn.normal(B, H, Nq, d), syn.F16)
    O, L = chunk(cq, q, None, None, 0, 0, B, H, Nq, 0, d, False, syn.F16)
    assert torch.all(O == 0) and torch.all(L == -float("inf"))


def _row_rel(a, b):
    """max over rows of max_c |a-b| / max_c |b|, plus LSE differences relative to max(1, |lse|)."""
    den = np.maximum(np.abs(b).max(axis=-1), 1e-30)
    return float((np.abs(a - b).max(axis=-1) / den).max())


@pytest.mark.parametrize("d,dtype", [(64, syn.F16), (128, syn.BF16), (64, syn.BF16), (128, syn.F16)])
@pytest.mark.parametrize("causal", [True, False])
def test_chunked_equals_monolithic_fp32(cq, d, dtype, causal):
    B, H, N, C = 1, 2, 1024, 256
    (qn, kn, vn), (q, k, v) = _inputs(B, H, N, d, dtype, seed=7, k_mul=3.0 if dtype == syn.BF16 else 1.0)
    Om, Lm = chunk(cq, q, k, v, 0, 0, B, H, N, N, d, causal, dtype)
    om, lm = to_np64(Om), to_np64(Lm)
    nch = N // C
    out_merge = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    lse_merge = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    for i in range(nch):
        qs = q[:, :, i * C:(i + 1) * C].contiguous()
        parts_o, parts_l = [], []
        Oa = torch.empty((B, H, C, d), dtype=torch.float32, device="cuda")
        La = torch.empty((B, H, C), dtype=torch.float32, device="cuda")
        js = range(i + 1) if causal else range(nch)
        for t, j in enumerate(js):
            ks = k[:, :, j * C:(j + 1) * C].contiguous()
            vs = v[:, :, j * C:(j + 1) * C].contiguous()
            Op, Lp = chunk(cq, qs, ks, vs, i * C, j * C, B, H, C, C, d, causal, dtype)
            parts_o.append(Op)
            parts_l.append(Lp)
            chunk(cq, qs, ks, vs, i * C, j * C, B, H, C, C, d, causal, dtype, O=Oa, L=La, accumulate=(t > 0))
        om_i = torch.empty((B, H, C, d), dtype=torch.float32, device="cuda")
        lm_i = torch.empty((B, H, C), dtype=torch.float32, device="cuda")
        cq.cqsa_merge_partials(parts_o, parts_l, len(parts_o), om_i, lm_i, B, H, C, d, cq.CQSA_F32)
        out_merge[:, :, i * C:(i + 1) * C] = om_i
        lse_merge[:, :, i * C:(i + 1) * C] = lm_i
        ref = om[:, :, i * C:(i + 1) * C]
        rl = lm[:, :, i * C:(i + 1) * C]
        for name, o_, l_ in (("accumulate", Oa, La), ("merge", om_i, lm_i)):
            rel = _row_rel(to_np64(o_), ref)
            lrel = float((np.abs(to_np64(l_) - rl) / np.maximum(1.0, np.abs(rl))).max())
            assert rel <= 1e-5 and lrel <= 1e-5, f"{name} chunk {i}: rel {rel:.2e}, lse rel {lrel:.2e}"
    # and the merged whole against the oracle (fp32 result)
    ref_o, ref_l = oracle.attn_full(qn, kn, vn, B=B, H=H, N=N, d=d, causal=causal, dtype=dtype)
    assert_close(to_np64(out_merge), ref_o, to_np64(lse_merge), ref_l, what="merged vs oracle")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 2, 17, 130])
def test_merge_kernel_vs_oracle(cq, d, n):
    B, H, Nq = 1, 3, 97
    rng = np.random.default_rng(n * 1000 + d)
    Os = [rng.normal(size=(B, H, Nq, d)).astype(np.float32) for _ in range(n)]
    Ls = [(rng.normal(size=(B, H, Nq)) * 5).astype(np.float32) for _ in range(n)]
    for L_ in Ls[::2]:
        L_[0, 0, rng.integers(0, Nq, size=10)] = -np.inf
    if n > 1:
        for L_ in Ls:
            L_[0, 1, 5] = -np.inf  # a row where every part is empty
    ref_o, ref_l = oracle.merge([o.astype(np.float64) for o in Os], [l_.astype(np.float64) for l_ in Ls])
    dO = [torch.from_numpy(o).cuda() for o in Os]
    dL = [torch.from_numpy(l_).cuda() for l_ in Ls]
    for odt, tdt in ((cq.CQSA_F32, torch.float32), (cq.CQSA_F16, torch.float16), (cq.CQSA_BF16, torch.bfloat16)):
        out = torch.empty((B, H, Nq, d), dtype=tdt, device="cuda")
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
        cq.cqsa_merge_partials(dO, dL, n, out, lse, B, H, Nq, d, odt)
        o, l_ = to_np64(out), to_np64(lse)
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(l_), fin)
        assert np.max(np.abs(l_[fin] - ref_l[fin])) <= 1e-5 * max(1.0, np.abs(ref_l[fin]).max())
        scale = np.abs(ref_o).max()
        tol = {torch.float32: 2e-6, torch.float16: 2.0 ** -10, torch.bfloat16: 2.0 ** -7}[tdt]
        assert np.max(np.abs(o - ref_o)) <= tol * scale, (odt, np.max(np.abs(o - ref_o)))
        assert np.all(o[~fin] == 0)


def test_determinism(cq):
    B, H, N, d = 1, 4, 2048, 64
    _, (q, k, v) = _inputs(B, H, N, d, syn.F16, seed=9)
    o1, l1 = mono(cq, q, k, v, B, H, N, d, True, syn.F16)
    o2, l2 = mono(cq, q, k, v, B, H, N, d, True, syn.F16)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("layout", [syn.LAYOUT_BNHD, syn.LAYOUT_BHND])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("out_on_host", [True, False])
@pytest.mark.parametrize("resident", [True, False])
def test_stream_driver_small(cq, layout, causal, out_on_host, resident):
    """Both schedules of the host-streaming driver against the oracle: K/V resident (one launch per Q chunk
    over its key prefix) and every (Q chunk, KV chunk) pair through the fp32 accumulator."""
    B, H, N, d, C = 2, 3, 1000, 64, 256
    qn, kn, vn = syn.qkv(B, H, N, d, seed=11, layout=layout)
    hq, hk, hv = (torch.from_numpy(x.view(np.int16)).view(torch.float16).pin_memory() for x in (qn, kn, vn))
    shape = (B, H, N, d) if layout == syn.LAYOUT_BHND else (B, N, H, d)
    if out_on_host:
        out = torch.empty(shape, dtype=torch.float16).pin_memory()
        lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    else:
        out = torch.empty(shape, dtype=torch.float16, device="cuda")
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    st = cq.cqsa_stream_stats()
    cq.cqsa_set_stream_kv_resident_bytes(1 << 40 if resident else 0)
    try:
        cq.cqsa_stream_attn_fwd(hq, hk, hv, layout, out, lse, out_on_host, B, H, N, d, causal, 0.0, cq.CQSA_F16, C,
                                st)
    finally:
        cq.cqsa_set_stream_kv_resident_bytes(-1)
    if resident and layout == syn.LAYOUT_BHND:
        # the same tiles, key order and fold segments as the monolithic call: bitwise equal
        q, k, v = (to_dev(x, syn.F16) for x in (qn, kn, vn))
        o_m, l_m = mono(cq, q, k, v, B, H, N, d, causal, syn.F16)
        assert torch.equal(out.cuda(), o_m) and torch.equal(lse.cuda(), l_m)
    o = to_np64(out)
    if layout == syn.LAYOUT_BNHD:
        o = o.transpose(0, 2, 1, 3)
        qb, kb, vb = (np.ascontiguousarray(x.transpose(0, 2, 1, 3)) for x in (qn, kn, vn))
    else:
        qb, kb, vb = qn, kn, vn
    ref_o, ref_l = oracle.attn_full(qb, kb, vb, B=B, H=H, N=N, d=d, causal=causal)
    assert_close(o, ref_o, to_np64(lse), ref_l, what="stream driver")
    nq = (N + C - 1) // C
    assert st.n_chunks == (nq if resident else (nq * (nq + 1) // 2 if causal else nq * nq))
    assert st.h2d_bytes >= 3 * B * H * N * d * 2 and st.peak_device_bytes > 0
    if out_on_host:
        assert st.d2h_bytes == B * H * N * d * 2 + B * H * N * 4


def test_no_device_error(cq):
    rc, code, _ = cq.cqsa_device_error()
    assert rc == cq.CQSA_OK and code == 0
