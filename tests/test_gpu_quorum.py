"""GPU parity of the quorum executor (cqsa_quorum_attn_fwd).

Every needed chunk pair is computed once and merged exactly, so the result must match the FP64
oracle within the stated tolerances, and match the streaming driver with the same chunk size (the same
chunk-pair partials merged in another order) to fp32 merge-order rounding.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._gpu import assert_bf16_rounds_fp32_result, assert_close, mono, to_dev, to_np64

pytestmark = pytest.mark.gpu

SETS = {3: (0, 1), 7: (0, 1, 3), 13: (0, 1, 3, 9)}


@pytest.fixture(scope="module")
def cq():
    import exact_long_context_tcgen05_gb300 as m
    return m


def _host(x, dtype):
    t = torch.from_numpy(x.view(np.int16))
    t = t.view(torch.float16 if dtype == syn.F16 else torch.bfloat16)
    return t.pin_memory()


def _oracle(qn, kn, vn, B, H, N, d, causal, dtype, layout):
    out, lse, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=N, d=d, causal=causal, dtype=dtype, layout=layout)
    return out.reshape(B, H, N, d), lse.reshape(B, H, N)


def _chunk_tokens(N, T):
    per = -(-N // T)
    return -(-per // 128) * 128


@pytest.mark.parametrize("c,itr,N,d,dtype,causal,layout,on_host", [
    (7, 1, 3000, 64, syn.F16, True, syn.LAYOUT_BHND, True),
    (7, 1, 3000, 64, syn.F16, False, syn.LAYOUT_BNHD, False),
    (3, 2, 2300, 64, syn.F16, True, syn.LAYOUT_BNHD, True),
    (13, 1, 4000, 128, syn.BF16, True, syn.LAYOUT_BHND, False),
    (3, 1, 1000, 128, syn.F16, False, syn.LAYOUT_BHND, True),
])
def test_quorum_vs_oracle_and_stream(cq, c, itr, N, d, dtype, causal, layout, on_host):
    B, H = 1, 2
    D = SETS[c]
    qn, kn, vn = syn.qkv(B, H, N, d, seed=c + itr, dtype=dtype, layout=layout)
    shape = (B, H, N, d) if layout == syn.LAYOUT_BHND else (B, N, H, d)
    tdt = torch.float16 if dtype == syn.F16 else torch.bfloat16
    if on_host:
        q, k, v = (_host(x, dtype) for x in (qn, kn, vn))
    else:
        q, k, v = (to_dev(x, dtype) for x in (qn, kn, vn))
    out = torch.empty(shape, dtype=tdt, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    st = cq.cqsa_quorum_stats()
    cq.cqsa_quorum_attn_fwd(q, k, v, layout, on_host, out, lse, False, B, H, N, d, causal, 0.0, dtype, c, D, itr,
                            stats=st)
    T = c ** itr
    C = _chunk_tokens(N, T)
    nne = -(-N // C)
    assert st.chunk_tokens == C
    assert st.n_pairs == (nne * (nne + 1) // 2 if causal else nne * nne)
    ro, rl = _oracle(qn, kn, vn, B, H, N, d, causal, dtype, layout)
    o64 = to_np64(out)
    if layout == syn.LAYOUT_BNHD:
        o64 = o64.transpose(0, 2, 1, 3)
    if dtype == syn.F16:
        assert_close(o64, ro, to_np64(lse), rl, what=f"quorum c={c} itr={itr}")
    else:
        # bf16 (the tolerance reading for bf16): the stated tolerances bind the fp32 result of the same
        # computation. The executor's fp32 accumulator stays inside the call, so the output is anchored
        # to the fp32 result over the whole key range (the chunk call): that result must meet the fp32
        # tolerances against the oracle, and the output must be the bf16 rounding of a value within the
        # chunked-vs-monolithic tolerance of it.
        assert layout == syn.LAYOUT_BHND
        qd, kd, vd = (to_dev(x, dtype) for x in (qn, kn, vn))
        O32 = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
        L32 = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        cq.cqsa_attn_fwd_chunk(qd, kd, vd, 0, 0, B, H, N, N, d, causal, 0.0, dtype, O32, L32, False)
        assert_close(to_np64(O32), ro, to_np64(L32), rl, what=f"quorum bf16 reference fp32 c={c}")
        assert_bf16_rounds_fp32_result(o64, to_np64(O32), f"quorum bf16 c={c}")
        lrel = np.abs(to_np64(lse) - to_np64(L32)) / np.maximum(1.0, np.abs(to_np64(L32)))
        assert lrel.max() <= 1e-5
    # the streaming driver's accumulating schedule with the same chunk size: same pair partials, merged
    # in key order (its resident schedule runs one launch per query chunk instead)
    hq, hk, hv = (_host(x, dtype) for x in (qn, kn, vn))
    out2 = torch.empty(shape, dtype=tdt, device="cuda")
    lse2 = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    cq.cqsa_set_stream_kv_resident_bytes(0)
    try:
        cq.cqsa_stream_attn_fwd(hq, hk, hv, layout, out2, lse2, False, B, H, N, d, causal, 0.0, dtype, C)
    finally:
        cq.cqsa_set_stream_kv_resident_bytes(-1)
    lrel = ((lse - lse2).abs() / lse2.abs().clamp_min(1.0)).max().item()
    assert lrel <= 1e-6, lrel
    diff = (out.float() - out2.float()).abs()
    tol = (out2.float().abs() * (2.0 ** -10 if dtype == syn.F16 else 2.0 ** -7)).clamp_min(2.0 ** -24)
    assert bool((diff <= tol).all()), "outputs differ by more than one ulp"


def test_quorum_host_output_and_itr_cost(cq):
    """Host output buffers; itr = 2 at c = 3: 9 subproblems, chunks staged once per subproblem need."""
    B, H, N, d = 1, 3, 2200, 64
    qn, kn, vn = syn.qkv(B, H, N, d, seed=5, layout=syn.LAYOUT_BNHD)
    q, k, v = (_host(x, syn.F16) for x in (qn, kn, vn))
    out = torch.empty((B, N, H, d), dtype=torch.float16).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    st = cq.cqsa_quorum_stats()
    cq.cqsa_quorum_attn_fwd(q, k, v, syn.LAYOUT_BNHD, True, out, lse, True, B, H, N, d, True, 0.0, syn.F16, 3, (0, 1),
                            2, stats=st)
    assert st.n_subproblems <= 9 and st.n_pairs == 45
    ro, rl = _oracle(qn, kn, vn, B, H, N, d, True, syn.F16, syn.LAYOUT_BNHD)
    assert_close(to_np64(out).transpose(0, 2, 1, 3), ro, to_np64(lse), rl, what="quorum host output")


def test_quorum_rejects_bad_set(cq):
    B, H, N, d = 1, 1, 256, 64
    x = torch.zeros((B, H, N, d), dtype=torch.float16, device="cuda")
    out = torch.empty_like(x)
    with pytest.raises(cq.CqsaError):
        cq.cqsa_quorum_attn_fwd(x, x, x, syn.LAYOUT_BHND, False, out, None, False, B, H, N, d, True, 0.0, syn.F16, 7,
                                (0, 1, 2), 1)


@pytest.mark.parametrize("c,itr,N,causal", [(7, 1, 5000, True), (3, 2, 2300, False), (13, 1, 6000, True)])
def test_host_accumulator_bitwise_equal(cq, c, itr, N, causal):
    """The host accumulator moves fp32 accumulators through pinned host memory unchanged, so the result
    equals the device-accumulator run bit for bit; it must actually spill (fewer slots than chunks)."""
    B, H, d = 1, 2, 64
    D = SETS[c]
    qn, kn, vn = syn.qkv(B, H, N, d, seed=17, layout=syn.LAYOUT_BNHD)
    q, k, v = (_host(x, syn.F16) for x in (qn, kn, vn))
    res = []
    for acc_on_host in (False, True):
        out = torch.empty((B, N, H, d), dtype=torch.float16, device="cuda")
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        st = cq.cqsa_quorum_stats()
        cq.cqsa_quorum_attn_fwd(q, k, v, syn.LAYOUT_BNHD, True, out, lse, False, B, H, N, d, causal, 0.0, syn.F16, c,
                                D, itr, acc_on_host=acc_on_host, stats=st)
        res.append((out, lse, st.acc_host_bytes, st.peak_device_bytes))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
    assert res[0][2] == 0 and res[1][2] > 0
    assert res[1][3] < res[0][3]
    ro, rl = _oracle(qn, kn, vn, B, H, N, d, causal, syn.F16, syn.LAYOUT_BNHD)
    assert_close(to_np64(res[1][0]).transpose(0, 2, 1, 3), ro, to_np64(res[1][1]), rl, what="host accumulator")


@pytest.mark.parametrize("npar", [2, 4])
def test_parallel_lanes_bitwise_equal(cq, npar):
    """Pairs of one query chunk stay in one lane in schedule order, so lanes change nothing bitwise."""
    B, H, N, d, c, D = 1, 2, 9000, 64, 13, (0, 1, 3, 9)
    qn, kn, vn = syn.qkv(B, H, N, d, seed=23)
    q, k, v = (to_dev(x, syn.F16) for x in (qn, kn, vn))
    res = []
    for p, acc_host in ((1, False), (npar, False), (npar, True)):
        out = torch.empty((B, H, N, d), dtype=torch.float16, device="cuda")
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        cq.cqsa_quorum_attn_fwd(q, k, v, syn.LAYOUT_BHND, False, out, lse, False, B, H, N, d, True, 0.0, syn.F16, c, D,
                                1, acc_on_host=acc_host, max_parallel=p)
        res.append((out, lse))
    for o, l in res[1:]:
        assert torch.equal(o, res[0][0]) and torch.equal(l, res[0][1])
    rows = syn.sample_rows(B, H, N, 256)
    ro, rl, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=N, d=d, causal=True, rows=rows)
    b, h, i = (torch.as_tensor(rows[:, j], device="cuda") for j in range(3))
    assert_close(to_np64(res[1][0][b, h, i]), ro, to_np64(res[1][1][b, h, i]), rl, what="parallel lanes")


@pytest.mark.parametrize("layout,on_host", [(syn.LAYOUT_BHND, False), (syn.LAYOUT_BHND, True), (syn.LAYOUT_BNHD, True)])
def test_quorum_batched_heads(cq, layout, on_host):
    """B = 2: chunk staging of strided [B,H,N,d] chunks (2-D copies) and of token-major chunks with B > 1."""
    B, H, N, d, c, D = 2, 3, 1800, 64, 7, (0, 1, 3)
    qn, kn, vn = syn.qkv(B, H, N, d, seed=29, layout=layout)
    shape = (B, H, N, d) if layout == syn.LAYOUT_BHND else (B, N, H, d)
    if on_host:
        q, k, v = (_host(x, syn.F16) for x in (qn, kn, vn))
    else:
        q, k, v = (to_dev(x, syn.F16) for x in (qn, kn, vn))
    out = torch.empty(shape, dtype=torch.float16).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    cq.cqsa_quorum_attn_fwd(q, k, v, layout, on_host, out, lse, True, B, H, N, d, True, 0.0, syn.F16, c, D, 1,
                            acc_on_host=True, max_parallel=3)
    ro, rl = _oracle(qn, kn, vn, B, H, N, d, True, syn.F16, layout)
    o64 = to_np64(out)
    if layout == syn.LAYOUT_BNHD:
        o64 = o64.transpose(0, 2, 1, 3)
    assert_close(o64, ro, to_np64(lse), rl, what="quorum B=2")


@pytest.mark.parametrize("c,itr,N,d,dtype,causal,layout,on_host,acc_host", [
    (7, 1, 3000, 64, syn.F16, True, syn.LAYOUT_BHND, False, False),
    (3, 2, 2300, 64, syn.F16, False, syn.LAYOUT_BNHD, True, False),
    (13, 1, 4000, 128, syn.BF16, True, syn.LAYOUT_BHND, False, True),
    (31, 1, 9000, 64, syn.F16, True, syn.LAYOUT_BNHD, True, True),
])
def test_wave_engine_equals_classic_and_oracle(cq, c, itr, N, d, dtype, causal, layout, on_host, acc_host):
    """The wave engine (one multi-pair launch per wave, at most one pair per query chunk). With host inputs
    it merges each query chunk's pairs in the classic engine's order, so the two agree bit for bit, also
    with a token budget of one chunk per launch. With device inputs read in place it runs each query
    chunk's adjacent key chunks as one key range: within one ulp of the classic engine, and, when every
    pair is in one group (no host accumulator), bitwise equal to the monolithic call (each query tile then
    meets the same key tiles in the same order). Against the oracle (fp16; bf16 through the classic test)."""
    B, H = 1, 2
    D = {3: (0, 1), 7: (0, 1, 3), 13: (0, 1, 3, 9), 31: (0, 1, 3, 8, 12, 18)}[c]
    qn, kn, vn = syn.qkv(B, H, N, d, seed=40 + c, dtype=dtype, layout=layout)
    shape = (B, H, N, d) if layout == syn.LAYOUT_BHND else (B, N, H, d)
    tdt = torch.float16 if dtype == syn.F16 else torch.bfloat16
    if on_host:
        q, k, v = (_host(x, dtype) for x in (qn, kn, vn))
    else:
        q, k, v = (to_dev(x, dtype) for x in (qn, kn, vn))
    res = []
    for engine, wt in ((cq.CQSA_ENGINE_CLASSIC, 0), (cq.CQSA_ENGINE_WAVE, 0), (cq.CQSA_ENGINE_WAVE, 1)):
        out = torch.empty(shape, dtype=tdt, device="cuda")
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        st = cq.cqsa_quorum_stats()
        cq.cqsa_quorum_attn_fwd_ex(q, k, v, layout, on_host, out, lse, False, B, H, N, d, causal, 0.0, dtype, c, D,
                                   itr, acc_on_host=acc_host, engine=engine, wave_tokens=wt, stats=st)
        res.append((out, lse, st.n_launches, st.n_pairs))
    for o, l_, nl, npairs in res[1:]:
        assert npairs == res[0][3]
        if on_host:
            assert torch.equal(o, res[0][0]) and torch.equal(l_, res[0][1])
        else:
            # one ulp of the element plus the fp32 merge's error relative to the row (an element that
            # cancels to near zero keeps the absolute error of its row)
            ref = res[0][0].float()
            rowmax = ref.abs().amax(dim=-1, keepdim=True)
            tol = ref.abs() * (2.0 ** -10 if dtype == syn.F16 else 2.0 ** -7) + 1e-5 * rowmax + 2.0 ** -24
            assert bool(((o.float() - ref).abs() <= tol).all())
            assert float(((l_ - res[0][1]).abs() / res[0][1].abs().clamp_min(1.0)).max()) <= 1e-6
    if on_host:
        # fewer launches than pairs with the default budget; one launch per pair with a one-token budget
        assert res[1][2] < res[0][2] and res[2][2] >= res[0][3]
    else:
        assert res[1][2] < res[0][2] and res[2][2] <= res[0][2]
        if not acc_host and layout == syn.LAYOUT_BHND:
            o_m, l_m = mono(cq, q, k, v, B, H, N, d, causal, dtype)
            assert torch.equal(res[1][0], o_m) and torch.equal(res[1][1], l_m)
    if dtype == syn.F16:
        ro, rl = _oracle(qn, kn, vn, B, H, N, d, causal, dtype, layout)
        o64 = to_np64(res[1][0])
        if layout == syn.LAYOUT_BNHD:
            o64 = o64.transpose(0, 2, 1, 3)
        assert_close(o64, ro, to_np64(res[1][1]), rl, what=f"wave engine c={c} itr={itr}")


def test_wave_engine_rejects_bad_engine(cq):
    x = torch.zeros((1, 1, 256, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(cq.CqsaError):
        cq.cqsa_quorum_attn_fwd_ex(x, x, x, syn.LAYOUT_BHND, False, torch.empty_like(x), None, False, 1, 1, 256, 64,
                                   True, 0.0, syn.F16, 7, (0, 1, 3), 1, engine=5)
