"""Pins of the oracle's attention backward (CPU, no GPU): its gradients against central finite
differences of the loss sum(dO * O), its forward part against the forward oracle, the key-shift
invariance sum_j dK_j = 0, and the uniform-score closed forms of dV and dK."""
import numpy as np
import pytest

import oracle
import synthetic as syn


def _loss(q, k, v, g, causal, scale):
    return float(np.sum(g * oracle.attn_bwd_f64(q, k, v, g, causal=causal, scale=scale)["out"]))


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_differences(causal):
    """dq, dk, dv are the derivatives of L = sum(dO * O): a dropped softmax term, a wrong sign or a
    transposed operand in any of them moves it far beyond the difference quotient's error (~1e-9)."""
    rng = np.random.default_rng(11 + int(causal))
    B, H, N, d = 1, 2, 7, 3
    q, k, v, g = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 0.7
    res = oracle.attn_bwd_f64(q, k, v, g, causal=causal, scale=scale)
    h = 1e-5
    for name, pos in (("dq", 0), ("dk", 1), ("dv", 2)):
        base = [q, k, v]
        fd = np.empty_like(q)
        for idx in np.ndindex(q.shape):
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[pos][idx] += h
            minus[pos][idx] -= h
            fd[idx] = (_loss(*plus, g, causal, scale) - _loss(*minus, g, causal, scale)) / (2 * h)
        np.testing.assert_allclose(res[name], fd, rtol=1e-6, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_part_matches_forward_oracle(causal):
    B, H, N, d = 1, 2, 40, 16
    q, k, v = syn.qkv(B, H, N, d, seed=3)
    g = syn.normal(B, H, N, d, seed=3, tensor_id=syn.TID_DO)
    res = oracle.attn_bwd(q, k, v, g, B=B, H=H, N=N, d=d, causal=causal)
    o, lse = oracle.attn_full(q, k, v, B=B, H=H, N=N, d=d, causal=causal)
    np.testing.assert_allclose(res["out"], o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(res["lse"], lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    """Adding one vector to every key adds the same amount to each score of a row, which the
    softmax ignores: the loss is flat along that direction, so the key gradients sum to zero."""
    B, H, N, d = 2, 1, 33, 8
    q, k, v = syn.qkv(B, H, N, d, seed=5)
    g = syn.normal(B, H, N, d, seed=5, tensor_id=syn.TID_DO)
    res = oracle.attn_bwd(q, k, v, g, B=B, H=H, N=N, d=d, causal=causal)
    tot = np.abs(res["dk"]).sum(axis=2)
    assert np.all(np.abs(res["dk"].sum(axis=2)) <= 1e-13 * np.maximum(tot, 1.0))


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_closed_form(causal):
    """q = 0 makes every allowed score 0: P_ij = 1/|A_i|, so dV_j = sum over the rows i that see key
    j of dO_i / |A_i|, and dK = scale * sum_i dS_ij q_i vanishes exactly."""
    B, H, N, d = 1, 2, 24, 8
    _, k, v = syn.qkv(B, H, N, d, seed=9)
    q = np.zeros_like(k)
    g = syn.normal(B, H, N, d, seed=9, tensor_id=syn.TID_DO)
    res = oracle.attn_bwd(q, k, v, g, B=B, H=H, N=N, d=d, causal=causal)
    gd = oracle.widen(g).reshape(B, H, N, d)
    want = np.zeros((B, H, N, d))
    for j in range(N):
        for i in range(N):
            if not causal or j <= i:
                want[:, :, j] += gd[:, :, i] / ((i + 1) if causal else N)
    np.testing.assert_allclose(res["dv"], want, rtol=1e-13, atol=1e-14)
    assert np.all(res["dk"] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_symbolic_gradient_tiny(causal):
    """N = 3, d = 2: the loss sum(dO * O) written out with sympy from the definition of attention
    and differentiated symbolically; its gradients, evaluated at the same point, pin every element
    of dq, dk and dv independently of the oracle's formulas."""
    sp = pytest.importorskip("sympy")
    N, d, scale = 3, 2, 0.6
    rng = np.random.default_rng(21 + int(causal))
    vals = {n: rng.standard_normal((N, d)) for n in ("q", "k", "v", "g")}
    sym = {n: sp.Matrix(N, d, lambda i, c, n=n: sp.Symbol(f"{n}{i}{c}")) for n in ("q", "k", "v")}
    loss = 0
    for i in range(N):
        keys = range(i + 1) if causal else range(N)
        e = {j: sp.exp(scale * sum(sym["q"][i, c] * sym["k"][j, c] for c in range(d))) for j in keys}
        z = sum(e.values())
        for c in range(d):
            o_ic = sum(e[j] * sym["v"][j, c] for j in keys) / z
            loss += vals["g"][i, c] * o_ic
    subs = {sym[n][i, c]: vals[n][i, c] for n in ("q", "k", "v") for i in range(N) for c in range(d)}
    res = oracle.attn_bwd_f64(*(vals[n][None, None] for n in ("q", "k", "v", "g")), causal=causal, scale=scale)
    for n, name in (("q", "dq"), ("k", "dk"), ("v", "dv")):
        want = np.array([[float(sp.diff(loss, sym[n][i, c]).evalf(subs=subs, n=30)) for c in range(d)]
                         for i in range(N)])
        np.testing.assert_allclose(res[name][0, 0], want, rtol=1e-12, atol=1e-13, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [syn.F16, syn.BF16])
def test_sampled_rows_and_columns_match_full_backward(causal, dtype):
    """attn_bwd_rows / attn_bwd_cols (for problems too large for the full N x N oracle) agree with the
    full oracle backward, which the other tests here pin, at every row and column of a small problem."""
    B, H, N, d = 2, 2, 150, 16
    q, k, v = syn.qkv(B, H, N, d, seed=8, dtype=dtype, k_mul=2.0)
    g = syn.normal(B, H, N, d, seed=8, tensor_id=syn.TID_DO, dtype=dtype)
    ref = oracle.attn_bwd(q, k, v, g, B=B, H=H, N=N, d=d, causal=causal, dtype=dtype)
    bb, hh, ii = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), indexing="ij")
    idx = np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1)
    perm = np.random.default_rng(1).permutation(len(idx))  # any order of the listed triples
    idx = idx[perm]
    dq = oracle.attn_bwd_rows(q, k, v, g, B=B, H=H, N=N, d=d, causal=causal, rows=idx, dtype=dtype)
    dk, dv = oracle.attn_bwd_cols(q, k, v, g, B=B, H=H, N=N, d=d, causal=causal, cols=idx, dtype=dtype)
    sel = (idx[:, 0], idx[:, 1], idx[:, 2])
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        r = ref[name][sel]
        assert np.max(np.abs(got - r)) <= 1e-12 * max(1.0, np.abs(r).max()), name
    # a subset of one head only evaluates that head's rows
    sub = idx[(idx[:, 0] == 1) & (idx[:, 1] == 0)][:7]
    dk1, dv1 = oracle.attn_bwd_cols(q, k, v, g, B=B, H=H, N=N, d=d, causal=causal, cols=sub, dtype=dtype)
    s1 = (sub[:, 0], sub[:, 1], sub[:, 2])
    assert np.max(np.abs(dk1 - ref["dk"][s1])) <= 1e-12 * max(1.0, np.abs(ref["dk"]).max())
    assert np.max(np.abs(dv1 - ref["dv"][s1])) <= 1e-12 * max(1.0, np.abs(ref["dv"]).max())


def test_sampled_backward_rejects_bad_indices():
    q, k, v = syn.qkv(1, 1, 8, 4, seed=0)
    with pytest.raises(ValueError):
        oracle.attn_bwd_rows(q, k, v, q, B=1, H=1, N=8, d=4, causal=True, rows=np.array([[0, 0, 8]]))
    with pytest.raises(ValueError):
        oracle.attn_bwd_cols(q, k, v, q, B=1, H=1, N=8, d=4, causal=True, cols=np.array([[0, 1, 0]]))
