"""Pins for the CPU FP64 oracle: closed forms, invariants, brute force and chunk+merge exactness.

Each test checks the oracle against something other than itself (see the oracle's header), chosen
so that a dropped term, a wrong sign or index, or a transposed operand fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _f16(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def _problem(B, H, N, d, seed=0, dtype=syn.F16, k_mul=1.0):
    return syn.qkv(B, H, N, d, seed=seed, dtype=dtype, k_mul=k_mul)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [syn.F16, syn.BF16])
def test_normalisation_v_ones(causal, dtype):
    # softmax rows sum to one: with V = 1 every output is exactly the row's weight sum
    B, H, N, d = 1, 2, 200, 16
    q, k, _ = _problem(B, H, N, d, dtype=dtype, k_mul=3.0)
    one = 0x3C00 if dtype == syn.F16 else 0x3F80
    v = np.full_like(q, one)
    out, _ = oracle.attn_full(q, k, v, B=B, H=H, N=N, d=d, causal=causal, dtype=dtype)
    assert np.max(np.abs(out - 1.0)) < 1e-14


@pytest.mark.parametrize("dtype", [syn.F16, syn.BF16])
def test_causal_row0_is_v0(dtype):
    B, H, N, d = 2, 3, 64, 32
    q, k, v = _problem(B, H, N, d, dtype=dtype)
    out, lse = oracle.attn_full(q, k, v, B=B, H=H, N=N, d=d, causal=True, dtype=dtype)
    v0 = oracle.widen(v, dtype)[:, :, 0, :]
    assert np.array_equal(out[:, :, 0, :], v0)
    qd, kd = oracle.widen(q, dtype), oracle.widen(k, dtype)
    s00 = oracle.default_scale(d) * np.einsum("bhc,bhc->bh", qd[:, :, 0], kd[:, :, 0])
    assert np.max(np.abs(lse[:, :, 0] - s00)) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_give_mean(causal):
    B, H, N, d = 1, 2, 300, 8
    _, k, v = _problem(B, H, N, d)
    q = np.zeros_like(k)
    out, lse = oracle.attn_full(q, k, v, B=B, H=H, N=N, d=d, causal=causal)
    vd = oracle.widen(v)
    if causal:
        ref = np.cumsum(vd, axis=2) / np.arange(1, N + 1)[None, None, :, None]
        ref_lse = np.log(np.arange(1, N + 1, dtype=np.float64))[None, None, :]
    else:
        ref = np.broadcast_to(vd.mean(axis=2, keepdims=True), vd.shape)
        ref_lse = np.full((B, H, N), np.log(N))
    assert np.max(np.abs(out - ref)) < 1e-13
    assert np.max(np.abs(lse - ref_lse)) < 1e-13


def test_affine_in_v():
    # O(q, k, a v + b) = a O(q, k, v) + b because each row's weights sum to one
    B, H, N, d = 1, 1, 150, 8
    q, k, _ = _problem(B, H, N, d)
    rng = np.random.default_rng(5)
    vf = rng.integers(-32, 33, size=(B, H, N, d)) / 8.0       # exact in fp16
    v, v2 = _f16(vf), _f16(2.0 * vf + 0.75)
    for causal in (False, True):
        o1, l1 = oracle.attn_full(q, k, v, B=B, H=H, N=N, d=d, causal=causal)
        o2, l2 = oracle.attn_full(q, k, v2, B=B, H=H, N=N, d=d, causal=causal)
        assert np.max(np.abs(o2 - (2.0 * o1 + 0.75))) < 1e-12
        assert np.array_equal(l1, l2)


def test_permutation_equivariance():
    B, H, N, d = 1, 1, 97, 16
    q, k, v = _problem(B, H, N, d)
    out, lse = oracle.attn_full(q, k, v, B=B, H=H, N=N, d=d, causal=False)
    perm = np.random.default_rng(3).permutation(N)
    o_kv, l_kv = oracle.attn_full(q, k[:, :, perm], v[:, :, perm], B=B, H=H, N=N, d=d, causal=False)
    assert np.max(np.abs(o_kv - out)) < 1e-13 and np.max(np.abs(l_kv - lse)) < 1e-13
    o_q, l_q = oracle.attn_full(q[:, :, perm], k, v, B=B, H=H, N=N, d=d, causal=False)
    assert np.array_equal(o_q, out[:, :, perm]) and np.array_equal(l_q, lse[:, :, perm])


def test_two_key_closed_form():
    # N = 2, non-causal: O_0 = sigmoid(s00 - s01) v0 + sigmoid(s01 - s00) v1,
    # LSE_0 = s00 + log(1 + exp(s01 - s00))
    B, H, N, d = 1, 4, 2, 64
    q, k, v = _problem(B, H, N, d, seed=11)
    out, lse = oracle.attn_full(q, k, v, B=B, H=H, N=N, d=d, causal=False)
    qd, kd, vd = oracle.widen(q), oracle.widen(k), oracle.widen(v)
    sc = oracle.default_scale(d)
    for h in range(H):
        for i in range(2):
            s0 = sc * float(np.dot(qd[0, h, i], kd[0, h, 0]))
            s1 = sc * float(np.dot(qd[0, h, i], kd[0, h, 1]))
            w0 = 1.0 / (1.0 + np.exp(s1 - s0))
            w1 = 1.0 / (1.0 + np.exp(s0 - s1))
            assert np.max(np.abs(out[0, h, i] - (w0 * vd[0, h, 0] + w1 * vd[0, h, 1]))) < 1e-13
            assert abs(lse[0, h, i] - (s0 + np.log1p(np.exp(s1 - s0)))) < 1e-13


def _bf16_exact(x):
    """bfloat16 storage bits of values that bf16 represents exactly (the upper half of the fp32 bits)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (b >> 16).astype(np.uint16)


def test_golden_closed_forms():
    import sympy
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    ns = {"E": sympy.E, "exp": sympy.exp, "log": sympy.log, "Rational": sympy.Rational}
    assert any(c.get("dtype") == "bf16" for c in cases)
    for c in cases:
        B, H, N, d = c["B"], c["H"], c["N"], c["d"]
        bf = c.get("dtype", "f16") == "bf16"
        enc = _bf16_exact if bf else _f16
        q, k, v = (enc(np.array(c[t]).reshape(B, H, N, d)) for t in ("q", "k", "v"))
        if not bf:
            assert np.array_equal(q.view(np.float16).astype(np.float64), np.array(c["q"]).reshape(B, H, N, d))
        out, lse = oracle.attn_full(q, k, v, B=B, H=H, N=N, d=d, causal=c["causal"], scale=c["scale"],
                                    dtype=syn.BF16 if bf else syn.F16)
        for i in range(N):
            for j in range(d):
                ref = float(sympy.N(sympy.sympify(c["out"][i][j], locals=ns), 30))
                assert abs(out[0, 0, i, j] - ref) < 1e-14 * max(1.0, abs(ref)), (c["name"], i, j)
            ref = float(sympy.N(sympy.sympify(c["lse"][i], locals=ns), 30))
            assert abs(lse[0, 0, i] - ref) < 1e-14 * max(1.0, abs(ref)), (c["name"], i)


def _same_values(a, b):
    """Equal as float64 values, NaN matching NaN, and zeros matching in sign."""
    nan = np.isnan(a)
    if not np.array_equal(nan, np.isnan(b)):
        return False
    a, b = a[~nan], b[~nan]
    return np.array_equal(a, b) and np.array_equal(np.signbit(a), np.signbit(b))


def test_widening_every_fp16_pattern():
    # all 65,536 binary16 patterns (normals, subnormals, +-0, +-inf, NaNs) against numpy's float16
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    assert _same_values(oracle.widen(bits, syn.F16), ref)


def test_widening_every_bf16_pattern():
    # all 65,536 bfloat16 patterns against two independent routes: the pattern placed in the upper half
    # of a binary32 (bfloat16's definition), and torch's bfloat16 dtype
    import torch
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen to NaN
        via_f32 = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    via_torch = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.widen(bits, syn.BF16)
    assert _same_values(got, via_f32)
    assert _same_values(got, via_torch)
    # spot values: smallest subnormal, largest subnormal, 1 + 2^-7, -(1/2 + 2^-7), largest finite
    spots = {0x0001: 2.0 ** -133, 0x007F: 127 * 2.0 ** -133, 0x3F81: 1 + 2.0 ** -7, 0xBF02: -(0.5 + 2.0 ** -7),
             0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127}
    for b, val in spots.items():
        assert got[b] == val, hex(b)


@pytest.mark.parametrize("dtype", [syn.F16, syn.BF16])
@pytest.mark.parametrize("causal", [False, True])
def test_bruteforce_tiny(dtype, causal):
    for (B, H, N, d) in [(1, 1, 1, 1), (1, 2, 3, 2), (2, 1, 7, 4), (1, 3, 16, 8), (2, 2, 13, 6)]:
        for seed in range(3):
            q, k, v = _problem(B, H, N, d, seed=seed, dtype=dtype)
            o1, l1 = oracle.attn_full(q, k, v, B=B, H=H, N=N, d=d, causal=causal, dtype=dtype)
            o2, l2 = oracle.bruteforce_ld(q, k, v, B=B, H=H, N=N, d=d, causal=causal, dtype=dtype)
            assert np.max(np.abs(o1 - o2)) < 1e-13
            assert np.max(np.abs(l1 - l2)) < 1e-13


def test_token_major_layout_same_values():
    B, H, N, d = 2, 3, 70, 8
    q, k, v = syn.qkv(B, H, N, d, seed=4)
    qt, kt, vt = syn.qkv(B, H, N, d, seed=4, layout=syn.LAYOUT_BNHD)
    o1, l1, _ = oracle.attn_rows(q, k, v, B=B, H=H, Nq=N, d=d, causal=True)
    o2, l2, _ = oracle.attn_rows(qt, kt, vt, B=B, H=H, Nq=N, d=d, causal=True, layout=oracle.LAYOUT_BNHD)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def _chunked(q, k, v, B, H, N, d, causal, q_cuts, kv_cuts):
    """Full result assembled from chunk-pair partials and the FP64 merge."""
    out = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    for qa, qb in zip(q_cuts[:-1], q_cuts[1:]):
        parts_o, parts_l = [], []
        for ka, kb in zip(kv_cuts[:-1], kv_cuts[1:]):
            o, l_, _ = oracle.attn_rows(np.ascontiguousarray(q[:, :, qa:qb]), np.ascontiguousarray(k[:, :, ka:kb]),
                                        np.ascontiguousarray(v[:, :, ka:kb]), B=B, H=H, Nq=qb - qa, Nkv=kb - ka,
                                        d=d, causal=causal, q_off=qa, kv_off=ka)
            parts_o.append(o.reshape(B, H, qb - qa, d))
            parts_l.append(l_.reshape(B, H, qb - qa))
        mo, ml = oracle.merge(parts_o, parts_l)
        out[:, :, qa:qb], lse[:, :, qa:qb] = mo, ml
    return out, lse


@pytest.mark.parametrize("causal", [False, True])
def test_chunk_merge_equals_monolithic(causal):
    B, H, N, d = 1, 2, 61, 8
    q, k, v = _problem(B, H, N, d, seed=2, k_mul=3.0)
    mono_o, mono_l = oracle.attn_full(q, k, v, B=B, H=H, N=N, d=d, causal=causal)
    rng = np.random.default_rng(0)
    partitions = [[0, N], [0, 1, N], [0, 30, 31, 61], list(range(0, N + 1))]
    for _ in range(6):
        cuts = sorted(set(rng.integers(1, N, size=rng.integers(1, 8)).tolist()))
        partitions.append([0, *cuts, N])
    for qc in partitions:
        for kc in partitions:
            o, l_ = _chunked(q, k, v, B, H, N, d, causal, qc, kc)
            rel = np.max(np.abs(o - mono_o)) / np.max(np.abs(mono_o))
            assert rel < 1e-12, (qc, kc)
            assert np.max(np.abs(l_ - mono_l) / np.maximum(1, np.abs(mono_l))) < 1e-12


def test_empty_pairs_and_merge_edge_cases():
    B, H, d = 1, 1, 4
    q, k, v = _problem(B, H, 32, d, seed=9)
    # a causal pair entirely above the diagonal: queries 0..15, keys 16..31
    o, l_, _ = oracle.attn_rows(np.ascontiguousarray(q[:, :, :16]), np.ascontiguousarray(k[:, :, 16:]),
                                np.ascontiguousarray(v[:, :, 16:]), B=B, H=H, Nq=16, Nkv=16, d=d, causal=True,
                                q_off=0, kv_off=16)
    assert np.all(o == 0) and np.all(l_ == -np.inf)
    # Nkv = 0
    o, l_, _ = oracle.attn_rows(q, k[:, :, :0], v[:, :, :0], B=B, H=H, Nq=32, Nkv=0, d=d, causal=False)
    assert np.all(o == 0) and np.all(l_ == -np.inf)
    # merging with an empty part changes nothing; all-empty gives 0 / -inf
    rng = np.random.default_rng(1)
    O1, L1 = rng.normal(size=(5, d)), rng.normal(size=5)
    Oe, Le = np.zeros((5, d)), np.full(5, -np.inf)
    mo, ml = oracle.merge([O1, Oe], [L1, Le])
    assert np.max(np.abs(mo - O1)) < 1e-15 and np.max(np.abs(ml - L1)) < 1e-15
    mo, ml = oracle.merge([Oe, Oe], [Le, Le])
    assert np.all(mo == 0) and np.all(ml == -np.inf)


def test_merge_two_equal_weight_parts():
    # two parts with equal LSE: the merged output is their mean and lse rises by ln 2
    rng = np.random.default_rng(2)
    O1, O2 = rng.normal(size=(7, 3)), rng.normal(size=(7, 3))
    L = rng.normal(size=7)
    mo, ml = oracle.merge([O1, O2], [L, L])
    assert np.max(np.abs(mo - (O1 + O2) / 2)) < 1e-15
    assert np.max(np.abs(ml - (L + np.log(2)))) < 1e-14


def test_bad_arguments_rejected():
    q, k, v = _problem(1, 1, 8, 4)
    with pytest.raises(ValueError):
        oracle.attn_rows(q, k, v, B=1, H=1, Nq=8, d=4, causal=False, rows=np.array([[0, 0, 8]]))
    with pytest.raises(TypeError):
        oracle.attn_rows(q.astype(np.float32), k, v, B=1, H=1, Nq=8, d=4, causal=False)
