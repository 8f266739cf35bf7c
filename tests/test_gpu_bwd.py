"""GPU parity of the attention backward (cqsa_attn_bwd) against the FP64 oracle backward.

The GPU forward supplies out and lse, as a caller's forward would; the oracle recomputes everything
from q, k, v and dout in double. Tolerance, per gradient tensor, from the arithmetic: the result is
rounded to the input dtype (relative half-ulp u = 2^-11 for fp16, 2^-8 for bf16), and P and dS enter
the tensor-core products rounded to the same dtype (one more relative error <= u per term, mostly
averaging out over the sums); D uses the rounded forward output. So the largest error is held to
8u of the tensor's largest |value| and the mean error to u of its mean |value|.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._gpu import mono, to_dev, to_np64

pytestmark = pytest.mark.gpu

U = {syn.F16: 2.0 ** -11, syn.BF16: 2.0 ** -8}


@pytest.fixture(scope="module")
def cq():
    import exact_long_context_tcgen05_gb300 as m
    return m


def _run(cq, B, H, N, d, causal, dtype, seed=0, q_zero=False):
    qn, kn, vn = syn.qkv(B, H, N, d, seed=seed, dtype=dtype)
    if q_zero:
        qn = np.zeros_like(qn)
    gn = syn.normal(B, H, N, d, seed=seed, tensor_id=syn.TID_DO, dtype=dtype)
    q, k, v, g = (to_dev(x, dtype) for x in (qn, kn, vn, gn))
    out, lse = mono(cq, q, k, v, B, H, N, d, causal, dtype)
    dq, dk, dv = cq.attention_backward(q, k, v, out, g, lse, causal=causal)
    torch.cuda.synchronize()
    rc, code, _ = cq.cqsa_device_error()
    assert rc == cq.CQSA_OK and code == 0
    return (qn, kn, vn, gn), (dq, dk, dv)


def _check(got: np.ndarray, ref: np.ndarray, dtype, what):
    u = U[dtype]
    e = np.abs(got - ref)
    mx, mn = float(e.max()), float(e.mean())
    ref_max, ref_mean = float(np.abs(ref).max()), float(np.abs(ref).mean())
    assert mx <= 8 * u * ref_max, f"{what}: max abs {mx:.3e} > {8 * u * ref_max:.3e} (8u of max |ref| {ref_max:.3e})"
    assert mn <= u * ref_mean, f"{what}: mean abs {mn:.3e} > {u * ref_mean:.3e} (u of mean |ref| {ref_mean:.3e})"
    return mx / ref_max, mn / ref_mean


@pytest.mark.parametrize("B,H,N,d,causal,dtype", [
    (1, 2, 1024, 64, True, syn.F16),     # several tiles, diagonal masking
    (1, 2, 640, 64, False, syn.F16),
    (2, 3, 333, 64, True, syn.F16),      # ragged last tile, several heads and batches
    (1, 2, 200, 64, False, syn.F16),
    (1, 1, 77, 64, True, syn.F16),       # one partial tile
    (1, 1, 1536, 64, False, syn.F16),    # twelve query tiles per key tile: the Q/dO ring wraps four times
    (1, 2, 512, 64, True, syn.BF16),
    (1, 1, 384, 64, False, syn.BF16),
    (1, 2, 640, 128, True, syn.F16),     # head dim 128: one Q/dO slot, dQ staged over dS^T
    (2, 2, 333, 128, False, syn.F16),    # ragged, several heads and batches
    (1, 1, 77, 128, True, syn.F16),      # one partial tile
    (1, 2, 512, 128, True, syn.BF16),
    (1, 1, 384, 128, False, syn.BF16),
])
def test_backward_matches_oracle(cq, B, H, N, d, causal, dtype):
    (qn, kn, vn, gn), (dq, dk, dv) = _run(cq, B, H, N, d, causal, dtype)
    ref = oracle.attn_bwd(qn, kn, vn, gn, B=B, H=H, N=N, d=d, causal=causal, dtype=dtype)
    rel = {}
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        rel[name] = _check(to_np64(t), ref[name], dtype, f"{name} N={N} causal={causal}")
    print(f"\nbwd N={N} d={d} causal={causal} dtype={dtype}: " +
          ", ".join(f"{n} max/maxref {a:.2e} mean/meanref {b:.2e}" for n, (a, b) in rel.items()))


def test_single_token(cq):
    """N = 1: P = 1, so dv = dout exactly (P rounds to 1.0) and dS = dP - D, which is zero up to the
    fp32 rounding of two orders of the same dot product, so dq and dk are ~1e-6 instead of O(1)."""
    (qn, kn, vn, gn), (dq, dk, dv) = _run(cq, 1, 2, 1, 64, True, syn.F16)
    assert float(dq.float().abs().max()) <= 1e-4 and float(dk.float().abs().max()) <= 1e-4
    np.testing.assert_array_equal(to_np64(dv), oracle.widen(gn).reshape(1, 2, 1, 64))


def test_uniform_scores_give_zero_dk(cq):
    """q = 0: dk = scale * sum_i dS_ij q_i is exactly zero on any hardware."""
    _, (dq, dk, dv) = _run(cq, 1, 2, 384, 64, True, syn.F16, q_zero=True)
    assert torch.count_nonzero(dk).item() == 0


def test_dk_dv_bitwise_reproducible(cq):
    """dk and dv are accumulated in a fixed order (one CTA per key tile); dq's atomic order may vary."""
    _, (dq1, dk1, dv1) = _run(cq, 1, 2, 768, 64, True, syn.F16, seed=4)
    _, (dq2, dk2, dv2) = _run(cq, 1, 2, 768, 64, True, syn.F16, seed=4)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert float((dq1.float() - dq2.float()).abs().max()) <= 2.0 ** -10 * float(dq1.float().abs().max())


@pytest.mark.parametrize("causal,d", [(True, 64), (False, 64), (True, 128)])
def test_sum_identities_large(cq, causal, d):
    """At a size the oracle cannot evaluate in full (8 heads x 8,192 tokens), two identities that hold
    for any inputs: sum_j dk_j = 0 (keys shifted together leave the softmax unchanged) and
    sum_j dv_j = sum_i dout_i (every P row sums to one)."""
    B, H, N = 1, 8, 8192
    (qn, kn, vn, gn), (dq, dk, dv) = _run(cq, B, H, N, d, causal, syn.F16, seed=2)
    dk64, dv64 = to_np64(dk), to_np64(dv)
    g64 = oracle.widen(gn).reshape(B, H, N, d)
    u = U[syn.F16]
    # each summed element carries a rounding error <= u |x|; the sums are checked against that budget
    assert np.all(np.abs(dk64.sum(axis=2)) <= 4 * u * np.abs(dk64).sum(axis=2) + 1e-6)
    assert np.all(np.abs(dv64.sum(axis=2) - g64.sum(axis=2)) <= 4 * u * np.abs(dv64).sum(axis=2) + 1e-6)


@pytest.mark.slow
def test_backward_32k_sampled_vs_oracle(cq):
    """The benchmark's backward shape (B=1 H=8 N=32768 d=64 fp16 causal) against the FP64 oracle: dq on
    2,048+ seeded sampled query rows (dq_i depends on row i alone), dk and dv on sampled key columns of two
    heads (each a sum over every query that sees the key), each held to the tolerance above over the
    sampled values."""
    B, H, N, d = 1, 8, 32768, 64
    (qn, kn, vn, gn), (dq, dk, dv) = _run(cq, B, H, N, d, True, syn.F16)
    rows = syn.sample_rows(B, H, N, 2048, causal_tile=128)
    js = syn.sample_rows(1, 1, N, 128, seed=5, must_i=(N - 128, N - 129, N // 2))[:, 2]
    cols = np.concatenate([np.stack([np.zeros_like(js), np.full_like(js, hh), js], axis=1) for hh in (0, H - 1)])

    def gather(t, idx):
        return to_np64(t[torch.as_tensor(idx[:, 0]), torch.as_tensor(idx[:, 1]), torch.as_tensor(idx[:, 2])])

    ref_dq = oracle.attn_bwd_rows(qn, kn, vn, gn, B=B, H=H, N=N, d=d, causal=True, rows=rows)
    ref_dk, ref_dv = oracle.attn_bwd_cols(qn, kn, vn, gn, B=B, H=H, N=N, d=d, causal=True, cols=cols)
    rel = {}
    for name, got, ref in (("dq", gather(dq, rows), ref_dq), ("dk", gather(dk, cols), ref_dk),
                           ("dv", gather(dv, cols), ref_dv)):
        rel[name] = _check(got, ref, syn.F16, f"32K {name}")
    print(f"\nbwd 32K causal on {len(rows)} rows / {len(cols)} columns: " +
          ", ".join(f"{n} max/maxref {a:.2e} mean/meanref {b:.2e}" for n, (a, b) in rel.items()))


def test_backward_d128_8k_sampled_vs_oracle(cq):
    """Head dim 128 at 8,192 tokens (B=1 H=4 bf16 non-causal, K scaled by 3 for peaked rows) against the
    FP64 oracle on 512 sampled query rows (dq) and 128 sampled key columns of two heads (dk, dv)."""
    B, H, N, d, dtype = 1, 4, 8192, 128, syn.BF16
    qn, kn, vn = syn.qkv(B, H, N, d, seed=7, dtype=dtype, k_mul=3.0)
    gn = syn.normal(B, H, N, d, seed=7, tensor_id=syn.TID_DO, dtype=dtype)
    q, k, v, g = (to_dev(x, dtype) for x in (qn, kn, vn, gn))
    out, lse = mono(cq, q, k, v, B, H, N, d, False, dtype)
    dq, dk, dv = cq.attention_backward(q, k, v, out, g, lse, causal=False)
    torch.cuda.synchronize()
    rc, code, _ = cq.cqsa_device_error()
    assert rc == cq.CQSA_OK and code == 0
    rows = syn.sample_rows(B, H, N, 512, seed=8)
    js = syn.sample_rows(1, 1, N, 64, seed=9, must_i=(0, N - 1, N // 2))[:, 2]
    cols = np.concatenate([np.stack([np.zeros_like(js), np.full_like(js, hh), js], axis=1) for hh in (0, H - 1)])

    def gather(t, idx):
        return to_np64(t[torch.as_tensor(idx[:, 0]), torch.as_tensor(idx[:, 1]), torch.as_tensor(idx[:, 2])])

    ref_dq = oracle.attn_bwd_rows(qn, kn, vn, gn, B=B, H=H, N=N, d=d, causal=False, rows=rows, dtype=dtype)
    ref_dk, ref_dv = oracle.attn_bwd_cols(qn, kn, vn, gn, B=B, H=H, N=N, d=d, causal=False, cols=cols, dtype=dtype)
    for name, got, ref in (("dq", gather(dq, rows), ref_dq), ("dk", gather(dk, cols), ref_dk),
                           ("dv", gather(dv, cols), ref_dv)):
        _check(got, ref, dtype, f"8K d=128 {name}")


@pytest.mark.slow
def test_backward_bf16_d128_bench_shape_sampled_vs_oracle(cq):
    """The benchmark's head-dim-128 backward (B=2 H=32 N=16,384 d=128 bf16 non-causal, K scaled by 3, the
    inputs of its bench line) against the FP64 oracle on 512+ sampled query rows (dq) and 64 sampled key
    columns of the first and last head (dk, dv)."""
    B, H, N, d, dtype = 2, 32, 16384, 128, syn.BF16
    qn, kn, vn = syn.qkv(B, H, N, d, seed=0, dtype=dtype, k_mul=3.0)
    gn = syn.normal(B, H, N, d, seed=0, tensor_id=syn.TID_DO, dtype=dtype)
    q, k, v, g = (to_dev(x, dtype) for x in (qn, kn, vn, gn))
    out, lse = mono(cq, q, k, v, B, H, N, d, False, dtype)
    dq, dk, dv = cq.attention_backward(q, k, v, out, g, lse, causal=False)
    torch.cuda.synchronize()
    rc, code, _ = cq.cqsa_device_error()
    assert rc == cq.CQSA_OK and code == 0
    rows = syn.sample_rows(B, H, N, 512, seed=11)
    js = syn.sample_rows(1, 1, N, 32, seed=12, must_i=(0, N - 1, N // 2))[:, 2]
    cols = np.concatenate([np.stack([np.full_like(js, bb), np.full_like(js, hh), js], axis=1)
                           for bb, hh in ((0, 0), (B - 1, H - 1))])

    def gather(t, idx):
        return to_np64(t[torch.as_tensor(idx[:, 0]), torch.as_tensor(idx[:, 1]), torch.as_tensor(idx[:, 2])])

    ref_dq = oracle.attn_bwd_rows(qn, kn, vn, gn, B=B, H=H, N=N, d=d, causal=False, rows=rows, dtype=dtype)
    ref_dk, ref_dv = oracle.attn_bwd_cols(qn, kn, vn, gn, B=B, H=H, N=N, d=d, causal=False, cols=cols, dtype=dtype)
    for name, got, ref in (("dq", gather(dq, rows), ref_dq), ("dk", gather(dk, cols), ref_dk),
                           ("dv", gather(dv, cols), ref_dv)):
        _check(got, ref, dtype, f"bf16 d=128 16K {name}")


def _chunked_backward(cq, q, k, v, g, out, lse, B, H, N, d, C, causal, dtype, skip_masked=True):
    """The backward over (query chunk, key chunk) pairs of C tokens through cqsa_attn_bwd_chunk, with
    per-chunk fp32 accumulators cast to dtype at the end."""
    dev = q.device
    starts = list(range(0, N, C))
    sz = {s0: min(C, N - s0) for s0 in starts}
    dq_acc = {s0: torch.zeros((B, H, sz[s0], d), dtype=torch.float32, device=dev) for s0 in starts}
    dk_acc = {s0: torch.zeros((B, H, sz[s0], d), dtype=torch.float32, device=dev) for s0 in starts}
    dv_acc = {s0: torch.zeros((B, H, sz[s0], d), dtype=torch.float32, device=dev) for s0 in starts}
    sl = lambda t, s0: t[:, :, s0:s0 + sz[s0]].contiguous()  # noqa: E731
    for qs in starts:
        nq = sz[qs]
        qb, gb, ob, lb = sl(q, qs), sl(g, qs), sl(out, qs), sl(lse, qs)
        db = torch.empty((B, H, nq), dtype=torch.float32, device=dev)
        cq.cqsa_attn_bwd_dvec(ob, gb, db, B, H, nq, d, dtype)
        for ks in starts:
            if skip_masked and causal and ks > qs + nq - 1:
                continue
            cq.cqsa_attn_bwd_chunk(qb, sl(k, ks), sl(v, ks), gb, lb, db, qs, ks, B, H, nq, sz[ks], d, causal, 0.0,
                                   dtype, dq_acc[qs], dk_acc[ks], dv_acc[ks])
    res = []
    for acc in (dq_acc, dk_acc, dv_acc):
        parts = []
        for s0 in starts:
            o = torch.empty((B, H, sz[s0], d), dtype=q.dtype, device=dev)
            cq.cqsa_attn_bwd_cast(acc[s0], o, acc[s0].numel(), dtype)
            parts.append(o)
        res.append(torch.cat(parts, dim=2))
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("N,C,causal,dtype,d", [
    (768, 256, True, syn.F16, 64),    # 3 x 3 chunks of two tiles, 6 causal pairs
    (640, 200, True, syn.F16, 64),    # chunks not aligned to the 128-token tiles, ragged last chunk
    (512, 192, False, syn.BF16, 64),  # every pair
    (640, 200, True, syn.F16, 128),
    (512, 256, False, syn.BF16, 128),
])
def test_chunked_backward(cq, N, C, causal, dtype, d):
    """Accumulating every chunk pair gives the oracle's gradients (same tolerance as the monolithic
    call) and the monolithic call's, within a few ulps of dtype (fp32 summation order differs)."""
    B, H = 1, 2
    (qn, kn, vn, gn), mono_grads = _run(cq, B, H, N, d, causal, dtype)
    q, k, v, g = (to_dev(x, dtype) for x in (qn, kn, vn, gn))
    out, lse = mono(cq, q, k, v, B, H, N, d, causal, dtype)
    grads = _chunked_backward(cq, q, k, v, g, out, lse, B, H, N, d, C, causal, dtype)
    rc, code, _ = cq.cqsa_device_error()
    assert rc == cq.CQSA_OK and code == 0
    ref = oracle.attn_bwd(qn, kn, vn, gn, B=B, H=H, N=N, d=d, causal=causal, dtype=dtype)
    u = U[dtype]
    for name, t, m in zip(("dq", "dk", "dv"), grads, mono_grads):
        _check(to_np64(t), ref[name], dtype, f"chunked {name} N={N} C={C}")
        diff = float((t.float() - m.float()).abs().max())
        assert diff <= 4 * u * float(m.float().abs().max()), (name, diff)


def test_chunk_pair_above_diagonal_adds_nothing(cq):
    """A causal pair whose keys all follow every query leaves the accumulators untouched."""
    B, H, N, d, C = 1, 2, 512, 64, 256
    (qn, kn, vn, gn), _ = _run(cq, B, H, N, d, True, syn.F16)
    q, k, v, g = (to_dev(x, syn.F16) for x in (qn, kn, vn, gn))
    out, lse = mono(cq, q, k, v, B, H, N, d, True, syn.F16)
    dev = q.device
    qb, gb, ob, lb = (t[:, :, :C].contiguous() for t in (q, g, out, lse))
    kb, vb = (t[:, :, C:].contiguous() for t in (k, v))
    db = torch.empty((B, H, C), dtype=torch.float32, device=dev)
    cq.cqsa_attn_bwd_dvec(ob, gb, db, B, H, C, d, syn.F16)
    accs = [torch.full((B, H, C, d), 0.5, dtype=torch.float32, device=dev) for _ in range(3)]
    cq.cqsa_attn_bwd_chunk(qb, kb, vb, gb, lb, db, 0, C, B, H, C, N - C, d, True, 0.0, syn.F16, *accs)
    torch.cuda.synchronize()
    assert all(bool((a == 0.5).all()) for a in accs)


@pytest.mark.parametrize("resident", [True, False])
@pytest.mark.parametrize("B,H,N,C,causal,d", [(2, 2, 640, 256, True, 64), (1, 2, 384, 128, False, 64),
                                             (1, 2, 640, 256, True, 128)])
def test_stream_backward(cq, B, H, N, C, causal, d, resident):
    """Host-resident backward over chunks (ragged last chunk, several batches and heads), with the inputs
    kept resident (one launch per key chunk over every query) and through double-buffered chunk pairs:
    equal to the monolithic device call within a few ulps (fp32 summation order differs)."""
    dtype = syn.F16
    (qn, kn, vn, gn), mono_grads = _run(cq, B, H, N, d, causal, dtype)
    q, k, v, g = (to_dev(x, dtype) for x in (qn, kn, vn, gn))
    out, lse = mono(cq, q, k, v, B, H, N, d, causal, dtype)
    host = [t.cpu().pin_memory() for t in (q, k, v, out, g, lse)]
    grads = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(3)]
    cq.cqsa_set_stream_kv_resident_bytes(1 << 40 if resident else 0)
    try:
        st = cq.cqsa_stream_attn_bwd_ex(*host, *grads, B, H, N, d, causal, 0.0, dtype, C)
    finally:
        cq.cqsa_set_stream_kv_resident_bytes(-1)
    n_chunks = -(-N // C)
    pairs = n_chunks * (n_chunks + 1) // 2 if causal else n_chunks * n_chunks
    assert st.n_chunks == (n_chunks if resident else pairs) and st.compute_ms > 0
    assert st.wall_ms >= st.compute_ms * 0.5
    # every input crosses the link at least once: q, out, dout, k, v and lse
    assert st.h2d_bytes >= 5 * B * H * N * d * 2 + B * H * N * 4
    assert st.d2h_bytes == 3 * B * H * N * d * 2
    u = U[dtype]
    for name, t, m in zip(("dq", "dk", "dv"), grads, mono_grads):
        m = m.float().cpu()
        diff = float((t.float() - m).abs().max())
        assert diff <= 4 * u * float(m.abs().max()), (name, diff)


@pytest.mark.slow
@pytest.mark.parametrize("resident", [True, False])
def test_stream_backward_32k_sampled_vs_oracle(cq, resident):
    """The host-resident backward at 32,768 tokens in 8,192-token chunks (B=1 H=4 d=64 fp16 causal), with
    the inputs kept resident (one launch per key chunk) and through double-buffered chunk pairs: dq on
    2,048+ seeded sampled query rows and dk, dv on sampled key columns of two heads against the FP64
    oracle, and every gradient against the monolithic device call within a few ulps."""
    B, H, N, d, C = 1, 4, 32768, 64, 8192
    dtype = syn.F16
    (qn, kn, vn, gn), mono_grads = _run(cq, B, H, N, d, True, dtype)
    q, k, v, g = (to_dev(x, dtype) for x in (qn, kn, vn, gn))
    out, lse = mono(cq, q, k, v, B, H, N, d, True, dtype)
    host = [t.cpu().pin_memory() for t in (q, k, v, out, g, lse)]
    grads = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(3)]
    cq.cqsa_set_stream_kv_resident_bytes(1 << 40 if resident else 0)
    try:
        st = cq.cqsa_stream_attn_bwd_ex(*host, *grads, B, H, N, d, True, 0.0, dtype, C)
    finally:
        cq.cqsa_set_stream_kv_resident_bytes(-1)
    n_chunks = N // C
    assert st.n_chunks == (n_chunks if resident else n_chunks * (n_chunks + 1) // 2)
    dq, dk, dv = grads
    rows = syn.sample_rows(B, H, N, 2048, chunk=C, causal_tile=128)
    js = syn.sample_rows(1, 1, N, 128, seed=5, must_i=(C - 1, C, N - 128, N // 2))[:, 2]
    cols = np.concatenate([np.stack([np.zeros_like(js), np.full_like(js, hh), js], axis=1) for hh in (0, H - 1)])

    def gather(t, idx):
        return t[torch.as_tensor(idx[:, 0]), torch.as_tensor(idx[:, 1]), torch.as_tensor(idx[:, 2])].float().numpy().astype(np.float64)

    ref_dq = oracle.attn_bwd_rows(qn, kn, vn, gn, B=B, H=H, N=N, d=d, causal=True, rows=rows)
    ref_dk, ref_dv = oracle.attn_bwd_cols(qn, kn, vn, gn, B=B, H=H, N=N, d=d, causal=True, cols=cols)
    for name, got, ref in (("dq", gather(dq, rows), ref_dq), ("dk", gather(dk, cols), ref_dk),
                           ("dv", gather(dv, cols), ref_dv)):
        _check(got, ref, dtype, f"stream 32K {name} resident={resident}")
    u = U[dtype]
    for name, t, m in zip(("dq", "dk", "dv"), grads, mono_grads):
        m = m.float().cpu()
        diff = float((t.float() - m).abs().max())
        assert diff <= 4 * u * float(m.abs().max()), (name, diff)
