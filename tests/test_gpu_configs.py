"""GPU parity at the full workload sizes, in the launch configuration the benchmark uses.

Large problems are checked on >= 2,048 seeded sampled query rows (always including rows 0, 1, 127,
128, N-1 and the chunk boundaries), each computed in full by the FP64 oracle. The chunked workload is
also compared with the monolithic fp32 result on every row.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._gpu import TORCH_DT, assert_close, to_dev, to_np64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def cq():
    import exact_long_context_tcgen05_gb300 as m
    return m


def _gather(t: torch.Tensor, rows: np.ndarray, layout=syn.LAYOUT_BHND) -> np.ndarray:
    b = torch.as_tensor(rows[:, 0], device=t.device)
    h = torch.as_tensor(rows[:, 1], device=t.device)
    i = torch.as_tensor(rows[:, 2], device=t.device)
    if layout == syn.LAYOUT_BHND:
        return to_np64(t[b, h, i])
    return to_np64(t[b, i, h])


def test_causal_32k_d64_fp16(cq):
    """B=1, H=8, N=32768, d=64, fp16 N(0,1), causal, monolithic (the benchmark workload)."""
    B, H, N, d = 1, 8, 32768, 64
    qn, kn, vn = syn.qkv(B, H, N, d, seed=0)
    q, k, v = (to_dev(x, syn.F16) for x in (qn, kn, vn))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    cq.cqsa_attn_fwd(q, k, v, out, lse, B, H, N, d, True, 0.0, cq.CQSA_F16)
    rows = syn.sample_rows(B, H, N, 2048, causal_tile=128)
    ro, rl, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=N, d=d, causal=True, rows=rows)
    mx, mn = assert_close(_gather(out, rows), ro, _gather(lse, rows), rl, what="32K causal")
    print(f"\n32K causal d64 fp16 on {len(rows)} rows: max abs {mx:.2e} mean abs {mn:.2e}")
    # the benchmark's end-to-end path on the same inputs: pinned host buffers through the streaming
    # driver in 4,096-token chunks (inputs resident, one launch per query chunk over its key prefix)
    # gives the monolithic call's bits
    hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
    hout = torch.empty((B, H, N, d), dtype=torch.float16).pin_memory()
    hlse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    st = cq.cqsa_stream_stats()
    cq.cqsa_stream_attn_fwd(hq, hk, hv, cq.CQSA_LAYOUT_BHND, hout, hlse, True, B, H, N, d, True, 0.0, cq.CQSA_F16,
                            N // 8, st)
    assert st.n_chunks == 8, "the 32K workload's inputs fit: one launch per query chunk"
    assert torch.equal(hout.cuda(), out) and torch.equal(hlse.cuda(), lse)


def test_noncausal_16k_d128_bf16_peaked(cq):
    """B=2, H=32, N=16384, d=128, bf16 N(0,1) with K scaled by 3 (peaked rows), non-causal."""
    B, H, N, d = 2, 32, 16384, 128
    qn, kn, vn = syn.qkv(B, H, N, d, seed=0, dtype=syn.BF16, k_mul=3.0)
    q, k, v = (to_dev(x, syn.BF16) for x in (qn, kn, vn))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    cq.cqsa_attn_fwd(q, k, v, out, lse, B, H, N, d, False, 0.0, cq.CQSA_BF16)
    O = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    L = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    cq.cqsa_attn_fwd_chunk(q, k, v, 0, 0, B, H, N, N, d, False, 0.0, cq.CQSA_BF16, O, L, False)
    rows = syn.sample_rows(B, H, N, 2048)
    ro, rl, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=N, d=d, causal=False, dtype=syn.BF16, rows=rows)
    o32 = _gather(O, rows)
    mx, mn = assert_close(o32, ro, _gather(L, rows), rl, what="16K bf16 fp32 result")
    # the bf16 output is the fp32 result rounded to nearest even (on every row)
    assert torch.equal(out, O.to(torch.bfloat16))
    assert torch.equal(lse, L)
    print(f"\n16K bf16 peaked (fp32 result) on {len(rows)} rows: max abs {mx:.2e} mean abs {mn:.2e}")


def test_bf16_d128_chunked_4096_equals_monolithic(cq):
    """B=2, H=32, N=16384, d=128, bf16 with K scaled by 3 (peaked rows), non-causal, cut into 4,096-token
    chunks: the 16 chunk-pair partials merged exactly equal the monolithic fp32 result within 1e-5 per
    row (relative to the row's largest |O|; LSE relative to max(1, |LSE|)), and the oracle on sampled
    rows within the stated tolerances."""
    B, H, N, d, C = 2, 32, 16384, 128, 4096
    qn, kn, vn = syn.qkv(B, H, N, d, seed=0, dtype=syn.BF16, k_mul=3.0)
    q, k, v = (to_dev(x, syn.BF16) for x in (qn, kn, vn))
    Om = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    Lm = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    cq.cqsa_attn_fwd_chunk(q, k, v, 0, 0, B, H, N, N, d, False, 0.0, cq.CQSA_BF16, Om, Lm, False)
    nch = N // C
    out32 = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    worst = 0.0
    ks = [k[:, :, j * C:(j + 1) * C].contiguous() for j in range(nch)]
    vs = [v[:, :, j * C:(j + 1) * C].contiguous() for j in range(nch)]
    for i in range(nch):
        qs = q[:, :, i * C:(i + 1) * C].contiguous()
        parts_o, parts_l = [], []
        for j in range(nch):
            Op = torch.empty((B, H, C, d), dtype=torch.float32, device="cuda")
            Lp = torch.empty((B, H, C), dtype=torch.float32, device="cuda")
            cq.cqsa_attn_fwd_chunk(qs, ks[j], vs[j], i * C, j * C, B, H, C, C, d, False, 0.0, cq.CQSA_BF16, Op, Lp,
                                   False)
            parts_o.append(Op)
            parts_l.append(Lp)
        o32 = torch.empty((B, H, C, d), dtype=torch.float32, device="cuda")
        l32 = torch.empty((B, H, C), dtype=torch.float32, device="cuda")
        cq.cqsa_merge_partials(parts_o, parts_l, nch, o32, l32, B, H, C, d, cq.CQSA_F32)
        out32[:, :, i * C:(i + 1) * C] = o32
        lse[:, :, i * C:(i + 1) * C] = l32
        ref = Om[:, :, i * C:(i + 1) * C]
        den = ref.abs().amax(dim=-1).clamp_min(1e-30)
        rel = ((o32 - ref).abs().amax(dim=-1) / den).max().item()
        lref = Lm[:, :, i * C:(i + 1) * C]
        lrel = ((l32 - lref).abs() / lref.abs().clamp_min(1.0)).max().item()
        worst = max(worst, rel)
        assert rel <= 1e-5 and lrel <= 1e-5, f"Q chunk {i}: rel {rel:.2e}, lse rel {lrel:.2e}"
        del parts_o, parts_l
    rows = syn.sample_rows(B, H, N, 2048, chunk=C)
    ro, rl, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=N, d=d, causal=False, dtype=syn.BF16, rows=rows)
    mx, mn = assert_close(_gather(out32, rows), ro, _gather(lse, rows), rl, what="16K bf16 d128 chunked vs oracle")
    print(f"\n16K bf16 d128 4096-token chunks: chunked-vs-mono worst row rel {worst:.2e}; vs oracle max abs "
          f"{mx:.2e} mean abs {mn:.2e}")


def test_chunked_131k_merge_equals_monolithic(cq):
    """B=1, H=8, N=131072, d=64, fp16, causal, 16384-token chunks: 36 pair partials + LSE merge,
    compared with the monolithic fp32 result on every row (1e-5 relative) and with the oracle on
    sampled rows."""
    B, H, N, d, C = 1, 8, 131072, 64, 16384
    qn, kn, vn = syn.qkv(B, H, N, d, seed=0)
    q, k, v = (to_dev(x, syn.F16) for x in (qn, kn, vn))
    Om = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    Lm = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    cq.cqsa_attn_fwd_chunk(q, k, v, 0, 0, B, H, N, N, d, True, 0.0, cq.CQSA_F16, Om, Lm, False)
    nch = N // C
    out = torch.empty((B, H, N, d), dtype=torch.float16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    out32 = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    worst = 0.0
    for i in range(nch):
        qs = q[:, :, i * C:(i + 1) * C].contiguous()
        parts_o, parts_l = [], []
        for j in range(i + 1):
            ks = k[:, :, j * C:(j + 1) * C].contiguous()
            vs = v[:, :, j * C:(j + 1) * C].contiguous()
            Op = torch.empty((B, H, C, d), dtype=torch.float32, device="cuda")
            Lp = torch.empty((B, H, C), dtype=torch.float32, device="cuda")
            cq.cqsa_attn_fwd_chunk(qs, ks, vs, i * C, j * C, B, H, C, C, d, True, 0.0, cq.CQSA_F16, Op, Lp, False)
            parts_o.append(Op)
            parts_l.append(Lp)
        o16 = torch.empty((B, H, C, d), dtype=torch.float16, device="cuda")
        o32 = torch.empty((B, H, C, d), dtype=torch.float32, device="cuda")
        l32 = torch.empty((B, H, C), dtype=torch.float32, device="cuda")
        cq.cqsa_merge_partials(parts_o, parts_l, len(parts_o), o32, l32, B, H, C, d, cq.CQSA_F32)
        cq.cqsa_merge_partials(parts_o, parts_l, len(parts_o), o16, None, B, H, C, d, cq.CQSA_F16)
        out[:, :, i * C:(i + 1) * C] = o16
        out32[:, :, i * C:(i + 1) * C] = o32
        lse[:, :, i * C:(i + 1) * C] = l32
        ref = Om[:, :, i * C:(i + 1) * C]
        den = ref.abs().amax(dim=-1).clamp_min(1e-30)
        rel = ((o32 - ref).abs().amax(dim=-1) / den).max().item()
        lrel = ((l32 - Lm[:, :, i * C:(i + 1) * C]).abs() / Lm[:, :, i * C:(i + 1) * C].abs().clamp_min(1.0)).max().item()
        worst = max(worst, rel)
        assert rel <= 1e-5 and lrel <= 1e-5, f"Q chunk {i}: rel {rel:.2e}, lse rel {lrel:.2e}"
        del parts_o, parts_l
    assert torch.equal(out, out32.to(torch.float16))
    rows = syn.sample_rows(B, H, N, 2048, chunk=C)
    ro, rl, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=N, d=d, causal=True, rows=rows)
    mx, mn = assert_close(_gather(out, rows), ro, _gather(lse, rows), rl, what="131K chunked vs oracle")
    print(f"\n131K chunked: chunked-vs-mono worst row rel {worst:.2e}; vs oracle max abs {mx:.2e} mean abs {mn:.2e}")


def test_wave_engine_262k_equals_monolithic(cq):
    """The quorum decomposition of the bench's wave-engine line (B=1 H=8 N=262,144 d=64 fp16 causal,
    c = 31, interest set (0, 1, 3, 8, 12, 18), token-major device inputs read in place): its adjacent key
    chunks run as one key range per query chunk, so the result is the monolithic call's, bit for bit."""
    B, H, N, d = 1, 8, 262_144, 64
    qn, kn, vn = syn.qkv(B, H, N, d, seed=3, layout=syn.LAYOUT_BNHD)
    q, k, v = (to_dev(x, syn.F16) for x in (qn, kn, vn))
    out = torch.empty((B, N, H, d), dtype=torch.float16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    st = cq.cqsa_quorum_stats()
    cq.cqsa_quorum_attn_fwd_ex(q, k, v, cq.CQSA_LAYOUT_BNHD, False, out, lse, False, B, H, N, d, True, 0.0,
                               cq.CQSA_F16, 31, (0, 1, 3, 8, 12, 18), 1, engine=cq.CQSA_ENGINE_WAVE, stats=st)
    assert st.n_pairs == 496
    qb, kb, vb = (x.permute(0, 2, 1, 3).contiguous() for x in (q, k, v))
    ob = torch.empty_like(qb)
    lb = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    cq.cqsa_attn_fwd(qb, kb, vb, ob, lb, B, H, N, d, True, 0.0, cq.CQSA_F16)
    torch.cuda.synchronize()
    assert torch.equal(out.permute(0, 2, 1, 3), ob) and torch.equal(lse, lb)


def test_streaming_4m_host_resident(cq):
    """B=1, H=8, N=4,000,000, d=64, fp16, causal, Q/K/V in pinned host memory (token-major), streamed in
    262,144-token chunks; 2,048+ sampled rows against the oracle."""
    B, H, N, d, C = 1, 8, 4_000_000, 64, 262_144
    shape = (B, N, H, d)
    t0 = time.time()
    host = [torch.empty(shape, dtype=torch.float16).pin_memory() for _ in range(3)]
    for tid, t in enumerate(host):
        syn.normal(B, H, N, d, seed=0, tensor_id=tid, layout=syn.LAYOUT_BNHD, out=t.numpy().view(np.uint16))
    out = torch.empty(shape, dtype=torch.float16).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    t_gen = time.time() - t0
    st = cq.cqsa_stream_stats()
    t1 = time.time()
    cq.cqsa_stream_attn_fwd(host[0], host[1], host[2], cq.CQSA_LAYOUT_BNHD, out, lse, True, B, H, N, d, True, 0.0,
                            cq.CQSA_F16, C, st)
    wall = time.time() - t1
    rows = syn.sample_rows(B, H, N, 2048, chunk=C)
    qn, kn, vn = (t.numpy().view(np.uint16) for t in host)
    t2 = time.time()
    ro, rl, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=N, d=d, causal=True, rows=rows, layout=oracle.LAYOUT_BNHD)
    t_or = time.time() - t2
    mx, mn = assert_close(_gather(out, rows, syn.LAYOUT_BNHD), ro, _gather(lse, rows), rl, what="4M streamed")
    flop = 4.0 * B * H * N * N * d / 2
    print(f"\n4M streamed: {wall:.1f} s wall ({flop / wall / 1e12:.0f} TFLOP/s), h2d {st.h2d_bytes / 1e9:.1f} GB in "
          f"{st.h2d_ms / 1e3:.2f} s of copy time ({st.h2d_bytes / st.h2d_ms / 1e6:.0f} GB/s), compute {st.compute_ms / 1e3:.1f} s, "
          f"stall {st.stall_ms:.0f} ms, device {st.peak_device_bytes / 2**30:.2f} GiB; "
          f"max abs {mx:.2e} mean abs {mn:.2e} on {len(rows)} rows; gen {t_gen:.0f} s, oracle {t_or:.0f} s")
    nq = (N + C - 1) // C
    # K/V (8.2 GB) stay resident by default on a GB300: one launch per Q chunk over its key prefix
    assert st.n_chunks in (nq, nq * (nq + 1) // 2)
