"""The no-allocation entry point (cqsa_attn_fwd_chunked_static) against the existing chunked path and
the FP64 oracle.

Some callers cannot let a library call cudaMalloc (they run under their own memory pool or a hard
device-memory budget). cqsa_attn_fwd_chunked_static serves them: its fp32 accumulator is a fixed
device array inside the library. These tests call it through the C ABI, twice in a row on different
problems, and check each result against cqsa_stream_attn_fwd (which allocates its own buffers) on the
same inputs and against the oracle, within the tolerances of the other parity tests. For bf16 the
output is anchored to the fp32 result of the same computation over the whole key range (the chunk
call), which itself meets the fp32 tolerances against the oracle. The file sorts last so that a run
stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._gpu import TORCH_DT, assert_bf16_rounds_fp32_result, assert_close, to_dev, to_np64

pytestmark = pytest.mark.gpu


def _run_both(cq, B, H, N, d, causal, C, seed, dtype=syn.F16, oracle_rows=None):
    qn, kn, vn = syn.qkv(B, H, N, d, seed=seed, dtype=dtype, k_mul=3.0 if dtype == syn.BF16 else 1.0)
    q, k, v = (to_dev(x, dtype) for x in (qn, kn, vn))
    tdt = TORCH_DT[dtype]
    out = torch.full((B, H, N, d), float("nan"), dtype=tdt, device="cuda")
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    cq.cqsa_attn_fwd_chunked_static(q, k, v, out, lse, B, H, N, d, causal, 0.0, dtype, C)
    hq, hk, hv = (torch.from_numpy(x.view(np.int16)).view(tdt).pin_memory() for x in (qn, kn, vn))
    ref = torch.empty((B, H, N, d), dtype=tdt, device="cuda")
    rl = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    cq.cqsa_stream_attn_fwd(hq, hk, hv, cq.CQSA_LAYOUT_BHND, ref, rl, False, B, H, N, d, causal, 0.0, dtype, C)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    what = f"static N={N} d={d} dtype={dtype} causal={causal}"
    if oracle_rows is None:
        bb, hh, ii = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), indexing="ij")
        rows = np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1)
    else:
        rows = syn.sample_rows(B, H, N, oracle_rows, chunk=C)
    ro, rll, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=N, d=d, causal=causal, dtype=dtype, rows=rows)
    b, h, i = (torch.as_tensor(rows[:, j], device="cuda") for j in range(3))
    if dtype == syn.F16:
        assert_close(to_np64(out), to_np64(ref), to_np64(lse), to_np64(rl), what=what + " vs streamed")
        assert_close(to_np64(out[b, h, i]), ro, to_np64(lse[b, h, i]), rll, what=what + " vs oracle")
    else:
        O32 = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
        L32 = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        cq.cqsa_attn_fwd_chunk(q, k, v, 0, 0, B, H, N, N, d, causal, 0.0, dtype, O32, L32, False)
        assert_close(to_np64(O32[b, h, i]), ro, to_np64(L32[b, h, i]), rll, what=what + " fp32 anchor vs oracle")
        assert_bf16_rounds_fp32_result(to_np64(out), to_np64(O32), what)
        assert_bf16_rounds_fp32_result(to_np64(ref), to_np64(O32), what + " (streamed)")
        lrel = (lse - L32).abs() / L32.abs().clamp_min(1.0)
        assert lrel.max().item() <= 1e-5
    # both entry points run the same chunk pairs: their LSEs agree to fp32 merge-order rounding
    assert ((lse - rl).abs() / rl.abs().clamp_min(1.0)).max().item() <= 1e-5


def test_no_alloc_entry_matches_existing_path_twice():
    import exact_long_context_tcgen05_gb300 as cq
    _run_both(cq, B=1, H=2, N=1000, d=64, causal=True, C=256, seed=21)
    _run_both(cq, B=2, H=3, N=700, d=128, causal=False, C=384, seed=22)
    rc, code, _ = cq.cqsa_device_error()
    assert rc == cq.CQSA_OK and code == 0


def test_no_alloc_bf16_and_causal_d128():
    import exact_long_context_tcgen05_gb300 as cq
    _run_both(cq, B=1, H=2, N=900, d=128, causal=True, C=256, seed=23, dtype=syn.BF16)
    _run_both(cq, B=2, H=2, N=777, d=64, causal=True, C=128, seed=24, dtype=syn.BF16)
    _run_both(cq, B=1, H=3, N=1100, d=128, causal=True, C=512, seed=25)


def test_no_alloc_head_groups():
    """A chunk size whose accumulators for all heads exceed the array: heads run in groups (7 + 1 here)."""
    import exact_long_context_tcgen05_gb300 as cq
    C, d = 16384, 64
    assert 8 * C * (d + 1) * 4 > cq.CQSA_STATIC_SCRATCH_BYTES >= 7 * C * (d + 1) * 4
    _run_both(cq, B=1, H=8, N=20000, d=d, causal=True, C=C, seed=26, oracle_rows=512)


def test_no_alloc_rejects_oversized_chunk():
    import exact_long_context_tcgen05_gb300 as cq
    fake = 0x10000
    C = 1 << 17  # 131072 * 65 * 4 bytes > 32 MiB
    rc = cq.lib.cqsa_attn_fwd_chunked_static(fake, fake, fake, fake, None, 1, 1, C, 64, 1, 0.0, cq.CQSA_F16, C, None)
    assert rc == cq.CQSA_ERR_UNSUPPORTED and "static scratch" in cq.last_error()
