"""The no-allocation entry point (cqsa_attn_fwd_chunked_static) against the existing chunked path.

Some callers cannot let a library call cudaMalloc (they run under their own memory pool or a hard
device-memory budget). cqsa_attn_fwd_chunked_static serves them: its fp32 accumulator is a fixed
device array inside the library. This test calls it twice in a row through the C ABI, on different
problems, and checks each result against cqsa_stream_attn_fwd (which allocates its own buffers) on
the same inputs, within the tolerances of the other parity tests. The file sorts last so that a run
stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import synthetic as syn
from tests._gpu import assert_close, to_dev, to_np64

pytestmark = pytest.mark.gpu


def _run_both(cq, B, H, N, d, causal, C, seed):
    qn, kn, vn = syn.qkv(B, H, N, d, seed=seed)
    q, k, v = (to_dev(x, syn.F16) for x in (qn, kn, vn))
    out = torch.full((B, H, N, d), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    cq.cqsa_attn_fwd_chunked_static(q, k, v, out, lse, B, H, N, d, causal, 0.0, cq.CQSA_F16, C)
    hq, hk, hv = (torch.from_numpy(x.view(np.int16)).view(torch.float16).pin_memory() for x in (qn, kn, vn))
    ref = torch.empty((B, H, N, d), dtype=torch.float16, device="cuda")
    rl = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    cq.cqsa_stream_attn_fwd(hq, hk, hv, cq.CQSA_LAYOUT_BHND, ref, rl, False, B, H, N, d, causal, 0.0, cq.CQSA_F16, C)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(to_np64(out), to_np64(ref), to_np64(lse), to_np64(rl), what=f"static vs streamed N={N} d={d}")


def test_no_alloc_entry_matches_existing_path_twice():
    import exact_long_context_tcgen05_gb300 as cq
    _run_both(cq, B=1, H=2, N=1000, d=64, causal=True, C=256, seed=21)
    _run_both(cq, B=2, H=3, N=700, d=128, causal=False, C=384, seed=22)
    rc, code, _ = cq.cqsa_device_error()
    assert rc == cq.CQSA_OK and code == 0


def test_no_alloc_rejects_oversized_chunk():
    import exact_long_context_tcgen05_gb300 as cq
    fake = 0x10000
    C = 1 << 17  # 131072 * 65 * 4 bytes > 32 MiB
    rc = cq.lib.cqsa_attn_fwd_chunked_static(fake, fake, fake, fake, None, 1, 1, C, 64, 1, 0.0, cq.CQSA_F16, C, None)
    assert rc == cq.CQSA_ERR_UNSUPPORTED and "static scratch" in cq.last_error()
