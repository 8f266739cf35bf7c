"""The library in a process that uses two GPUs: each device gets its own one-time set-up (kernel
attributes, SM count), so the same call gives the same bits on cuda:0 and then cuda:1, and the forward,
the backward and the merge each work on the second device after the first. Skips on a one-GPU machine."""
import numpy as np
import pytest
import torch

import synthetic as syn
from tests._gpu import to_np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cq():
    import exact_long_context_tcgen05_gb300 as m
    return m


def _inputs(dev, B, H, N, d):
    qn, kn, vn = syn.qkv(B, H, N, d, seed=21)
    return [torch.from_numpy(x.view(np.int16)).view(torch.float16).to(dev) for x in (qn, kn, vn)]


def test_forward_and_backward_on_two_devices(cq):
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    B, H, N, d = 1, 2, 640, 64
    res = []
    for idx in (0, 1):
        dev = torch.device("cuda", idx)
        with torch.cuda.device(dev):
            q, k, v = _inputs(dev, B, H, N, d)
            out, lse = cq.attention(q, k, v, causal=True, return_lse=True)
            g = torch.ones_like(q)
            dq, dk, dv = cq.attention_backward(q, k, v, out, g, lse, causal=True)
            torch.cuda.synchronize(dev)
            rc, code, _ = cq.cqsa_device_error()
            assert rc == cq.CQSA_OK and code == 0
            res.append([to_np64(t) for t in (out, lse, dq, dk, dv)])
    for a, b in zip(res[0], res[1]):
        assert np.array_equal(a, b)
