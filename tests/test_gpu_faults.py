"""Failure detection without a GPU fault: a device wait that can never complete must give up after
the configured limit, record a code the host reads, drain its in-flight copies and MMAs, free tensor
memory and return, leaving the context usable. The failure is made on the host (a test hook tells one
CTA to skip a load); nothing traps, hangs or touches a bad address."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._gpu import assert_close, mono, to_dev, to_np64

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_survives():
    import exact_long_context_tcgen05_gb300 as cq
    B, H, N, d = 1, 2, 1024, 64
    qn, kn, vn = syn.qkv(B, H, N, d, seed=31)
    q, k, v = (to_dev(x, syn.F16) for x in (qn, kn, vn))
    assert cq.cqsa_device_error(clear=True)[0] == cq.CQSA_OK
    cq.cqsa_set_timeout_ms(200)
    try:
        cq.cqsa_debug_set_fault(1)
        mono(cq, q, k, v, B, H, N, d, True, syn.F16)
        torch.cuda.synchronize()  # the kernel returned by itself: no CUDA error
        rc, code, block = cq.cqsa_device_error(clear=True)
        assert rc == cq.CQSA_ERR_TIMEOUT and code != 0 and block == 0
        assert "gave up" in cq.last_error()
    finally:
        cq.cqsa_debug_set_fault(0)
        cq.cqsa_set_timeout_ms(0)
    assert cq.cqsa_device_error(clear=True)[0] == cq.CQSA_OK
    out, lse = mono(cq, q, k, v, B, H, N, d, True, syn.F16)
    ref_o, ref_l = oracle.attn_full(qn, kn, vn, B=B, H=H, N=N, d=d, causal=True)
    assert_close(to_np64(out), ref_o, to_np64(lse), ref_l, what="after recovery")


def test_fault_hook_rejects_unknown_kind():
    import exact_long_context_tcgen05_gb300 as cq
    with pytest.raises(cq.CqsaError):
        cq.cqsa_debug_set_fault(7)


def test_streamed_backward_reports_a_wait_that_gave_up():
    """The host-resident backward reads the backward's device error word after its stream drains: a
    kernel whose bounded wait gave up (the hook skips block 0's key/value load) makes the call return
    CQSA_ERR_TIMEOUT instead of incomplete gradients; the next call, without the hook, is correct."""
    import exact_long_context_tcgen05_gb300 as cq
    B, H, N, d, C = 1, 2, 512, 64, 256
    qn, kn, vn = syn.qkv(B, H, N, d, seed=33)
    gn = syn.normal(B, H, N, d, seed=33, tensor_id=syn.TID_DO)
    q, k, v, g = (to_dev(x, syn.F16) for x in (qn, kn, vn, gn))
    out, lse = mono(cq, q, k, v, B, H, N, d, False, syn.F16)
    host = [t.cpu().pin_memory() for t in (q, k, v, out, g, lse)]
    grads = [torch.empty((B, H, N, d), dtype=torch.float16).pin_memory() for _ in range(3)]
    assert cq.cqsa_device_error(clear=True)[0] == cq.CQSA_OK
    cq.cqsa_set_timeout_ms(200)
    try:
        cq.cqsa_debug_set_fault(2)
        with pytest.raises(cq.CqsaError) as ei:
            cq.cqsa_stream_attn_bwd(*host, *grads, B, H, N, d, False, 0.0, cq.CQSA_F16, C)
        assert ei.value.status == cq.CQSA_ERR_TIMEOUT and "gave up" in str(ei.value)
    finally:
        cq.cqsa_debug_set_fault(0)
        cq.cqsa_set_timeout_ms(0)
    assert cq.cqsa_device_error(clear=True)[0] == cq.CQSA_OK  # the call cleared the word it reported
    cq.cqsa_stream_attn_bwd(*host, *grads, B, H, N, d, False, 0.0, cq.CQSA_F16, C)
    ref = cq.attention_backward(q, k, v, out, g, lse, causal=False)
    torch.cuda.synchronize()
    for got, r in zip(grads, ref):
        e = (got.float() - r.cpu().float()).abs().max().item()
        assert e <= 8 * 2.0 ** -11 * r.float().abs().max().item()
