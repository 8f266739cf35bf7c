"""Helpers shared by the GPU parity tests: seeded inputs to the device, calls through the C ABI."""
import numpy as np
import torch

import synthetic as syn

TORCH_DT = {syn.F16: torch.float16, syn.BF16: torch.bfloat16}


def to_dev(bits: np.ndarray, dtype: int) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH_DT[dtype]).cuda()


def to_np64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def mono(cq, q, k, v, B, H, N, d, causal, dtype, scale=0.0):
    """Device q/k/v -> (out tensor, lse tensor) via cqsa_attn_fwd."""
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    cq.cqsa_attn_fwd(q, k, v, out, lse, B, H, N, d, causal, scale, dtype)
    return out, lse


def chunk(cq, q, k, v, q_off, kv_off, B, H, Nq, Nkv, d, causal, dtype, O=None, L=None, accumulate=False, scale=0.0):
    if O is None:
        O = torch.empty((B, H, Nq, d), dtype=torch.float32, device=q.device)
        L = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    cq.cqsa_attn_fwd_chunk(q, k, v, q_off, kv_off, B, H, Nq, Nkv, d, causal, scale, dtype, O, L, accumulate)
    return O, L


def errs(got: np.ndarray, ref: np.ndarray):
    e = np.abs(got - ref)
    return float(e.max()), float(e.mean())


def assert_close(out, ref_o, lse=None, ref_l=None, max_abs=4e-3, mean_abs=2e-4, lse_abs=1e-3, what=""):
    mx, mn = errs(out, ref_o)
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max abs {mx:.3e} (<= {max_abs}), mean abs {mn:.3e} (<= {mean_abs})"
    if lse is not None:
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(lse), fin), f"{what}: -inf rows differ"
        if fin.any():
            le = float(np.abs(lse[fin] - ref_l[fin]).max())
            assert le <= lse_abs, f"{what}: lse max abs {le:.3e} (<= {lse_abs})"
    return mx, mn


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def assert_bf16_rounds_fp32_result(got: np.ndarray, o32: np.ndarray, what: str, rel_row: float = 1e-5):
    """A bf16 output of a path whose fp32 result is not exposed, against the fp32 result of the same
    attention by another route (o32; the two fp32 results may differ by the chunked-vs-monolithic
    tolerance, rel_row times the row's largest |O|): each element must be the round-to-nearest-even
    bf16 value of some number within that tolerance of o32, i.e. within half a bf16 ulp of the output
    plus the tolerance."""
    tol = 0.5 * bf16_ulp(got) + rel_row * np.abs(o32).max(axis=-1, keepdims=True)
    excess = np.abs(got - o32) - tol
    assert np.all(excess <= 0), f"{what}: bf16 output off the fp32 result by {excess.max():.3e} beyond tolerance"
