"""Pins for the seeded input generator (no attention arithmetic here)."""
import numpy as np
import pytest
import torch

import synthetic as syn


def test_splitmix64_published_sequence():
    # The first outputs of SplitMix64 seeded with 1234567, the test sequence that accompanies
    # Vigna's public-domain reference implementation (splitmix64.c) and many ports of it.
    assert [syn.sm64_at(1234567, n) for n in range(5)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_normal_moments_and_ks():
    from scipy import stats
    z = syn.normal(1, 1, 4096, 64, dtype=syn.F32).ravel().astype(np.float64)
    assert abs(z.mean()) < 0.01
    assert abs(z.var() - 1.0) < 0.01
    assert stats.kstest(z, "norm").pvalue > 1e-3
    # the cos and sin halves of each Box-Muller pair are uncorrelated
    assert abs(np.corrcoef(z[0::2], z[1::2])[0, 1]) < 0.01


def test_fp16_rounding_matches_numpy():
    z = syn.normal(1, 2, 256, 64, dtype=syn.F32)
    bits = syn.normal(1, 2, 256, 64, dtype=syn.F16)
    assert np.array_equal(bits, z.astype(np.float16).view(np.uint16))
    edge = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e-8, 2.0**-25, 2.0**-24, 3 * 2.0**-26,
                     5.960464477539063e-08 * 1.5, 6.1e-5, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11, -2.5],
                    dtype=np.float32)
    assert np.array_equal(syn.f32_to_f16_bits(edge), edge.astype(np.float16).view(np.uint16))


def test_bf16_rounding_matches_torch():
    z = syn.normal(1, 2, 256, 64, dtype=syn.F32, mul=3.0)
    bits = syn.normal(1, 2, 256, 64, dtype=syn.BF16, mul=3.0)
    ref = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)


def test_chunks_and_layouts_are_slices_of_the_whole():
    B, H, N, d = 2, 3, 300, 8
    full = syn.normal(B, H, N, d, tensor_id=1)
    part = syn.normal(B, H, N, d, tensor_id=1, n0=100, n_cnt=77)
    assert np.array_equal(part, full[:, :, 100:177])
    tm = syn.normal(B, H, N, d, tensor_id=1, layout=syn.LAYOUT_BNHD)
    assert np.array_equal(tm, full.transpose(0, 2, 1, 3))
    tm_part = syn.normal(B, H, N, d, tensor_id=1, layout=syn.LAYOUT_BNHD, n0=5, n_cnt=40)
    assert np.array_equal(tm_part, tm[:, 5:45])


def test_streams_differ_and_repeat():
    a = syn.normal(1, 1, 64, 64, tensor_id=0)
    b = syn.normal(1, 1, 64, 64, tensor_id=1)
    assert not np.array_equal(a, b)
    assert np.array_equal(a, syn.normal(1, 1, 64, 64, tensor_id=0))
    assert not np.array_equal(a, syn.normal(1, 1, 64, 64, tensor_id=0, seed=1))


def test_sample_rows():
    rows = syn.sample_rows(2, 4, 5000, 300, chunk=1024)
    assert rows.shape[1] == 3 and len(rows) >= 300
    assert rows[:, 0].max() < 2 and rows[:, 1].max() < 4 and rows[:, 2].max() < 5000
    assert len(np.unique(rows, axis=0)) == len(rows)
    for i in (0, 1, 127, 128, 4999, 1023, 1024, 4095, 4096):
        assert ((rows[:, 0] == 0) & (rows[:, 1] == 0) & (rows[:, 2] == i)).any()
    assert np.array_equal(rows, syn.sample_rows(2, 4, 5000, 300, chunk=1024))


def test_bad_ranges_rejected():
    with pytest.raises(ValueError):
        syn.normal(1, 1, 10, 8, n0=5, n_cnt=6)
    with pytest.raises(ValueError):
        syn.normal(1, 1, 10, 0)
