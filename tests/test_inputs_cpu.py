"""The seeded input module shared by the oracle side and the CUDA side (CPU only).

Both sides must see identical bits: bf16 inputs are drawn in float32, rounded to
the bf16 grid by ``inputs.bf16_round`` (round to nearest, ties to even) for the
oracle, and handed to the library as the same bit patterns by ``inputs.to_torch``.
"""

import numpy as np
import torch

from kernelized_causal_self_gb300 import inputs


def _torch_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_bf16_round_matches_torch_conversion():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200_000).astype(np.float32) * np.float32(s)
                        for s in (1e-30, 1e-3, 0.125, 1.0, 1e3, 1e30)])
    special = np.array([
        0.0, -0.0, np.inf, -np.inf, np.nan,
        1.0 + 2.0 ** -8,        # halfway between 1 and 1 + 2^-7: ties to even (1)
        1.0 + 3 * 2.0 ** -8,    # halfway between 1 + 2^-7 and 1 + 2^-6: ties to even (1 + 2^-6)
        -(1.0 + 2.0 ** -8), 1.0 + 2.0 ** -9,
        3.4028235e38,           # float32 max: past the last bf16 halfway point, so +inf
        3.3895314e38,           # bf16 max
        1e-40, -1e-40, 1.4e-45,  # float32 subnormals
    ], dtype=np.float32)
    x = np.concatenate([x, special])
    got, want = inputs.bf16_round(x), _torch_bf16(x)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_to_torch_keeps_the_bits():
    x = inputs.normal(5, (3, 4, 70, 16), 0.125, inputs.BF16)
    t = inputs.to_torch(x, inputs.BF16, "cpu")
    assert t.dtype == torch.bfloat16 and tuple(t.shape) == x.shape
    assert np.array_equal(t.float().numpy().view(np.uint32), x.view(np.uint32))
    f = inputs.to_torch(x, inputs.F32, "cpu")
    assert f.dtype == torch.float32 and np.array_equal(f.numpy(), x)


def test_draws_are_seeded_and_streams_differ():
    a = inputs.qkv(11, 2, 3, 50, 8, 8, 0.125, inputs.BF16)
    b = inputs.qkv(11, 2, 3, 50, 8, 8, 0.125, inputs.BF16)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    q, k, v = a
    assert not np.array_equal(q, k) and not np.array_equal(q[..., :8], v)
    assert not np.array_equal(q, inputs.qkv(12, 2, 3, 50, 8, 8, 0.125, inputs.BF16)[0])
    assert np.array_equal(inputs.bf16_round(q), q)  # already on the bf16 grid
    assert abs(float(np.std(inputs.normal(3, (200_000,), 0.125))) - 0.125) < 2e-3


def test_stream_lengths_are_seeded_and_in_range():
    a = inputs.stream_lengths(930, 256, 1, 1024)
    b = inputs.stream_lengths(930, 256, 1, 1024)
    assert a.dtype == np.int32 and a.shape == (256,)
    assert np.array_equal(a, b)
    assert a.min() >= 1 and a.max() <= 1024
    assert not np.array_equal(a, inputs.stream_lengths(931, 256, 1, 1024))
    assert np.all(inputs.stream_lengths(5, 64, 7, 7) == 7)
