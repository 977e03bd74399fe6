"""Seeded synthetic inputs and the named workloads.

This module holds no arithmetic of the attention method: only random draws,
the fixed input scale, and round-to-nearest-even conversion of float32 to
bfloat16 so that the CUDA path and the fp64 oracle see bit-identical inputs.
It imports neither the CUDA binding nor the oracle.

Workloads stand in for the paper's settings (autoregressive image generation
over pixel sequences of length 784 / 3072, the synthetic fwd/bwd benchmark up
to N = 16384, and many-stream recurrent generation); every tensor is i.i.d.
normal, scaled by 1/sqrt(64) for the bf16 cases.
"""

from dataclasses import dataclass

import numpy as np

F32, BF16 = "f32", "bf16"


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str          # "fwd", "fwdbwd" or "decode"
    causal: bool
    B: int             # batch (decode: number of independent streams)
    H: int
    N: int             # sequence length (decode: prefill length)
    D: int
    M: int
    dtype: str
    scale: float       # inputs are N(0, 1) * scale
    seed: int
    steps: int = 0     # decode steps after the prefill


WORKLOADS = {
    w.name: w
    for w in (
        Workload("causal_fwd_f32_b1h1n64d32", "fwd", True, 1, 1, 64, 32, 32, F32, 1.0, 0),
        Workload("noncausal_fwd_b4h8n4096d64", "fwd", False, 4, 8, 4096, 64, 64, BF16, 0.125, 1),
        Workload("causal_fwd_b8h8n3072d64", "fwd", True, 8, 8, 3072, 64, 64, BF16, 0.125, 2),
        Workload("causal_fwdbwd_b4h8n16384d64", "fwdbwd", True, 4, 8, 16384, 64, 64, BF16, 0.125, 3),
        Workload("decode_s256h8d64_prefill1024_steps3072", "decode", True, 256, 8, 1024, 64, 64,
                 BF16, 0.125, 4, steps=3072),
    )
}


def bf16_round(x):
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    rounded = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32)


def bf16_bits(x):
    """uint16 bit patterns of float32 values that are already bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def normal(seed, shape, scale=1.0, dtype=F32, stream=0):
    """i.i.d. N(0, 1) * scale from PCG64(seed, stream), rounded to `dtype`'s grid.

    Returned as float32 (bf16 values are exactly representable in float32), so the
    oracle can upcast to float64 without any further rounding.
    """
    rng = np.random.Generator(np.random.PCG64([seed, stream]))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x = (x * np.float32(scale)).astype(np.float32)
    return bf16_round(x) if dtype == BF16 else x


def uniform(seed, shape, lo, hi, stream=0):
    """i.i.d. uniform on [lo, hi) from PCG64(seed, stream), float32."""
    rng = np.random.Generator(np.random.PCG64([seed, stream]))
    return (lo + (hi - lo) * rng.random(size=shape)).astype(np.float32)


def qkv(seed, B, H, N, D, M, scale=1.0, dtype=F32):
    """q, k: [B, H, N, D]; v: [B, H, N, M]; drawn in that order (streams 0, 1, 2)."""
    q = normal(seed, (B, H, N, D), scale, dtype, stream=0)
    k = normal(seed, (B, H, N, D), scale, dtype, stream=1)
    v = normal(seed, (B, H, N, M), scale, dtype, stream=2)
    return q, k, v


def upstream_grad(seed, B, H, N, M, scale=1.0, dtype=F32):
    """dout: [B, H, N, M] (stream 3)."""
    return normal(seed, (B, H, N, M), scale, dtype, stream=3)


def decode_tokens(seed, steps, S, H, D, M, scale=1.0, dtype=F32):
    """Per-step q, k: [steps, S, H, D]; v: [steps, S, H, M] (streams 4, 5, 6)."""
    q = normal(seed, (steps, S, H, D), scale, dtype, stream=4)
    k = normal(seed, (steps, S, H, D), scale, dtype, stream=5)
    v = normal(seed, (steps, S, H, M), scale, dtype, stream=6)
    return q, k, v


def stream_lengths(seed, B, lo, hi, stream=7):
    """B stream lengths, i.i.d. uniform integers in [lo, hi] (a serving batch's mix)."""
    rng = np.random.Generator(np.random.PCG64([seed, stream]))
    return rng.integers(lo, hi + 1, size=B).astype(np.int32)


def to_torch(x, dtype, device):
    """float32 numpy array (on `dtype`'s grid) -> torch tensor of that dtype."""
    import torch
    if dtype == BF16:
        t = torch.from_numpy(bf16_bits(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device)


def torch_normal(gen, shape, scale, dtype, device):
    """Device-side draw for large benchmark inputs: N(0,1)*scale, rounded to dtype."""
    import torch
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16) if dtype == BF16 else x
