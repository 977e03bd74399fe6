"""Sequence-sharded causal forward and backward on the CUDA path.

A causal sequence cut into consecutive shards needs one exchange per direction
(paperlayer.ai summary §3.3 / §3.3.1: a prefix recurrence forward, cumulative
sums in opposite directions backward): the exclusive prefix of the shards' own
(S, Z) sums for the forward and for dq, and the exclusive suffix of their own
reverse sums (R, r) for dk and dv. Here the shards are run one after another in
one process (the exchange is a sum over torch tensors), with ragged shard
lengths that take every kernel path: shards of one token, of one chunk
(<= 128 tokens), and of several segments; the concatenated results must match
the fp64 oracle over the whole sequence. tests/test_shard_dist_gpu.py runs the
same exchange between two processes with torch.distributed (gloo).
"""

import numpy as np
import pytest

import oracle
from kernelized_causal_self_gb300 import inputs
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"


@pytest.fixture(scope="module")
def la():
    from kernelized_causal_self_gb300 import build
    build.build()
    import kernelized_causal_self_gb300 as pkg
    pkg.load_library()
    return pkg


def run_shards(la, tq, tk, tv, tg, cuts):
    """Forward and backward of the sequence cut at `cuts`, shard by shard. Returns
    (out, dq, dk, dv) concatenated over the shards, and each shard's own (S, Z)."""
    sl = [slice(a, b) for a, b in zip(cuts[:-1], cuts[1:])]
    part = [[t[:, :, s].contiguous() for t in (tq, tk, tv, tg)] for s in sl]
    own = [la.la_state_sums(k, v) for _, k, v, _ in part]            # exchange 1: (S_r, Z_r)
    pre = []
    S0, Z0 = torch.zeros_like(own[0][0]), torch.zeros_like(own[0][1])
    for S_r, Z_r in own:
        pre.append((S0.clone(), Z0.clone()))
        S0, Z0 = S0 + S_r, Z0 + Z_r
    outs = [la.la_forward_shard(q, k, v, *p) for (q, k, v, _), p in zip(part, pre)]
    first = [la.la_backward_shard_q(q, k, v, g, *p) for (q, k, v, g), p in zip(part, pre)]
    suf = [None] * len(part)                                          # exchange 2: (R_r, r_r)
    R0, r0 = torch.zeros_like(first[0][1]), torch.zeros_like(first[0][2])
    for i in range(len(part) - 1, -1, -1):
        suf[i] = (R0.clone(), r0.clone())
        R0, r0 = R0 + first[i][1], r0 + first[i][2]
    second = [la.la_backward_shard_kv(q, k, v, g, *suf[i], first[i][3])
              for i, (q, k, v, g) in enumerate(part)]
    torch.cuda.synchronize()
    cat = lambda ts: torch.cat(ts, dim=2).float().cpu().numpy()  # noqa: E731
    return (cat(outs), cat([f[0] for f in first]), cat([s[0] for s in second]),
            cat([s[1] for s in second]), own)


CASES = [
    ("bf16", 2, 3, 64, 64, [0, 700, 737, 1737, 1738]),   # multi-segment, one chunk, one token
    ("bf16", 1, 2, 64, 64, [0, 128, 256, 1300]),          # shards on chunk boundaries
    ("f32", 1, 2, 32, 48, [0, 50, 120, 123]),             # the CUDA-core path
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-d{c[3]}m{c[4]}-{len(c[5]) - 1}shards")
def test_shards_reproduce_the_unsharded_forward_and_backward(la, case):
    dt, B, H, D, M, cuts = case
    scale = 0.125 if dt == inputs.BF16 else 1.0
    N = cuts[-1]
    q, k, v = inputs.qkv(950 + N, B, H, N, D, M, scale, dt)
    g = inputs.upstream_grad(950 + N, B, H, N, M, scale, dt)
    tq, tk, tv, tg = (inputs.to_torch(x, dt, DEV) for x in (q, k, v, g))
    out, dq, dk, dv, own = run_shards(la, tq, tk, tv, tg, cuts)
    assert_close(out, oracle.forward(q, k, v, True), dt, "sharded out")
    wq, wk, wv = oracle.backward(q, k, v, g, True)
    for name, got, want in (("dq", dq, wq), ("dk", dk, wk), ("dv", dv, wv)):
        assert_close(got, want, dt, f"sharded {name}")
    for (S_r, Z_r), a, b in zip(own, cuts[:-1], cuts[1:]):   # each shard's own sums
        _, S_ref, Z_ref = oracle.linearized_attention(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b])
        assert_close(S_r.cpu().numpy(), S_ref, dt, f"S of shard [{a}, {b})")
        assert_close(Z_r.cpu().numpy(), Z_ref, dt, f"Z of shard [{a}, {b})")


def test_forward_shard_leaves_its_initial_state_alone(la):
    B, H, N = 1, 2, 300
    q, k, v = inputs.qkv(960, B, H, N, 64, 64, 0.125, inputs.BF16)
    S0 = torch.rand((B, H, 64, 64), device=DEV) * 4.0
    Z0 = torch.rand((B, H, 64), device=DEV) * 4.0 + 1.0
    S_keep, Z_keep = S0.clone(), Z0.clone()
    out = la.la_forward_shard(*(inputs.to_torch(x, inputs.BF16, DEV) for x in (q, k, v)), S0, Z0)
    torch.cuda.synchronize()
    assert torch.equal(S0, S_keep) and torch.equal(Z0, Z_keep)
    want, _, _ = oracle.recurrent_attention(q, k, v, S0.cpu().numpy(), Z0.cpu().numpy())
    assert_close(out.float().cpu().numpy(), want, "bf16", "out from a given state")


def test_empty_shard_adds_nothing(la):
    """A shard with no tokens: zero state sums and zero reverse sums."""
    e = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device=DEV)
    S, Z = la.la_state_sums(e, e)
    z4, z3 = torch.zeros((1, 2, 64, 64), device=DEV), torch.zeros((1, 2, 64), device=DEV)
    _, R, r, _ = la.la_backward_shard_q(e, e, e, e, z4, z3)
    torch.cuda.synchronize()
    for t in (S, Z, R, r):
        assert float(t.abs().max()) == 0.0
