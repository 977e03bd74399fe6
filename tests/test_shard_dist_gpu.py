"""Two ranks, one sequence: the sharded causal forward and backward with the
exchanges done by torch.distributed (gloo, host tensors).

Rank r holds tokens [r N/2, (r+1) N/2) of every (b, h) sequence and runs the
library's CUDA kernels on cuda:0 (the ranks share the one GPU; no kernel of
one waits on the other's). Exchange 1 all-gathers each shard's own (S, Z)
sums, and rank r starts from the sum over the ranks before it; exchange 2
all-gathers each shard's own reverse sums (R, r) after the first backward pass,
and rank r continues with the sum over the ranks after it. Each exchange moves
D*M + D float32 per head per rank. The gathered outputs and gradients must match
the fp64 oracle over the whole sequence.
"""

import os
import socket

import pytest

import oracle
from kernelized_causal_self_gb300 import inputs
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

B, H, N, D, M, SEED = 2, 3, 1500, 64, 64, 970


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import kernelized_causal_self_gb300 as la
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        xq, xk, xv = inputs.qkv(SEED, B, H, N, D, M, 0.125, inputs.BF16)
        xg = inputs.upstream_grad(SEED, B, H, N, M, 0.125, inputs.BF16)
        lo, hi = rank * N // world, (rank + 1) * N // world
        tq, tk, tv, tg = (inputs.to_torch(x[:, :, lo:hi], inputs.BF16, dev) for x in (xq, xk, xv, xg))

        def gather(*ts):
            flat = torch.cat([t.reshape(-1) for t in ts]).cpu()
            parts = [torch.empty_like(flat) for _ in range(world)]
            dist.all_gather(parts, flat)
            return parts

        def split(flat):
            n = B * H * D * M
            return (flat[:n].reshape(B, H, D, M).to(dev), flat[n:].reshape(B, H, D).to(dev))

        S_r, Z_r = la.la_state_sums(tk, tv)
        parts = gather(S_r, Z_r)                                   # exchange 1
        S0, Z0 = split(sum(parts[:rank], torch.zeros_like(parts[0])))
        out = la.la_forward_shard(tq, tk, tv, S0, Z0)
        dq, R_r, r_r, ws = la.la_backward_shard_q(tq, tk, tv, tg, S0, Z0)
        parts = gather(R_r, r_r)                                   # exchange 2
        R0, r0 = split(sum(parts[rank + 1:], torch.zeros_like(parts[0])))
        dk, dv = la.la_backward_shard_kv(tq, tk, tv, tg, R0, r0, ws)
        torch.cuda.synchronize()
        q.put((rank, [t.float().cpu().numpy() for t in (out, dq, dk, dv)]))
    finally:
        dist.destroy_process_group()


def test_two_ranks_exchange_prefix_and_suffix_sums():
    import numpy as np
    import torch.multiprocessing as mp
    from kernelized_causal_self_gb300 import build
    build.build()
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=300) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out, dq, dk, dv = (np.concatenate([g[1][i] for g in got], axis=2) for i in range(4))
    xq, xk, xv = inputs.qkv(SEED, B, H, N, D, M, 0.125, inputs.BF16)
    xg = inputs.upstream_grad(SEED, B, H, N, M, 0.125, inputs.BF16)
    assert_close(out, oracle.forward(xq, xk, xv, True), "bf16", "two-rank out")
    wq, wk, wv = oracle.backward(xq, xk, xv, xg, True)
    for name, g, w in (("dq", dq, wq), ("dk", dk, wk), ("dv", dv, wv)):
        assert_close(g, w, "bf16", f"two-rank {name}")
