"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks.

The path shards into independent replicas (no collective on the data path);
what bench.py does across ranks is a barrier around the timed region and the
maximum of the ranks' times. These run here with the gloo backend.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(0, 2.5), (1, 2.5)]


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1, None) == 3.25


def _shard_worker(rank, world, port, q):
    """Rank r holds tokens [r N / world, (r + 1) N / world) of every (b, h) sequence."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import numpy as np

    import oracle
    from kernelized_causal_self_gb300 import inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H, N, D, M = 2, 2, 90, 8, 6
        xq, xk, xv = inputs.qkv(21, B, H, N, D, M, 0.5, inputs.F32)
        lo, hi = rank * N // world, (rank + 1) * N // world
        sq, sk, sv = xq[:, :, lo:hi], xk[:, :, lo:hi], xv[:, :, lo:hi]
        # the one exchange: every shard's own sums (S_r, Z_r), all-gathered
        _, S_r, Z_r = oracle.linearized_attention(sq, sk, sv)
        packed = torch.from_numpy(np.concatenate([S_r.reshape(-1), Z_r.reshape(-1)]))
        parts = [torch.empty_like(packed) for _ in range(world)]
        dist.all_gather(parts, packed)
        # the exclusive prefix over the shards before this one is the state it starts from
        pre = sum((parts[r].numpy() for r in range(rank)), np.zeros_like(packed.numpy()))
        S0 = pre[: B * H * D * M].reshape(B, H, D, M)
        Z0 = pre[B * H * D * M:].reshape(B, H, D)
        out, _, _ = oracle.recurrent_attention(sq, sk, sv, S0=S0, Z0=Z0)
        q.put((rank, out, oracle.forward(xq, xk, xv, True)[:, :, lo:hi]))
    finally:
        dist.destroy_process_group()


def test_sequence_shards_with_an_exclusive_state_prefix_equal_the_causal_forward():
    """Sequence sharding needs one exchange: the exclusive prefix over the shards'
    (S, Z) sums. Two gloo ranks, each holding half of every sequence, reproduce the
    unsharded causal forward (fp64 oracle on both sides)."""
    import numpy as np
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=120) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, out, want in got:
        np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-13)
    # the prefix matters: the second half run from a zero state is far from the truth
    import oracle
    from kernelized_causal_self_gb300 import inputs
    xq, xk, xv = inputs.qkv(21, 2, 2, 90, 8, 6, 0.5, inputs.F32)
    alone = oracle.recurrent_attention(xq[:, :, 45:], xk[:, :, 45:], xv[:, :, 45:])[0]
    assert np.max(np.abs(alone - got[1][2])) > 1e-2


# The stand-in for bench.py's step used below: the same rank set-up, barrier and
# max over ranks that run_ours uses, with no GPU work in between.
_STUB_STEP = '''
import json, sys
sys.path.insert(0, {root!r})
import torch
import bench
world, rank, local = bench.dist_setup(None)
bench.barrier(world)
t = bench.max_over_ranks(1.0 + rank, world, torch.device("cpu"))
if rank == 0:
    print(json.dumps({{"n_gpus": world, "ms": t, "local_rank": local}}), flush=True)
bench.barrier(world)
if world > 1:
    import torch.distributed as dist
    dist.destroy_process_group()
'''


def test_gpus_flag_starts_one_replica_per_gpu(tmp_path, capfd):
    """bench.py --gpus 2 outside torchrun starts two ranks itself (RANK, LOCAL_RANK,
    WORLD_SIZE, 127.0.0.1 rendezvous); they meet in the barrier and the max over
    ranks, and rank 0 alone prints, with n_gpus = 2."""
    import json

    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    stub = tmp_path / "stub_step.py"
    stub.write_text(_STUB_STEP.format(root=root))
    assert bench.launch_replicas(2, ["--gpus", "2"], script=str(stub)) == 0
    lines = [ln for ln in capfd.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    got = json.loads(lines[0])
    assert got == {"n_gpus": 2, "ms": 2.0, "local_rank": 0}


def test_gpus_flag_refuses_more_gpus_than_visible(monkeypatch):
    import sys

    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "2"])
    monkeypatch.setattr(torch.cuda, "device_count", lambda: 1)
    started = []
    monkeypatch.setattr(bench, "launch_replicas", lambda *a, **k: started.append(a) or 0)
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert "only 1 CUDA device" in str(e.value.code) and not started
    monkeypatch.setattr(torch.cuda, "device_count", lambda: 2)
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert e.value.code == 0 and started == [(2, ["--gpus", "2"])]
