"""Failure detection on the GPU without a GPU fault.

Every wait inside the tensor-core kernels is bounded. These tests make one such
wait run out on purpose through the library's test hooks: CTA 0 of the main
kernel skips issuing one of its TMA loads (nothing is copied, so the barrier it
would have completed never does) and bounds its waits by 100 us. The kernel
must then return on its own, the workspace status must say LA_ERR_TIMEOUT at
the load-wait site, and the next ordinary call on the same context must still
match the fp64 oracle. Nothing here traps, faults or hangs the GPU: the wait
that runs out is a bounded poll, and the winding-down waits (for the copies and
MMAs that were issued) complete normally.
"""

import ctypes
import time

import pytest

import oracle
from kernelized_causal_self_gb300 import inputs
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
LIMIT_NS = 100_000  # 100 us


@pytest.fixture(scope="module")
def la():
    from kernelized_causal_self_gb300 import build
    build.build()
    import kernelized_causal_self_gb300 as pkg
    pkg.load_library()
    return pkg


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _case():
    # 8 chunks in 2 sequences; the hooks withhold CTA 0's first load (load 0), which
    # every segment layout gives it
    B, H, N = 1, 2, 1000
    q, k, v = inputs.qkv(901, B, H, N, 64, 64, 0.125, inputs.BF16)
    g = inputs.upstream_grad(901, B, H, N, 64, 0.125, inputs.BF16)
    return (B, H, N), (q, k, v, g)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_fused_forward_load_wait_runs_out_and_the_cluster_finishes(la, causal):
    """The one-launch forward (a thread-block cluster per sequence; this shape has 8
    segments of one chunk): CTA 0 withholds its first load, the one of its segment-sum
    phase, so its wait runs out after 100 us; it still reaches both of its cluster's
    barriers, so the kernel returns on its own, the status names the site, and the next
    ordinary call is exact."""
    (B, H, N), (q, k, v, g) = _case()
    tq, tk, tv = (inputs.to_torch(x, inputs.BF16, DEV) for x in (q, k, v))
    out = torch.empty_like(tv)
    nbytes = la.la_forward_workspace_bytes(B, H, N, 64, 64, causal, la.LA_BF16)
    ws = torch.empty((nbytes,), dtype=torch.uint8, device=DEV)
    lib = la.load_library()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    rc = lib.la_debug_forward_fused_fault(_p(tq), _p(tk), _p(tv), _p(out), B, H, N, 64, 64,
                                          int(causal), la.LA_BF16, _p(ws), nbytes, 0, LIMIT_NS, st)
    assert rc == la.LA_OK
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.0          # returned on its own, well inside 2 s
    assert la.la_workspace_wait_site(ws) == la.LA_SITE_FORWARD_FUSED_LOAD
    assert la.la_workspace_status(ws) == la.LA_ERR_TIMEOUT
    assert la.la_workspace_status(ws) == la.LA_OK   # read and cleared
    la.la_forward(tq, tk, tv, causal=causal, out=out, workspace=ws)
    assert la.la_workspace_status(ws) == la.LA_OK
    assert_close(out.float().cpu().numpy(), oracle.forward(q, k, v, causal), "bf16", "out after")


def test_forward_load_wait_runs_out_and_the_next_call_is_exact(la):
    (B, H, N), (q, k, v, g) = _case()
    tq, tk, tv = (inputs.to_torch(x, inputs.BF16, DEV) for x in (q, k, v))
    out = torch.empty_like(tv)
    nbytes = la.la_forward_workspace_bytes(B, H, N, 64, 64, True, la.LA_BF16)
    ws = torch.empty((nbytes,), dtype=torch.uint8, device=DEV)
    lib = la.load_library()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    rc = lib.la_debug_forward_fault(_p(tq), _p(tk), _p(tv), _p(out), B, H, N, 64, 64, 1,
                                    la.LA_BF16, _p(ws), nbytes, 0, LIMIT_NS, st)
    assert rc == la.LA_OK
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.0          # returned on its own, well inside 2 s
    assert la.la_workspace_wait_site(ws) == la.LA_SITE_FORWARD_LOAD
    assert la.la_workspace_status(ws) == la.LA_ERR_TIMEOUT
    assert la.la_workspace_status(ws) == la.LA_OK   # read and cleared
    # the same context, workspace and buffers: an ordinary call is exact again
    la.la_forward(tq, tk, tv, causal=True, out=out, workspace=ws)
    assert la.la_workspace_status(ws) == la.LA_OK
    assert_close(out.float().cpu().numpy(), oracle.forward(q, k, v, True), "bf16", "out after")


def test_backward_load_wait_runs_out_and_the_next_call_is_exact(la):
    (B, H, N), (q, k, v, g) = _case()
    tq, tk, tv, tg = (inputs.to_torch(x, inputs.BF16, DEV) for x in (q, k, v, g))
    dq, dk, dv = (torch.empty(tq.shape, dtype=torch.float32, device=DEV) for _ in range(3))
    nbytes = la.la_backward_workspace_bytes(B, H, N, 64, 64, True, la.LA_BF16)
    ws = torch.empty((nbytes,), dtype=torch.uint8, device=DEV)
    lib = la.load_library()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    rc = lib.la_debug_backward_fault(_p(tq), _p(tk), _p(tv), _p(tg), _p(dq), _p(dk), _p(dv),
                                     B, H, N, 64, 64, 1, la.LA_BF16, _p(ws), nbytes, 0, LIMIT_NS,
                                     st)
    assert rc == la.LA_OK
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.0
    assert la.la_workspace_wait_site(ws) == la.LA_SITE_BACKWARD_LOAD
    assert la.la_workspace_status(ws) == la.LA_ERR_TIMEOUT
    la.la_backward(tq, tk, tv, tg, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
    assert la.la_workspace_status(ws) == la.LA_OK
    wq, wk, wv = oracle.backward(q, k, v, g, True)
    for name, got, want in (("dq", dq, wq), ("dk", dk, wk), ("dv", dv, wv)):
        assert_close(got.cpu().numpy(), want, "bf16", f"{name} after")


def test_hook_without_a_withheld_load_changes_nothing(la):
    """A load number past the last one CTA 0 issues: nothing is withheld, the call
    completes with LA_OK and exact outputs although its waits are bounded by 100 us."""
    (B, H, N), (q, k, v, g) = _case()
    tq, tk, tv = (inputs.to_torch(x, inputs.BF16, DEV) for x in (q, k, v))
    out = torch.empty_like(tv)
    nbytes = la.la_forward_workspace_bytes(B, H, N, 64, 64, True, la.LA_BF16)
    ws = torch.empty((nbytes,), dtype=torch.uint8, device=DEV)
    lib = la.load_library()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.la_debug_forward_fault(_p(tq), _p(tk), _p(tv), _p(out), B, H, N, 64, 64, 1,
                                    la.LA_BF16, _p(ws), nbytes, 1000, 1_000_000, st)
    assert rc == la.LA_OK
    assert la.la_workspace_status(ws) == la.LA_OK
    assert la.la_workspace_wait_site(ws) == 0
    assert_close(out.float().cpu().numpy(), oracle.forward(q, k, v, True), "bf16", "out")
