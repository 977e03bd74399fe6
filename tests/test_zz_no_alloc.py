"""la_forward_noalloc: the forward for callers that cannot allocate device memory.

Such callers only receive device pointers for their inputs and outputs (the
application or framework around them owns the allocator), so they cannot hand
la_forward a workspace. la_forward_noalloc runs the same computation with its
scratch in a fixed array inside the library's device memory. These tests call
it through the C ABI and compare it with the fp64 oracle and with la_forward
(caller workspace) on two calls in a row; check that a shape needing more
scratch than the array holds is refused before anything is launched, that a
successful call allocates nothing and launches exactly la_forward's kernels,
and that the array's status word is read and cleared by
la_forward_noalloc_status. This file is collected last, so a run that stops at
the first failure has run every other test before it.
"""

import ctypes

import pytest

import oracle
from kernelized_causal_self_gb300 import inputs
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    from kernelized_causal_self_gb300 import build
    build.build()
    import kernelized_causal_self_gb300 as pkg
    torch.cuda.set_device(0)  # the device the pointers and the stream belong to, made current
    return pkg


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(pkg, q, k, v, out, causal):
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = pkg.LA_BF16 if q.dtype == torch.bfloat16 else pkg.LA_F32
    return pkg.load_library().la_forward_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), B, H, N, D, M, int(causal), dt, _stream())


CASES = [
    (2, 3, 700, 64, 64, inputs.BF16, True),
    (2, 3, 700, 64, 64, inputs.BF16, False),
    (4, 8, 3072, 64, 64, inputs.BF16, True),
    (1, 2, 129, 32, 32, inputs.F32, True),
]
IDS = ["bf16-causal", "bf16-noncausal", "bf16-causal-b4h8n3072", "f32-causal"]


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_noalloc_matches_oracle_and_la_forward_twice(lib, case):
    B, H, N, D, M, dtype, causal = case
    scale = 0.125 if dtype == inputs.BF16 else 1.0
    q, k, v = inputs.qkv(77, B, H, N, D, M, scale, dtype)
    tq, tk, tv = (inputs.to_torch(x, dtype, DEV) for x in (q, k, v))
    ref = lib.la_forward(tq, tk, tv, causal=causal)
    torch.cuda.synchronize()
    got_ref = ref.float().cpu().numpy()
    want = oracle.forward(q, k, v, causal)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(lib, tq, tk, tv, out, causal) == lib.LA_OK
        torch.cuda.synchronize()
        assert lib.la_forward_noalloc_status() == lib.LA_OK
        got = out.float().cpu().numpy()
        assert_close(got, want, dtype, "la_forward_noalloc vs the oracle")
        assert_close(got, got_ref, dtype, "la_forward_noalloc vs la_forward")


def test_noalloc_allocates_nothing_and_launches_la_forwards_kernels(lib):
    B, H, N, D, M = 2, 3, 700, 64, 64
    q, k, v = inputs.qkv(78, B, H, N, D, M, 0.125, inputs.BF16)
    tq, tk, tv = (inputs.to_torch(x, inputs.BF16, DEV) for x in (q, k, v))
    out = torch.empty_like(tv)
    ws = torch.empty((lib.la_forward_workspace_bytes(B, H, N, D, M, True, lib.LA_BF16),),
                     dtype=torch.uint8, device=DEV)
    n0 = lib.la_kernel_launches()
    lib.la_forward(tq, tk, tv, causal=True, out=out, workspace=ws)
    per_call = lib.la_kernel_launches() - n0
    assert per_call >= 1
    # one call first: the CUDA loader maps the library's device array (the fixed
    # scratch) when it is first looked up, which is module loading, not a call's work
    assert _noalloc(lib, tq, tk, tv, out, True) == lib.LA_OK
    torch.cuda.synchronize()
    mem0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    free0 = torch.cuda.mem_get_info()[0]
    n1 = lib.la_kernel_launches()
    assert _noalloc(lib, tq, tk, tv, out, True) == lib.LA_OK
    torch.cuda.synchronize()
    assert lib.la_kernel_launches() - n1 == per_call
    assert torch.cuda.memory_allocated() == mem0 and torch.cuda.memory_reserved() == reserved0
    assert torch.cuda.mem_get_info()[0] == free0       # nothing allocated outside torch either


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    # 4096 short sequences need far more than the fixed array's segment states
    B, H, N, D, M = 512, 8, 256, 64, 64
    need = lib.la_forward_workspace_bytes(B, H, N, D, M, True, lib.LA_BF16)
    assert need > (32 << 20)
    e = torch.empty((1,), dtype=torch.bfloat16, device=DEV)
    n0 = lib.la_kernel_launches()
    st = lib.load_library().la_forward_noalloc(
        ctypes.c_void_p(e.data_ptr()), ctypes.c_void_p(e.data_ptr()), ctypes.c_void_p(e.data_ptr()),
        ctypes.c_void_p(e.data_ptr()), B, H, N, D, M, 1, lib.LA_BF16, None)
    assert st == lib.LA_ERR_TOO_LARGE
    assert lib.la_kernel_launches() == n0              # refused before anything was launched
    assert "scratch" in lib.la_status_string(st)


def test_noalloc_status_word_is_read_and_cleared(lib):
    """The status a timed-out kernel would leave in the fixed array's header (written
    here by the test hook, no kernel made to wait) is reported once, then cleared."""
    c = lib.load_library()
    assert c.la_debug_noalloc_set_status(lib.LA_ERR_TIMEOUT, lib.LA_SITE_FORWARD_LOAD,
                                         _stream()) == lib.LA_OK
    assert lib.la_forward_noalloc_status() == lib.LA_ERR_TIMEOUT
    assert lib.la_forward_noalloc_status() == lib.LA_OK
    # a call clears the word on entry: a stale status does not outlive the next call
    assert c.la_debug_noalloc_set_status(lib.LA_ERR_TIMEOUT, 0, _stream()) == lib.LA_OK
    q, k, v = inputs.qkv(79, 1, 2, 300, 64, 64, 0.125, inputs.BF16)
    tq, tk, tv = (inputs.to_torch(x, inputs.BF16, DEV) for x in (q, k, v))
    out = torch.empty_like(tv)
    assert _noalloc(lib, tq, tk, tv, out, True) == lib.LA_OK
    assert lib.la_forward_noalloc_status() == lib.LA_OK
