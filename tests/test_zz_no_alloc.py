"""la_forward_noalloc: the forward for callers that cannot allocate device memory.

Such callers only receive device pointers for their inputs and outputs (the
application or framework around them owns the allocator), so they cannot hand
la_forward a workspace. la_forward_noalloc runs the same computation with its
scratch in a fixed array inside the library's device memory. These tests call
it through the C ABI and compare it with la_forward (caller workspace) on two
calls in a row, and check that a shape needing more scratch than the array
holds is refused before anything is launched.
"""

import ctypes

import numpy as np
import pytest

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
    return pkg


def _noalloc(pkg, q, k, v, out, causal):
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = pkg.LA_BF16 if q.dtype == torch.bfloat16 else pkg.LA_F32
    return pkg.load_library().la_forward_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), B, H, N, D, M, int(causal), dt,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("case", [
    (2, 3, 700, 64, 64, inputs.BF16, True),
    (2, 3, 700, 64, 64, inputs.BF16, False),
    (4, 8, 3072, 64, 64, inputs.BF16, True),
    (1, 2, 129, 32, 32, inputs.F32, True),
], ids=["bf16-causal", "bf16-noncausal", "bf16-causal-b4h8n3072", "f32-causal"])
def test_noalloc_matches_la_forward_twice(lib, case):
    B, H, N, D, M, dtype, causal = case
    scale = 0.125 if dtype == inputs.BF16 else 1.0
    q, k, v = inputs.qkv(77, B, H, N, D, M, scale, dtype)
    tq, tk, tv = (inputs.to_torch(x, dtype, DEV) for x in (q, k, v))
    ref = lib.la_forward(tq, tk, tv, causal=causal)
    torch.cuda.synchronize()
    want = ref.float().cpu().numpy()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(lib, tq, tk, tv, out, causal) == lib.LA_OK
        torch.cuda.synchronize()
        assert_close(out.float().cpu().numpy(), want, dtype, "la_forward_noalloc vs la_forward")


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    # 4096 short sequences need far more than the fixed array's segment states
    B, H, N, D, M = 512, 8, 256, 64, 64
    need = lib.la_forward_workspace_bytes(B, H, N, D, M, True, lib.LA_BF16)
    assert need > (32 << 20)
    e = torch.empty((1,), dtype=torch.bfloat16, device=DEV)
    st = lib.load_library().la_forward_noalloc(
        ctypes.c_void_p(e.data_ptr()), ctypes.c_void_p(e.data_ptr()), ctypes.c_void_p(e.data_ptr()),
        ctypes.c_void_p(e.data_ptr()), B, H, N, D, M, 1, lib.LA_BF16, None)
    assert st == lib.LA_ERR_TOO_LARGE
    assert "scratch" in lib.la_status_string(st)
