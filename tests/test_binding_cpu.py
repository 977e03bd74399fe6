"""Argument checks of the Python binding (no GPU needed).

The library receives raw pointers and sizes taken from q and v, so a tensor of
the wrong shape or dtype would make a kernel read or write past its memory.
The binding rejects such calls before anything reaches the library; with
well-formed CPU tensors a call gets as far as the device check.
"""

import pytest
import torch

import kernelized_causal_self_gb300 as la

BF, F32 = torch.bfloat16, torch.float32


def _t(*shape, dtype=BF):
    return torch.zeros(shape, dtype=dtype)


def _raises(match, fn, *args, **kw):
    with pytest.raises(ValueError, match=match):
        fn(*args, **kw)


def test_forward_checks_every_tensor():
    q, v = _t(2, 3, 10, 16), _t(2, 3, 10, 8)
    _raises("k must be", la.la_forward, q, _t(2, 3, 11, 16), v)
    _raises("k must be", la.la_forward, q, _t(2, 3, 10, 16, dtype=F32), v)
    _raises("v must be", la.la_forward, q, q, _t(2, 3, 9, 8))
    _raises("out must be", la.la_forward, q, q, v, out=_t(2, 3, 10, 16))
    _raises("out must be", la.la_forward, q, q, v, out=_t(2, 3, 10, 8, dtype=F32))
    _raises("4 dimensions", la.la_forward, _t(3, 10, 16), _t(3, 10, 16), _t(3, 10, 8))
    _raises("CUDA device", la.la_forward, q, q, v, out=_t(2, 3, 10, 8))
    _raises("CUDA device", la.la_forward_noalloc, q, q, v)
    _raises("out must be", la.la_forward_noalloc, q, q, v, out=_t(2, 3, 10, 9))
    with pytest.raises(TypeError):
        la.la_forward(q.half(), q.half(), v.half())


def test_prefill_checks_state_outputs():
    q, v = _t(2, 3, 10, 16), _t(2, 3, 10, 8)
    _raises("S must be", la.la_prefill, q, q, v, S=_t(2, 3, 8, 16, dtype=F32))
    _raises("S must be", la.la_prefill, q, q, v, S=_t(2, 3, 16, 8))  # bf16 state
    _raises("Z must be", la.la_prefill, q, q, v, Z=_t(2, 3, 8, dtype=F32))
    _raises("CUDA device", la.la_prefill, q, q, v, S=_t(2, 3, 16, 8, dtype=F32),
            Z=_t(2, 3, 16, dtype=F32))


def test_extend_checks_pool_and_indices():
    q, v = _t(2, 3, 4, 16), _t(2, 3, 4, 8)
    S, Z = _t(5, 3, 16, 8, dtype=F32), _t(5, 3, 16, dtype=F32)
    _raises("S_pool must be", la.la_extend, q, q, v, _t(5, 2, 16, 8, dtype=F32), Z)
    _raises("Z_pool must be", la.la_extend, q, q, v, S, _t(4, 3, 16, dtype=F32))
    _raises("S_pool must be", la.la_extend, q, q, v, _t(5, 3, 16, 8), Z)
    _raises("slots must be", la.la_extend, q, q, v, S, Z, slots=torch.zeros(2, dtype=torch.int64))
    _raises("lens must be", la.la_extend, q, q, v, S, Z, lens=torch.zeros(3, dtype=torch.int32))
    _raises("out must be", la.la_extend, q, q, v, S, Z, out=_t(2, 3, 4, 16))
    _raises("CUDA device", la.la_extend, q, q, v, S, Z, slots=torch.tensor([1, 3], dtype=torch.int32))


def test_extend_packed_checks_layout_and_offsets():
    q, v = _t(9, 3, 16), _t(9, 3, 8)
    S, Z = _t(5, 3, 16, 8, dtype=F32), _t(5, 3, 16, dtype=F32)
    cu = torch.tensor([0, 4, 9], dtype=torch.int32)
    _raises("3 dimensions", la.la_extend_packed, _t(1, 9, 3, 16), _t(1, 9, 3, 16), _t(1, 9, 3, 8),
            S, Z, cu, 8)
    _raises("k must be", la.la_extend_packed, q, _t(9, 3, 8), v, S, Z, cu, 8)
    _raises("v must be", la.la_extend_packed, q, q, _t(8, 3, 8), S, Z, cu, 8)
    _raises("S_pool must be", la.la_extend_packed, q, q, v, _t(5, 2, 16, 8, dtype=F32), Z, cu, 8)
    _raises("Z_pool must be", la.la_extend_packed, q, q, v, S, _t(5, 3, 8, dtype=F32), cu, 8)
    _raises("cu_seqlens must be", la.la_extend_packed, q, q, v, S, Z, cu.long(), 8)
    _raises("cu_seqlens must be", la.la_extend_packed, q, q, v, S, Z, cu[:1], 8)
    _raises("slots must be", la.la_extend_packed, q, q, v, S, Z, cu, 8,
            slots=torch.zeros(3, dtype=torch.int32))
    _raises("out must be", la.la_extend_packed, q, q, v, S, Z, cu, 8, out=_t(9, 3, 16))
    _raises("CUDA device", la.la_extend_packed, q, q, v, S, Z, cu, 8)


def test_backward_checks_gradients():
    q, v = _t(2, 3, 10, 16), _t(2, 3, 10, 8)
    _raises("dout must be", la.la_backward, q, q, v, _t(2, 3, 10, 16))
    _raises("dout must be", la.la_backward, q, q, v, _t(2, 3, 10, 8, dtype=F32))
    _raises("dq must be", la.la_backward, q, q, v, v, dq=_t(2, 3, 10, 16))  # bf16 gradient
    _raises("dk must be", la.la_backward, q, q, v, v, dk=_t(2, 3, 10, 8, dtype=F32))
    _raises("dv must be", la.la_backward, q, q, v, v, dv=_t(2, 3, 10, 16, dtype=F32))
    _raises("CUDA device", la.la_backward, q, q, v, v, dq=_t(2, 3, 10, 16, dtype=F32),
            dk=_t(2, 3, 10, 16, dtype=F32), dv=_t(2, 3, 10, 8, dtype=F32))


def test_decode_checks_state_and_output():
    q, v = _t(4, 3, 16), _t(4, 3, 8)
    S, Z = _t(4, 3, 16, 8, dtype=F32), _t(4, 3, 16, dtype=F32)
    _raises("3 dimensions", la.la_decode_step, _t(4, 3, 1, 16), _t(4, 3, 1, 16), _t(4, 3, 1, 8), S, Z)
    _raises("S must be", la.la_decode_step, q, q, v, _t(5, 3, 16, 8, dtype=F32), Z)
    _raises("Z must be", la.la_decode_step, q, q, v, S, _t(4, 3, 8, dtype=F32))
    _raises("out must be", la.la_decode_step, q, q, v, S, Z, out=_t(4, 3, 16))
    _raises("CUDA device", la.la_decode_step, q, q, v, S, Z)


def test_every_library_call_runs_with_the_tensors_device_current(monkeypatch):
    """The library looks up per-device state on the current device and launches on the
    stream it is given (the tensors' device's), so each wrapper makes the tensors' device
    current around its call into the library. Checked with a recording stand-in for the
    device guard and for the library."""
    events = []

    class Guard:
        def __init__(self, dev):
            self.dev = str(dev)

        def __enter__(self):
            events.append(("enter", self.dev))

        def __exit__(self, *exc):
            events.append(("exit", self.dev))

    class FakeLib:
        def __getattr__(self, name):
            def fn(*args):
                events.append(("call", name))
                return 256 if name.endswith("_bytes") else 0
            return fn

    monkeypatch.setattr(la, "_on_device", Guard)
    monkeypatch.setattr(la, "load_library", lambda: FakeLib())
    monkeypatch.setattr(la, "_need_cuda", lambda *a, **k: None)
    monkeypatch.setattr(la, "_stream_ptr", lambda dev: 0)
    q, v = _t(2, 3, 10, 16), _t(2, 3, 10, 8)
    S, Z = _t(2, 3, 16, 8, dtype=F32), _t(2, 3, 16, dtype=F32)
    ws = torch.zeros(256, dtype=torch.uint8)
    la.la_forward(q, q, v)
    la.la_forward_noalloc(q, q, v)
    la.la_prefill(q, q, v)
    la.la_extend(q, q, v, S, Z)
    pq, pv = _t(10, 3, 16), _t(10, 3, 8)
    la.la_extend_packed(pq, pq, pv, S, Z, torch.tensor([0, 4, 10], dtype=torch.int32), 6)
    la.la_backward(q, q, v, v)
    la.la_decode_step(q[:, :, 0], q[:, :, 0], v[:, :, 0], S, Z)
    la.la_workspace_status(ws)
    la.la_workspace_wait_site(ws)
    la.la_forward_noalloc_status(device="cpu")
    calls = [i for i, e in enumerate(events) if e[0] == "call" and not e[1].endswith("_bytes")]
    assert [events[i][1] for i in calls] == [
        "la_forward", "la_forward_noalloc", "la_prefill", "la_extend", "la_extend_packed",
        "la_backward",
        "la_decode_step", "la_workspace_status", "la_workspace_wait_site",
        "la_forward_noalloc_status"]
    for i in calls:
        assert events[i - 1] == ("enter", "cpu") and events[i + 1] == ("exit", "cpu"), events[i]
