"""Thin Python binding over the C ABI in ``include/la.h``.

Argument marshalling only: every tensor is checked for shape and dtype against
the layouts of ``include/la.h`` (sizes taken from ``q`` and ``v``), then for
being a contiguous CUDA tensor on ``q``'s device, since the library sees only
raw pointers; their ``data_ptr()`` and the current CUDA stream are handed to the
shared library, and outputs/workspaces are allocated with PyTorch (the caller's
allocator). Every step of the computation runs in the library's CUDA kernels;
there is no fallback. If the library is missing the calls raise.
"""

import ctypes
import os

__all__ = [
    "la_forward", "la_prefill", "la_extend", "la_extend_packed", "la_backward", "la_decode_step",
    "la_forward_workspace_bytes", "la_backward_workspace_bytes",
    "la_workspace_status", "la_status_string", "la_kernel_launches", "library_path",
    "load_library",
    "LAError", "LA_OK", "LA_ERR_INVALID_ARG", "LA_ERR_WORKSPACE", "LA_ERR_CUDA",
    "LA_ERR_TIMEOUT", "LA_ERR_TOO_LARGE", "LA_F32", "LA_BF16", "la_forward_noalloc",
    "la_forward_noalloc_status", "la_workspace_wait_site",
    "la_state_sums", "la_forward_shard", "la_backward_shard_q", "la_backward_shard_kv",
    "la_forward_poly2", "la_poly2_workspace_bytes", "la_forward_rff", "la_rff_workspace_bytes",
    "LA_SITE_FORWARD_LOAD", "LA_SITE_BACKWARD_LOAD",
]

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_WORKSPACE, LA_ERR_CUDA, LA_ERR_TIMEOUT = 0, 1, 2, 3, 4
LA_ERR_TOO_LARGE = 5
LA_F32, LA_BF16 = 0, 1
LA_SITE_FORWARD_LOAD, LA_SITE_FORWARD_FUSED_LOAD, LA_SITE_BACKWARD_LOAD = 11, 16, 21

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "liblagb300.so")
_lib = None

_c_int, _c_size, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p

_SIGNATURES = {
    "la_status_string": (ctypes.c_char_p, [_c_int]),
    "la_version": (_c_int, []),
    "la_kernel_launches": (ctypes.c_ulonglong, []),
    "la_forward_workspace_bytes": (_c_size, [_c_int] * 7),
    "la_backward_workspace_bytes": (_c_size, [_c_int] * 7),
    "la_forward": (_c_int, [_vp] * 4 + [_c_int] * 7 + [_vp, _c_size, _vp]),
    "la_prefill": (_c_int, [_vp] * 6 + [_c_int] * 6 + [_vp, _c_size, _vp]),
    "la_extend": (_c_int, [_vp] * 8 + [_c_int] * 7 + [_vp, _c_size, _vp]),
    "la_extend_packed": (_c_int, [_vp] * 8 + [_c_int] * 8 + [_vp, _c_size, _vp]),
    "la_backward": (_c_int, [_vp] * 7 + [_c_int] * 7 + [_vp, _c_size, _vp]),
    "la_decode_step": (_c_int, [_vp] * 6 + [_c_int] * 5 + [_vp]),
    "la_workspace_status": (_c_int, [_vp, _c_size, _vp]),
    "la_forward_noalloc": (_c_int, [_vp] * 4 + [_c_int] * 7 + [_vp]),
    "la_forward_noalloc_status": (_c_int, [_vp]),
    "la_state_sums": (_c_int, [_vp] * 4 + [_c_int] * 6 + [_vp, _c_size, _vp]),
    "la_poly2_workspace_bytes": (_c_size, [_c_int] * 7),
    "la_rff_workspace_bytes": (_c_size, [_c_int] * 8),
    "la_forward_rff": (_c_int, [_vp] * 6 + [_c_int] * 8 + [_vp, _c_size, _vp]),
    "la_backward_from_forward": (_c_int, [_vp] * 7 + [_c_int] * 7 + [_vp, _c_size, _vp, _c_size,
                                                                     _vp]),
    "la_forward_poly2": (_c_int, [_vp] * 4 + [_c_int] * 7 + [_vp, _c_size, _vp]),
    "la_forward_shard": (_c_int, [_vp] * 6 + [_c_int] * 6 + [_vp, _c_size, _vp]),
    "la_backward_shard_q": (_c_int, [_vp] * 9 + [_c_int] * 6 + [_vp, _c_size, _vp]),
    "la_backward_shard_kv": (_c_int, [_vp] * 8 + [_c_int] * 6 + [_vp, _c_size, _vp]),
    "la_debug_noalloc_set_status": (_c_int, [_c_int, _c_int, _vp]),
    "la_workspace_wait_site": (_c_int, [_vp, _c_size, _vp]),
    "la_debug_forward_fault": (_c_int, [_vp] * 4 + [_c_int] * 7 + [_vp, _c_size, _c_int,
                                                                    ctypes.c_ulonglong, _vp]),
    "la_debug_forward_fused_fault": (_c_int, [_vp] * 4 + [_c_int] * 7 + [_vp, _c_size, _c_int,
                                                                          ctypes.c_ulonglong, _vp]),
    "la_debug_backward_fault": (_c_int, [_vp] * 7 + [_c_int] * 7 + [_vp, _c_size, _c_int,
                                                                     ctypes.c_ulonglong, _vp]),
}


class LAError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {la_status_string(status)} (status {status})")


def library_path():
    return _LIB_PATH


def load_library():
    """Load the shared library (ctypes); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"CUDA library not built: {_LIB_PATH} is missing "
                "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def la_status_string(status):
    return load_library().la_status_string(int(status)).decode()


def _check(fn, status):
    if status != LA_OK:
        raise LAError(fn, status)


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return LA_F32
    if t.dtype == torch.bfloat16:
        return LA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _on_device(device):
    """Context that makes `device` current around a library call: the library looks up
    per-device state (la_forward_noalloc's fixed scratch) on the current device, and the
    stream it is handed belongs to `device`."""
    import torch
    return torch.cuda.device(device)


def _stream_ptr(device):
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def _need_cuda(*ts, device=None):
    """Contiguous CUDA tensors, all on `device` (default: the first one's)."""
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if device is None:
            device = t.device
        elif t.device != device:
            raise ValueError(f"tensors must all be on {device}, got one on {t.device}")


def _expect(fn, name, t, shape, dtype):
    """`t` has exactly `shape` and `dtype` (the library reads and writes that many elements)."""
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{fn}: {name} must be {dtype} of shape {tuple(shape)}, "
                         f"got {t.dtype} of shape {tuple(t.shape)}")


def _dims(fn, q, v, rank):
    """(leading sizes of q, D, M) for q [..., D], v [..., M] of the given rank."""
    if q.dim() != rank or v.dim() != rank:
        raise ValueError(f"{fn}: q and v must have {rank} dimensions")
    return tuple(q.shape[:-1]), q.shape[-1], v.shape[-1]


def _workspace(nbytes, device, workspace):
    import torch
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        _need_cuda(workspace, device=device)
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def la_kernel_launches():
    """Kernels launched by the library in this process so far."""
    return int(load_library().la_kernel_launches())


def la_forward_workspace_bytes(B, H, N, D, M, causal=True, dtype=LA_BF16):
    return load_library().la_forward_workspace_bytes(B, H, N, D, M, int(bool(causal)), dtype)


def la_backward_workspace_bytes(B, H, N, D, M, causal=True, dtype=LA_BF16):
    return load_library().la_backward_workspace_bytes(B, H, N, D, M, int(bool(causal)), dtype)


def la_forward(q, k, v, causal=True, out=None, workspace=None):
    """out[B,H,N,M] = kernelized attention of q, k [B,H,N,D] and v [B,H,N,M]."""
    import torch
    (B, H, N), D, M = _dims("la_forward", q, v, 4)
    _expect("la_forward", "k", k, q.shape, q.dtype)
    _expect("la_forward", "v", v, (B, H, N, M), q.dtype)
    if out is not None:
        _expect("la_forward", "out", out, (B, H, N, M), q.dtype)
    dt = _dtype_code(q)
    _need_cuda(q, k, v, *([] if out is None else [out]))
    lib = load_library()
    if out is None:
        out = torch.empty((B, H, N, M), dtype=q.dtype, device=q.device)
    nbytes = lib.la_forward_workspace_bytes(B, H, N, D, M, int(bool(causal)), dt)
    ws = _workspace(nbytes, q.device, workspace)
    with _on_device(q.device):
        st = lib.la_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N, D,
                            M, int(bool(causal)), dt, ws.data_ptr(),
                            ws.numel() * ws.element_size(), _stream_ptr(q.device))
    _check("la_forward", st)
    return out


def la_forward_noalloc(q, k, v, causal=True, out=None):
    """la_forward without a workspace: the library's fixed device scratch array is used.

    For callers that cannot allocate device memory. Calls that overlap on the
    GPU share that array and race; the first call on a device must not be
    made during stream capture.
    """
    import torch
    (B, H, N), D, M = _dims("la_forward_noalloc", q, v, 4)
    _expect("la_forward_noalloc", "k", k, q.shape, q.dtype)
    _expect("la_forward_noalloc", "v", v, (B, H, N, M), q.dtype)
    if out is not None:
        _expect("la_forward_noalloc", "out", out, (B, H, N, M), q.dtype)
    dt = _dtype_code(q)
    _need_cuda(q, k, v, *([] if out is None else [out]))
    lib = load_library()
    if out is None:
        out = torch.empty((B, H, N, M), dtype=q.dtype, device=q.device)
    with _on_device(q.device):
        st = lib.la_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H,
                                    N, D, M, int(bool(causal)), dt, _stream_ptr(q.device))
    _check("la_forward_noalloc", st)
    return out


def la_prefill(q, k, v, out=None, S=None, Z=None, workspace=None):
    """Causal forward plus the final float32 state S [B,H,D,M], Z [B,H,D]."""
    import torch
    fn, f32 = "la_prefill", torch.float32
    (B, H, N), D, M = _dims(fn, q, v, 4)
    _expect(fn, "k", k, q.shape, q.dtype)
    _expect(fn, "v", v, (B, H, N, M), q.dtype)
    given = [(n, t) for n, t in (("out", out), ("S", S), ("Z", Z)) if t is not None]
    for name, t in given:
        _expect(fn, name, t, {"out": (B, H, N, M), "S": (B, H, D, M), "Z": (B, H, D)}[name],
                q.dtype if name == "out" else f32)
    dt = _dtype_code(q)
    _need_cuda(q, k, v, *[t for _, t in given])
    lib = load_library()
    dev = q.device
    out = torch.empty((B, H, N, M), dtype=q.dtype, device=dev) if out is None else out
    S = torch.empty((B, H, D, M), dtype=f32, device=dev) if S is None else S
    Z = torch.empty((B, H, D), dtype=f32, device=dev) if Z is None else Z
    nbytes = lib.la_forward_workspace_bytes(B, H, N, D, M, 1, dt)
    ws = _workspace(nbytes, dev, workspace)
    with _on_device(dev):
        st = lib.la_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), S.data_ptr(),
                            Z.data_ptr(), B, H, N, D, M, dt, ws.data_ptr(),
                            ws.numel() * ws.element_size(), _stream_ptr(dev))
    _check("la_prefill", st)
    return out, S, Z


def la_extend(q, k, v, S_pool, Z_pool, slots=None, lens=None, out=None, workspace=None):
    """Causal forward over new tokens of B streams continuing from stored state.

    S_pool [P,H,D,M], Z_pool [P,H,D] float32 hold per-stream states; stream b uses
    entry slots[b] (int32 device tensor of B distinct entries; None: entry b) and
    its entry is advanced past its tokens in place: the first lens[b] of the N
    (int32 device tensor; None: all N). Returns out [B,H,N,M]; rows at or past
    lens[b] are unspecified.
    """
    import torch
    fn, f32 = "la_extend", torch.float32
    (B, H, N), D, M = _dims(fn, q, v, 4)
    _expect(fn, "k", k, q.shape, q.dtype)
    _expect(fn, "v", v, (B, H, N, M), q.dtype)
    if S_pool.dim() != 4:
        raise ValueError(f"{fn}: S_pool must be [pool, H, D, M]")
    P = S_pool.shape[0]
    _expect(fn, "S_pool", S_pool, (P, H, D, M), f32)
    _expect(fn, "Z_pool", Z_pool, (P, H, D), f32)
    if out is not None:
        _expect(fn, "out", out, (B, H, N, M), q.dtype)
    for name, t in (("slots", slots), ("lens", lens)):
        if t is not None and (t.dtype != torch.int32 or t.numel() != B):
            raise ValueError(f"{name} must be a contiguous int32 tensor of B entries")
    dt = _dtype_code(q)
    _need_cuda(q, k, v, S_pool, Z_pool,
               *[t for t in (out, slots, lens) if t is not None])
    lib = load_library()
    dev = q.device
    out = torch.empty((B, H, N, M), dtype=q.dtype, device=dev) if out is None else out
    nbytes = lib.la_forward_workspace_bytes(B, H, N, D, M, 1, dt)
    ws = _workspace(nbytes, dev, workspace)
    with _on_device(dev):
        st = lib.la_extend(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           S_pool.data_ptr(), Z_pool.data_ptr(),
                           0 if slots is None else slots.data_ptr(),
                           0 if lens is None else lens.data_ptr(), P,
                           B, H, N, D, M, dt, ws.data_ptr(), ws.numel() * ws.element_size(),
                           _stream_ptr(dev))
    _check("la_extend", st)
    return out


def la_extend_packed(q, k, v, S_pool, Z_pool, cu_seqlens, max_len, slots=None, out=None,
                     workspace=None):
    """la_extend on a packed batch: q, k [T,H,D] and v [T,H,M], stream b in rows
    cu_seqlens[b] .. cu_seqlens[b+1]-1 (int32 device tensor of B + 1 offsets), each
    stream at most max_len tokens. Returns out [T,H,M] (rows of no stream are left
    as they were in `out`, uninitialised if it is None).
    """
    import torch
    fn, f32 = "la_extend_packed", torch.float32
    (T, H), D, M = _dims(fn, q, v, 3)
    _expect(fn, "k", k, q.shape, q.dtype)
    _expect(fn, "v", v, (T, H, M), q.dtype)
    if S_pool.dim() != 4:
        raise ValueError(f"{fn}: S_pool must be [pool, H, D, M]")
    P = S_pool.shape[0]
    _expect(fn, "S_pool", S_pool, (P, H, D, M), f32)
    _expect(fn, "Z_pool", Z_pool, (P, H, D), f32)
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be a contiguous int32 tensor of B + 1 offsets")
    B = cu_seqlens.numel() - 1
    if slots is not None and (slots.dtype != torch.int32 or slots.numel() != B):
        raise ValueError("slots must be a contiguous int32 tensor of B entries")
    if out is not None:
        _expect(fn, "out", out, (T, H, M), q.dtype)
    dt = _dtype_code(q)
    _need_cuda(q, k, v, S_pool, Z_pool, cu_seqlens,
               *[t for t in (out, slots) if t is not None])
    lib = load_library()
    dev = q.device
    out = torch.empty((T, H, M), dtype=q.dtype, device=dev) if out is None else out
    nbytes = lib.la_forward_workspace_bytes(B, H, max_len, D, M, 1, dt)
    ws = _workspace(nbytes, dev, workspace)
    with _on_device(dev):
        st = lib.la_extend_packed(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  S_pool.data_ptr(), Z_pool.data_ptr(),
                                  0 if slots is None else slots.data_ptr(),
                                  cu_seqlens.data_ptr(), P, B, H, T, int(max_len), D, M, dt,
                                  ws.data_ptr(), ws.numel() * ws.element_size(), _stream_ptr(dev))
    _check(fn, st)
    return out


def la_backward(q, k, v, dout, causal=True, dq=None, dk=None, dv=None, workspace=None,
                fwd_workspace=None):
    """float32 gradients (dq, dk, dv) of sum(dout * la_forward(q, k, v)).

    fwd_workspace: the workspace of a la_forward call on the same q, k, v (and causal), not
    reused since; its segment states are then read instead of recomputed
    (la_backward_from_forward)."""
    import torch
    fn, f32 = "la_backward", torch.float32
    (B, H, N), D, M = _dims(fn, q, v, 4)
    _expect(fn, "k", k, q.shape, q.dtype)
    _expect(fn, "v", v, (B, H, N, M), q.dtype)
    _expect(fn, "dout", dout, (B, H, N, M), q.dtype)
    given = [(n, t) for n, t in (("dq", dq), ("dk", dk), ("dv", dv)) if t is not None]
    for name, t in given:
        _expect(fn, name, t, (B, H, N, M) if name == "dv" else (B, H, N, D), f32)
    dt = _dtype_code(q)
    _need_cuda(q, k, v, dout, *[t for _, t in given])
    lib = load_library()
    dev = q.device
    dq = torch.empty((B, H, N, D), dtype=f32, device=dev) if dq is None else dq
    dk = torch.empty((B, H, N, D), dtype=f32, device=dev) if dk is None else dk
    dv = torch.empty((B, H, N, M), dtype=f32, device=dev) if dv is None else dv
    nbytes = lib.la_backward_workspace_bytes(B, H, N, D, M, int(bool(causal)), dt)
    ws = _workspace(nbytes, dev, workspace)
    if fwd_workspace is not None:
        _need_cuda(fwd_workspace, device=dev)
    with _on_device(dev):
        if fwd_workspace is None:
            st = lib.la_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                                 dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, D, M,
                                 int(bool(causal)), dt, ws.data_ptr(),
                                 ws.numel() * ws.element_size(), _stream_ptr(dev))
        else:
            st = lib.la_backward_from_forward(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(), dq.data_ptr(),
                dk.data_ptr(), dv.data_ptr(), B, H, N, D, M, int(bool(causal)), dt,
                fwd_workspace.data_ptr(), fwd_workspace.numel() * fwd_workspace.element_size(),
                ws.data_ptr(), ws.numel() * ws.element_size(), _stream_ptr(dev))
    _check("la_backward", st)
    return dq, dk, dv


def la_decode_step(q, k, v, S, Z, out=None):
    """One recurrent step: q, k [S,H,D], v [S,H,M]; S, Z updated in place; returns out."""
    import torch
    fn, f32 = "la_decode_step", torch.float32
    (n, H), D, M = _dims(fn, q, v, 3)
    _expect(fn, "k", k, q.shape, q.dtype)
    _expect(fn, "v", v, (n, H, M), q.dtype)
    _expect(fn, "S", S, (n, H, D, M), f32)
    _expect(fn, "Z", Z, (n, H, D), f32)
    if out is not None:
        _expect(fn, "out", out, (n, H, M), q.dtype)
    dt = _dtype_code(q)
    _need_cuda(q, k, v, S, Z, *([] if out is None else [out]))
    lib = load_library()
    out = torch.empty((n, H, M), dtype=q.dtype, device=q.device) if out is None else out
    with _on_device(q.device):
        st = lib.la_decode_step(q.data_ptr(), k.data_ptr(), v.data_ptr(), S.data_ptr(),
                                Z.data_ptr(), out.data_ptr(), n, H, D, M, dt,
                                _stream_ptr(q.device))
    _check("la_decode_step", st)
    return out


def la_workspace_status(workspace):
    """Synchronise and read (then clear) the status word a call left in `workspace`."""
    lib = load_library()
    with _on_device(workspace.device):
        return lib.la_workspace_status(workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(),
                                       _stream_ptr(workspace.device))


def la_workspace_wait_site(workspace):
    """Synchronise and read the code of the bounded wait that last gave up in the call that
    used `workspace` (0: none). Nothing is cleared."""
    lib = load_library()
    with _on_device(workspace.device):
        return lib.la_workspace_wait_site(workspace.data_ptr(),
                                          workspace.numel() * workspace.element_size(),
                                          _stream_ptr(workspace.device))


def la_forward_noalloc_status(device=None):
    """Synchronise and read (then clear) the status word of la_forward_noalloc's fixed
    scratch on `device` (default: the current CUDA device)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    lib = load_library()
    with _on_device(dev):
        return lib.la_forward_noalloc_status(_stream_ptr(dev))


# ------------------------------------------------------------ sequence shards

def _state_shapes(B, H, D, M):
    return (B, H, D, M), (B, H, D)


def la_state_sums(k, v, S=None, Z=None, workspace=None):
    """A shard's own sums S = sum_j phi(k_j) v_j^T [B,H,D,M], Z = sum_j phi(k_j) [B,H,D]."""
    import torch
    fn, f32 = "la_state_sums", torch.float32
    (B, H, N), D, M = _dims(fn, k, v, 4)
    _expect(fn, "v", v, (B, H, N, M), k.dtype)
    sS, sZ = _state_shapes(B, H, D, M)
    for name, t, shp in (("S", S, sS), ("Z", Z, sZ)):
        if t is not None:
            _expect(fn, name, t, shp, f32)
    dt = _dtype_code(k)
    _need_cuda(k, v, *[t for t in (S, Z) if t is not None])
    lib = load_library()
    dev = k.device
    S = torch.empty(sS, dtype=f32, device=dev) if S is None else S
    Z = torch.empty(sZ, dtype=f32, device=dev) if Z is None else Z
    ws = _workspace(lib.la_forward_workspace_bytes(B, H, N, D, M, 1, dt), dev, workspace)
    with _on_device(dev):
        st = lib.la_state_sums(k.data_ptr(), v.data_ptr(), S.data_ptr(), Z.data_ptr(), B, H, N, D,
                               M, dt, ws.data_ptr(), ws.numel() * ws.element_size(),
                               _stream_ptr(dev))
    _check(fn, st)
    return S, Z


def la_forward_shard(q, k, v, S0, Z0, out=None, workspace=None):
    """Causal forward of a shard's tokens after the state (S0, Z0) of the tokens before them."""
    import torch
    fn, f32 = "la_forward_shard", torch.float32
    (B, H, N), D, M = _dims(fn, q, v, 4)
    _expect(fn, "k", k, q.shape, q.dtype)
    _expect(fn, "v", v, (B, H, N, M), q.dtype)
    sS, sZ = _state_shapes(B, H, D, M)
    _expect(fn, "S0", S0, sS, f32)
    _expect(fn, "Z0", Z0, sZ, f32)
    if out is not None:
        _expect(fn, "out", out, (B, H, N, M), q.dtype)
    dt = _dtype_code(q)
    _need_cuda(q, k, v, S0, Z0, *([] if out is None else [out]))
    lib = load_library()
    dev = q.device
    out = torch.empty((B, H, N, M), dtype=q.dtype, device=dev) if out is None else out
    ws = _workspace(lib.la_forward_workspace_bytes(B, H, N, D, M, 1, dt), dev, workspace)
    with _on_device(dev):
        st = lib.la_forward_shard(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  S0.data_ptr(), Z0.data_ptr(), B, H, N, D, M, dt, ws.data_ptr(),
                                  ws.numel() * ws.element_size(), _stream_ptr(dev))
    _check(fn, st)
    return out


def la_backward_shard_q(q, k, v, dout, S0, Z0, dq=None, R_own=None, r_own=None, workspace=None):
    """First backward pass of a shard: (dq, R_own, r_own, workspace); pass the workspace on
    to la_backward_shard_kv."""
    import torch
    fn, f32 = "la_backward_shard_q", torch.float32
    (B, H, N), D, M = _dims(fn, q, v, 4)
    _expect(fn, "k", k, q.shape, q.dtype)
    _expect(fn, "v", v, (B, H, N, M), q.dtype)
    _expect(fn, "dout", dout, (B, H, N, M), q.dtype)
    sS, sZ = _state_shapes(B, H, D, M)
    _expect(fn, "S0", S0, sS, f32)
    _expect(fn, "Z0", Z0, sZ, f32)
    given = [(n, t, shp) for n, t, shp in (("dq", dq, (B, H, N, D)), ("R_own", R_own, sS),
                                           ("r_own", r_own, sZ)) if t is not None]
    for name, t, shp in given:
        _expect(fn, name, t, shp, f32)
    dt = _dtype_code(q)
    _need_cuda(q, k, v, dout, S0, Z0, *[t for _, t, _ in given])
    lib = load_library()
    dev = q.device
    dq = torch.empty((B, H, N, D), dtype=f32, device=dev) if dq is None else dq
    R_own = torch.empty(sS, dtype=f32, device=dev) if R_own is None else R_own
    r_own = torch.empty(sZ, dtype=f32, device=dev) if r_own is None else r_own
    ws = _workspace(lib.la_backward_workspace_bytes(B, H, N, D, M, 1, dt), dev, workspace)
    with _on_device(dev):
        st = lib.la_backward_shard_q(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                                     dq.data_ptr(), S0.data_ptr(), Z0.data_ptr(), R_own.data_ptr(),
                                     r_own.data_ptr(), B, H, N, D, M, dt, ws.data_ptr(),
                                     ws.numel() * ws.element_size(), _stream_ptr(dev))
    _check(fn, st)
    return dq, R_own, r_own, ws


def la_backward_shard_kv(q, k, v, dout, R0, r0, workspace, dk=None, dv=None):
    """Second backward pass of a shard: (dk, dv) given the reverse sums (R0, r0) of the tokens
    after it and the workspace of its la_backward_shard_q call."""
    import torch
    fn, f32 = "la_backward_shard_kv", torch.float32
    (B, H, N), D, M = _dims(fn, q, v, 4)
    _expect(fn, "k", k, q.shape, q.dtype)
    _expect(fn, "v", v, (B, H, N, M), q.dtype)
    _expect(fn, "dout", dout, (B, H, N, M), q.dtype)
    sS, sZ = _state_shapes(B, H, D, M)
    _expect(fn, "R0", R0, sS, f32)
    _expect(fn, "r0", r0, sZ, f32)
    given = [(n, t, shp) for n, t, shp in (("dk", dk, (B, H, N, D)), ("dv", dv, (B, H, N, M)))
             if t is not None]
    for name, t, shp in given:
        _expect(fn, name, t, shp, f32)
    dt = _dtype_code(q)
    lib = load_library()
    nbytes = lib.la_backward_workspace_bytes(B, H, N, D, M, 1, dt)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"{fn}: workspace too small")
    _need_cuda(q, k, v, dout, R0, r0, workspace, *[t for _, t, _ in given])
    dev = q.device
    dk = torch.empty((B, H, N, D), dtype=f32, device=dev) if dk is None else dk
    dv = torch.empty((B, H, N, M), dtype=f32, device=dev) if dv is None else dv
    with _on_device(dev):
        st = lib.la_backward_shard_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                                      dk.data_ptr(), dv.data_ptr(), R0.data_ptr(), r0.data_ptr(),
                                      B, H, N, D, M, dt, workspace.data_ptr(),
                                      workspace.numel() * workspace.element_size(),
                                      _stream_ptr(dev))
    _check(fn, st)
    return dk, dv


# ---------------------------------------------- degree-2 polynomial feature map

def la_poly2_workspace_bytes(B, H, N, D, M, causal=True, dtype=LA_BF16):
    return load_library().la_poly2_workspace_bytes(B, H, N, D, M, int(bool(causal)), dtype)


def la_forward_poly2(q, k, v, causal=True, out=None, workspace=None):
    """out[B,H,N,M] = causal attention with sim(q, k) = (q . k)^2 (feature map vec(x x^T))."""
    import torch
    fn = "la_forward_poly2"
    (B, H, N), D, M = _dims(fn, q, v, 4)
    _expect(fn, "k", k, q.shape, q.dtype)
    _expect(fn, "v", v, (B, H, N, M), q.dtype)
    if out is not None:
        _expect(fn, "out", out, (B, H, N, M), q.dtype)
    dt = _dtype_code(q)
    _need_cuda(q, k, v, *([] if out is None else [out]))
    lib = load_library()
    dev = q.device
    out = torch.empty((B, H, N, M), dtype=q.dtype, device=dev) if out is None else out
    ws = _workspace(lib.la_poly2_workspace_bytes(B, H, N, D, M, int(bool(causal)), dt), dev,
                    workspace)
    with _on_device(dev):
        st = lib.la_forward_poly2(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H,
                                  N, D, M, int(bool(causal)), dt, ws.data_ptr(),
                                  ws.numel() * ws.element_size(), _stream_ptr(dev))
    _check(fn, st)
    return out


# ------------------------------------------------------ random Fourier features

def la_rff_workspace_bytes(B, H, N, D, M, F, causal=True, dtype=LA_BF16):
    return load_library().la_rff_workspace_bytes(B, H, N, D, M, F, int(bool(causal)), dtype)


def la_forward_rff(q, k, v, W, bias, causal=True, out=None, workspace=None):
    """out[B,H,N,M] = attention with phi(x) = sqrt(2/F) cos(W x + bias) (random Fourier
    features of the RBF kernel); W [F, D] in q's dtype, bias [F] float32."""
    import torch
    fn = "la_forward_rff"
    (B, H, N), D, M = _dims(fn, q, v, 4)
    _expect(fn, "k", k, q.shape, q.dtype)
    _expect(fn, "v", v, (B, H, N, M), q.dtype)
    if W.dim() != 2:
        raise ValueError(f"{fn}: W must be [F, D]")
    F = W.shape[0]
    _expect(fn, "W", W, (F, D), q.dtype)
    _expect(fn, "bias", bias, (F,), torch.float32)
    if out is not None:
        _expect(fn, "out", out, (B, H, N, M), q.dtype)
    dt = _dtype_code(q)
    _need_cuda(q, k, v, W, bias, *([] if out is None else [out]))
    lib = load_library()
    dev = q.device
    out = torch.empty((B, H, N, M), dtype=q.dtype, device=dev) if out is None else out
    ws = _workspace(lib.la_rff_workspace_bytes(B, H, N, D, M, F, int(bool(causal)), dt), dev,
                    workspace)
    with _on_device(dev):
        st = lib.la_forward_rff(q.data_ptr(), k.data_ptr(), v.data_ptr(), W.data_ptr(),
                                bias.data_ptr(), out.data_ptr(), B, H, N, D, M, F,
                                int(bool(causal)), dt, ws.data_ptr(),
                                ws.numel() * ws.element_size(), _stream_ptr(dev))
    _check(fn, st)
    return out
