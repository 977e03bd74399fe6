"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every symbol include/la.h declares, and rejects bad arguments on the
host before anything is launched."""

import ctypes
import os
import re
import subprocess

import pytest

import kernelized_causal_self_gb300 as la
from kernelized_causal_self_gb300 import build as labuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]

FAKE = 0x10000      # 16-byte aligned, never dereferenced: every call below returns first
ODD = 0x10008       # 8-byte aligned only


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(la_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    labuild.build()
    return la.load_library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("la_forward", "la_backward", "la_decode_step", "la_prefill", "la_extend",
              "la_extend_packed", "la_forward_workspace_bytes", "la_backward_workspace_bytes",
              "la_status_string", "la_workspace_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", la.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (la_\w+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)


def test_binding_mirrors_the_abi_names():
    for n in ("la_forward", "la_backward", "la_decode_step", "la_prefill", "la_extend",
              "la_extend_packed", "la_forward_workspace_bytes", "la_backward_workspace_bytes",
              "la_status_string", "la_workspace_status"):
        assert callable(getattr(la, n))


def test_status_strings(lib):
    for code in range(0, 6):
        s = lib.la_status_string(code)
        assert s and len(s) > 1
    assert lib.la_status_string(0) == b"ok"
    assert lib.la_version() >= 100


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, H=1, N=16, D=64, M=64, causal=1, dtype=1,
         ws=FAKE, wsb=1 << 20):
    return lib.la_forward(q, k, v, out, B, H, N, D, M, causal, dtype, ws, wsb, None)


def test_forward_rejects_bad_arguments(lib):
    assert _fwd(lib, q=0) == la.LA_ERR_INVALID_ARG
    assert _fwd(lib, out=ODD) == la.LA_ERR_INVALID_ARG
    for D, M in ((0, 64), (12, 64), (64, 7), (136, 64), (64, 256)):
        assert _fwd(lib, D=D, M=M) == la.LA_ERR_INVALID_ARG
    assert _fwd(lib, B=0) == la.LA_ERR_INVALID_ARG
    assert _fwd(lib, N=-1) == la.LA_ERR_INVALID_ARG
    assert _fwd(lib, dtype=7) == la.LA_ERR_INVALID_ARG
    assert _fwd(lib, ws=0) == la.LA_ERR_WORKSPACE
    assert _fwd(lib, ws=ODD) == la.LA_ERR_WORKSPACE
    assert _fwd(lib, wsb=16) == la.LA_ERR_WORKSPACE


def _ext(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, S=FAKE, Z=FAKE, slots=FAKE, lens=FAKE, pool=4, B=2,
         H=1, N=16, D=64, M=64, dtype=1, ws=FAKE, wsb=1 << 20):
    return lib.la_extend(q, k, v, out, S, Z, slots, lens, pool, B, H, N, D, M, dtype, ws, wsb, None)


def _extp(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, S=FAKE, Z=FAKE, slots=FAKE, cu=FAKE, pool=4, B=2,
          H=1, T=64, max_len=16, D=64, M=64, dtype=1, ws=FAKE, wsb=1 << 20):
    return lib.la_extend_packed(q, k, v, out, S, Z, slots, cu, pool, B, H, T, max_len, D, M, dtype,
                                ws, wsb, None)


def test_extend_packed_rejects_bad_arguments(lib):
    assert _extp(lib, cu=0) == la.LA_ERR_INVALID_ARG
    assert _extp(lib, cu=FAKE + 2) == la.LA_ERR_INVALID_ARG          # offsets 4-byte aligned
    assert _extp(lib, slots=FAKE + 2) == la.LA_ERR_INVALID_ARG
    assert _extp(lib, S=0) == la.LA_ERR_INVALID_ARG
    assert _extp(lib, q=ODD) == la.LA_ERR_INVALID_ARG
    assert _extp(lib, pool=1, slots=0) == la.LA_ERR_INVALID_ARG      # identity slots need B
    assert _extp(lib, T=-1) == la.LA_ERR_INVALID_ARG
    assert _extp(lib, T=(1 << 30) + 1) == la.LA_ERR_INVALID_ARG
    assert _extp(lib, max_len=-1) == la.LA_ERR_INVALID_ARG
    assert _extp(lib, B=0) == la.LA_ERR_INVALID_ARG
    assert _extp(lib, D=12) == la.LA_ERR_INVALID_ARG
    assert _extp(lib, dtype=7) == la.LA_ERR_INVALID_ARG
    assert _extp(lib, ws=0) == la.LA_ERR_WORKSPACE
    assert _extp(lib, wsb=16) == la.LA_ERR_WORKSPACE
    assert _extp(lib, T=0) == la.LA_OK                               # nothing to do
    assert _extp(lib, max_len=0) == la.LA_OK


def test_extend_rejects_bad_arguments(lib):
    assert _ext(lib, S=0) == la.LA_ERR_INVALID_ARG
    assert _ext(lib, Z=ODD) == la.LA_ERR_INVALID_ARG
    assert _ext(lib, slots=FAKE + 2) == la.LA_ERR_INVALID_ARG        # slots must be 4-byte aligned
    assert _ext(lib, lens=FAKE + 2) == la.LA_ERR_INVALID_ARG         # lens too
    assert _ext(lib, pool=0) == la.LA_ERR_INVALID_ARG
    assert _ext(lib, slots=0, pool=1, B=2) == la.LA_ERR_INVALID_ARG  # identity slots need B entries
    assert _ext(lib, D=12) == la.LA_ERR_INVALID_ARG
    assert _ext(lib, q=0) == la.LA_ERR_INVALID_ARG
    assert _ext(lib, ws=0) == la.LA_ERR_WORKSPACE
    assert _ext(lib, wsb=16) == la.LA_ERR_WORKSPACE
    assert _ext(lib, q=0, k=0, v=0, out=0, N=0) == la.LA_OK           # nothing to extend


def test_empty_sequence_is_a_noop(lib):
    assert _fwd(lib, q=0, k=0, v=0, out=0, N=0) == la.LA_OK
    assert lib.la_backward(0, 0, 0, 0, 0, 0, 0, 1, 1, 0, 64, 64, 1, 1, 0, 0, None) == la.LA_OK


def test_backward_and_decode_reject_bad_arguments(lib):
    ws = lib.la_backward_workspace_bytes(1, 1, 16, 64, 64, 1, 1)
    args = [FAKE] * 7 + [1, 1, 16, 64, 64, 1, 1, FAKE, ws, None]
    assert lib.la_backward(*args[:6], 0, *args[7:]) == la.LA_ERR_INVALID_ARG
    assert lib.la_backward(*args[:14], FAKE, ws - 1, None) == la.LA_ERR_WORKSPACE
    assert lib.la_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 8, 64, 64, 1, None) == \
        la.LA_ERR_INVALID_ARG
    assert lib.la_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 60, 64, 1, None) == \
        la.LA_ERR_INVALID_ARG
    assert lib.la_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, 64, 64, 1, None) == \
        la.LA_ERR_INVALID_ARG


def test_workspace_sizes(lib):
    for causal in (0, 1):
        a = lib.la_forward_workspace_bytes(4, 8, 1024, 64, 64, causal, 1)
        b = lib.la_forward_workspace_bytes(4, 8, 16384, 64, 64, causal, 1)
        assert 256 <= a <= b
        c = lib.la_backward_workspace_bytes(4, 8, 1024, 64, 64, causal, 1)
        d = lib.la_backward_workspace_bytes(4, 8, 16384, 64, 64, causal, 1)
        assert 256 <= c <= d
        assert a % 16 == 0 and c % 16 == 0


def test_workspace_queries_of_rejected_shapes_need_only_the_header(lib):
    # B * H beyond an int, and non-positive sizes: the entry points reject these,
    # so the queries answer with the 256-byte header alone (no overflowed product)
    # (65537 * 65537 wraps to +131073 in 32 bits, 46341 * 46341 to a negative int)
    for B, H, N in ((65537, 65537, 128), (46341, 46341, 128), (0, 8, 16), (4, 8, -1)):
        for causal in (0, 1):
            assert lib.la_forward_workspace_bytes(B, H, N, 64, 64, causal, 1) == 256
            assert lib.la_backward_workspace_bytes(B, H, N, 64, 64, causal, 1) == 256


def test_fault_hooks_reject_bad_arguments(lib):
    lib.la_debug_forward_fault.restype = ctypes.c_int
    ok = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, H=2, N=1000, D=64, M=64, causal=1, dtype=1,
              ws=FAKE, wsb=1 << 24, load=1, ns=100_000)

    for hook in (lib.la_debug_forward_fault, lib.la_debug_forward_fused_fault):
        hook.restype = ctypes.c_int

        def fwd(**kw):
            a = dict(ok, **kw)
            return hook(a["q"], a["k"], a["v"], a["out"], a["B"], a["H"], a["N"], a["D"], a["M"],
                        a["causal"], a["dtype"], a["ws"], a["wsb"], a["load"], a["ns"], None)
        assert fwd(dtype=0) == la.LA_ERR_INVALID_ARG        # float32: not the tensor-core path
        assert fwd(D=32, M=32) == la.LA_ERR_INVALID_ARG     # D = M = 64 only
        assert fwd(load=-1) == la.LA_ERR_INVALID_ARG
        assert fwd(ns=10) == la.LA_ERR_INVALID_ARG          # below 1 us
        assert fwd(ns=3_000_000_000) == la.LA_ERR_INVALID_ARG
        assert fwd(N=0) == la.LA_ERR_INVALID_ARG
        assert fwd(q=0) == la.LA_ERR_INVALID_ARG
        assert fwd(ws=0) == la.LA_ERR_WORKSPACE
        assert fwd(wsb=16) == la.LA_ERR_WORKSPACE
    args = [FAKE] * 7 + [1, 2, 1000, 64, 64, 1, 0, FAKE, 1 << 24, 1, 100_000, None]
    assert lib.la_debug_backward_fault(*args) == la.LA_ERR_INVALID_ARG   # dtype float32
    args[13] = 1
    args[16] = -2
    assert lib.la_debug_backward_fault(*args) == la.LA_ERR_INVALID_ARG   # negative load number
    assert lib.la_workspace_wait_site(None, 0, None) == -1


def test_shard_entry_points_reject_bad_arguments(lib):
    wsf = lib.la_forward_workspace_bytes(1, 2, 300, 64, 64, 1, 1)
    wsb = lib.la_backward_workspace_bytes(1, 2, 300, 64, 64, 1, 1)
    # la_state_sums(k, v, S, Z, B, H, N, D, M, dtype, ws, wsb, stream)
    assert lib.la_state_sums(FAKE, FAKE, 0, FAKE, 1, 2, 300, 64, 64, 1, FAKE, wsf, None) == \
        la.LA_ERR_INVALID_ARG
    assert lib.la_state_sums(FAKE, FAKE, FAKE, FAKE, 1, 2, 300, 64, 60, 1, FAKE, wsf, None) == \
        la.LA_ERR_INVALID_ARG
    assert lib.la_state_sums(0, FAKE, FAKE, FAKE, 1, 2, 300, 64, 64, 1, FAKE, wsf, None) == \
        la.LA_ERR_INVALID_ARG
    assert lib.la_state_sums(FAKE, FAKE, FAKE, FAKE, 1, 2, 300, 64, 64, 1, FAKE, 16, None) == \
        la.LA_ERR_WORKSPACE
    # la_forward_shard(q, k, v, out, S0, Z0, B, H, N, D, M, dtype, ws, wsb, stream)
    assert lib.la_forward_shard(FAKE, FAKE, FAKE, FAKE, ODD, FAKE, 1, 2, 300, 64, 64, 1, FAKE, wsf,
                                None) == la.LA_ERR_INVALID_ARG
    assert lib.la_forward_shard(FAKE, FAKE, FAKE, 0, FAKE, FAKE, 1, 2, 300, 64, 64, 1, FAKE, wsf,
                                None) == la.LA_ERR_INVALID_ARG
    assert lib.la_forward_shard(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 300, 64, 64, 1, 0, wsf,
                                None) == la.LA_ERR_WORKSPACE
    assert lib.la_forward_shard(0, 0, 0, 0, FAKE, FAKE, 1, 2, 0, 64, 64, 1, 0, 0, None) == la.LA_OK
    # la_backward_shard_q(q, k, v, dout, dq, S0, Z0, R_own, r_own, B, H, N, D, M, dtype, ws, wsb, st)
    args = [FAKE] * 9 + [1, 2, 300, 64, 64, 1, FAKE, wsb, None]
    bad = list(args)
    bad[7] = 0                                                   # R_own missing
    assert lib.la_backward_shard_q(*bad) == la.LA_ERR_INVALID_ARG
    bad = list(args)
    bad[16] = wsb - 1
    assert lib.la_backward_shard_q(*bad) == la.LA_ERR_WORKSPACE
    # la_backward_shard_kv(q, k, v, dout, dk, dv, R0, r0, B, H, N, D, M, dtype, ws, wsb, st)
    args = [FAKE] * 8 + [1, 2, 300, 64, 64, 1, FAKE, wsb, None]
    bad = list(args)
    bad[6] = ODD
    assert lib.la_backward_shard_kv(*bad) == la.LA_ERR_INVALID_ARG
    bad = list(args)
    bad[15] = 0
    assert lib.la_backward_shard_kv(*bad) == la.LA_ERR_WORKSPACE


def test_backward_from_forward_rejects_bad_arguments(lib):
    wsb = lib.la_backward_workspace_bytes(1, 2, 300, 64, 64, 1, 1)
    wsf = lib.la_forward_workspace_bytes(1, 2, 300, 64, 64, 1, 1)
    args = [FAKE] * 7 + [1, 2, 300, 64, 64, 1, 1, FAKE, wsf, FAKE, wsb, None]
    bad = list(args)
    bad[4] = 0                                  # dq missing
    assert lib.la_backward_from_forward(*bad) == la.LA_ERR_INVALID_ARG
    bad = list(args)
    bad[14] = 0                                 # no forward workspace
    assert lib.la_backward_from_forward(*bad) == la.LA_ERR_WORKSPACE
    bad = list(args)
    bad[15] = wsf - 16                          # forward workspace too small for this shape
    assert lib.la_backward_from_forward(*bad) == la.LA_ERR_WORKSPACE
    bad = list(args)
    bad[17] = 16                                # backward workspace too small
    assert lib.la_backward_from_forward(*bad) == la.LA_ERR_WORKSPACE
