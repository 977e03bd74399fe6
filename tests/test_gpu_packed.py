"""GPU parity of la_extend_packed: streams of different lengths stored back to
back in one token-major batch ([T][H][D], stream b in rows cu[b] .. cu[b+1]-1),
each continuing from its pool entry's state. Every stream's outputs and advanced
state are compared with the fp64 recurrence from that state (the oracle); rows
of no stream must keep what they held, and bad offsets must be reported.
"""

import numpy as np
import pytest

import oracle
from kernelized_causal_self_gb300 import inputs
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
SENTINEL = 7.0


@pytest.fixture(scope="module")
def la():
    from kernelized_causal_self_gb300 import build
    build.build()
    import kernelized_causal_self_gb300 as pkg
    pkg.load_library()
    return pkg


def _t(x, dtype):
    return inputs.to_torch(x, dtype, DEV)


def _offsets(lens):
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return cu


def _packed_inputs(seed, T, H, D, M, dt, tail_nan):
    """q, k [T, H, D], v [T, H, M]; the last `tail_nan` rows (no stream's) are NaN."""
    scale = 0.125 if dt == inputs.BF16 else 1.0
    q, k, v = inputs.qkv(seed, 1, H, T, D, M, scale, dt)
    q, k, v = (np.ascontiguousarray(x[0].transpose(1, 0, 2)) for x in (q, k, v))
    if tail_nan:
        for x in (q, k, v):
            x[T - tail_nan:] = np.nan
    return q, k, v


def _pool(seed, P, H, D, M):
    S0 = np.abs(inputs.normal(seed, (P, H, D, M), 1.0, inputs.F32, 0)) * 4.0
    Z0 = np.abs(inputs.normal(seed, (P, H, D), 1.0, inputs.F32, 1)) * 4.0 + 1.0
    return S0, Z0


def _run(la, q, k, v, S0, Z0, cu, max_len, slots, dt, ws=None):
    T, H, M = v.shape
    tS, tZ = _t(S0, inputs.F32), _t(Z0, inputs.F32)
    out = torch.full((T, H, M), SENTINEL, dtype=torch.bfloat16 if dt == inputs.BF16
                     else torch.float32, device=DEV)
    la.la_extend_packed(_t(q, dt), _t(k, dt), _t(v, dt), tS, tZ,
                        torch.from_numpy(cu).to(DEV), max_len,
                        slots=None if slots is None else torch.from_numpy(slots).to(DEV),
                        out=out, workspace=ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), tS.cpu().numpy(), tZ.cpu().numpy()


def _check_stream(got_out, got_S, got_Z, q, k, v, S0, Z0, a, n, slot, dt, tag):
    """Stream in rows a .. a+n-1 against the recurrence from pool entry `slot`."""
    qs, ks, vs = (x[a:a + n].transpose(1, 0, 2) for x in (q, k, v))  # [H, n, .]
    want, S_ref, Z_ref = oracle.recurrent_attention(qs, ks, vs, S0[slot], Z0[slot])
    if n:
        assert_close(got_out[a:a + n].transpose(1, 0, 2), want, dt, f"{tag} out")
    assert_close(got_S[slot], S_ref, dt, f"{tag} S")
    assert_close(got_Z[slot], Z_ref, dt, f"{tag} Z")


# (stream lengths, H, D, M, dtype, max_len): the tensor-core path through the
# segment scan (several chunks, ragged ends, empty streams, a stream ending on a
# chunk boundary), its one-chunk path (max_len <= 128), and the CUDA-core path
PACKED = [
    ((300, 129, 0, 257, 1, 128, 517), 2, 64, 64, inputs.BF16, 600),
    ((100, 1, 37, 0, 128, 64), 2, 64, 64, inputs.BF16, 128),
    ((45, 12, 0, 33), 3, 32, 48, inputs.F32, 45),
]


@pytest.mark.parametrize("case", PACKED, ids=lambda c: "n%d-h%dd%dm%d-%s-max%d" % (
    len(c[0]), *c[1:]))
def test_extend_packed_against_recurrence(la, case):
    lens, H, D, M, dt, max_len = case
    B, tail = len(lens), 5
    P = 2 * B + 1
    cu = _offsets(lens)
    T = int(cu[-1]) + tail
    q, k, v = _packed_inputs(900 + B, T, H, D, M, dt, tail)
    S0, Z0 = _pool(901, P, H, D, M)
    slots = np.array([(2 * b + 1) % P for b in range(B)], dtype=np.int32)  # distinct, permuted
    got, gS, gZ = _run(la, q, k, v, S0, Z0, cu, max_len, slots, dt)
    for b in range(B):
        _check_stream(got, gS, gZ, q, k, v, S0, Z0, int(cu[b]), lens[b], slots[b], dt,
                      f"stream {b}")
    assert np.all(got[T - tail:] == SENTINEL), "rows of no stream were written"
    untouched = sorted(set(range(P)) - set(slots.tolist()))
    assert np.array_equal(gS[untouched], S0[untouched].astype(np.float32))
    assert np.array_equal(gZ[untouched], Z0[untouched].astype(np.float32))


def test_extend_packed_equals_padded_extend(la):
    """The packed call and la_extend on the same streams padded to max_len (with
    per-stream lengths) give the same outputs and states."""
    lens, H, D, M, dt = (211, 3, 128, 140), 2, 64, 64, inputs.BF16
    B, N = len(lens), max(lens)
    cu = _offsets(lens)
    q, k, v = _packed_inputs(910, int(cu[-1]), H, D, M, dt, 0)
    S0, Z0 = _pool(911, B, H, D, M)
    got, gS, gZ = _run(la, q, k, v, S0, Z0, cu, N, None, dt)
    pad = [np.zeros((B, H, N, x.shape[-1]), np.float32) for x in (q, k, v)]
    for b, n in enumerate(lens):
        for dst, src in zip(pad, (q, k, v)):
            dst[b, :, :n] = src[cu[b]:cu[b] + n].transpose(1, 0, 2)
    tS, tZ = _t(S0, inputs.F32), _t(Z0, inputs.F32)
    o = la.la_extend(*(_t(x, dt) for x in pad), tS, tZ,
                     lens=torch.tensor(lens, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    o = o.float().cpu().numpy()
    for b, n in enumerate(lens):
        assert np.array_equal(got[cu[b]:cu[b] + n], o[b, :, :n].transpose(1, 0, 2)), f"out[{b}]"
    assert np.array_equal(gS, tS.cpu().numpy())
    assert np.array_equal(gZ, tZ.cpu().numpy())


@pytest.mark.parametrize("max_len", [300, 100])
def test_extend_packed_reports_bad_offsets(la, max_len):
    """A stream that starts before row 0 or ends past row T is empty; one longer than
    max_len runs over its first max_len tokens and leaves its other rows alone; both
    are reported, and nothing else is written."""
    H, D, M, dt = 2, 64, 64, inputs.BF16
    T = 700
    cu = np.array([-10, 90, 400, 750], dtype=np.int32)  # 0: starts at -10; 2: ends past T
    q, k, v = _packed_inputs(920, T, H, D, M, dt, 0)
    S0, Z0 = _pool(921, 3, H, D, M)
    nbytes = la.la_forward_workspace_bytes(3, H, max_len, D, M, True, la.LA_BF16)
    ws = torch.zeros((nbytes,), dtype=torch.uint8, device=DEV)
    got, gS, gZ = _run(la, q, k, v, S0, Z0, cu, max_len, None, dt, ws)
    assert la.la_workspace_status(ws) == la.LA_ERR_INVALID_ARG
    n1 = min(310, max_len)
    _check_stream(got, gS, gZ, q, k, v, S0, Z0, 90, n1, 1, dt, "stream 1")
    assert np.all(got[:90] == SENTINEL) and np.all(got[90 + n1:] == SENTINEL), \
        "rows of an empty stream or past max_len were written"
    for b in (0, 2):
        assert np.array_equal(gS[b], S0[b].astype(np.float32)), f"empty stream {b}'s state moved"
        assert np.array_equal(gZ[b], Z0[b].astype(np.float32))


def test_extend_packed_serving_batch_sampled(la):
    """256 streams of 1..1024 tokens (8 heads, 131k tokens in all) from a pool of
    512 states: eight streams checked one by one against the recurrence, every
    advanced state checked for finiteness and every row of the batch written."""
    B, H, D, M, dt, P = 256, 8, 64, 64, inputs.BF16, 512
    lens = inputs.stream_lengths(930, B, 1, 1024)
    cu = _offsets(lens)
    T = int(cu[-1])
    q, k, v = _packed_inputs(931, T, H, D, M, dt, 0)
    S0, Z0 = _pool(932, P, H, D, M)
    slots = np.array([(5 * b + 3) % P for b in range(B)], dtype=np.int32)
    got, gS, gZ = _run(la, q, k, v, S0, Z0, cu, int(lens.max()), slots, dt)
    assert not np.any(got == SENTINEL), "a row of the batch was not written"
    assert np.all(np.isfinite(gS[slots])) and np.all(np.isfinite(gZ[slots]))
    for b in (0, 1, 17, 64, 100, 191, 254, 255):
        _check_stream(got, gS, gZ, q, k, v, S0, Z0, int(cu[b]), int(lens[b]), slots[b], dt,
                      f"stream {b}")
