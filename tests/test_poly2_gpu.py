"""The degree-2 polynomial feature map (paperlayer.ai summary §3.2.1: sim(x, y) =
(x . y)^2 has the exact finite feature map vec(x x^T)) on the CUDA path, against
the fp64 oracle run with that feature map: the explicit masked form and the S/Z
recurrence over the 4096 features on small shapes (tiles, ragged tails, N = 1),
and sampled rows of the full B4 H8 N16384 workload. bf16 tolerance as
elsewhere (tests/helpers.py)."""

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


def _run(la, seed, B, H, N, scale=0.125):
    q, k, v = inputs.qkv(seed, B, H, N, 64, 64, scale, inputs.BF16)
    out = la.la_forward_poly2(*(inputs.to_torch(x, inputs.BF16, DEV) for x in (q, k, v)))
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (q, k, v)


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 2, 5), (2, 1, 127), (1, 2, 128), (2, 2, 129),
                                   (1, 1, 300), (1, 2, 641)], ids=lambda s: "b%dh%dn%d" % s)
def test_poly2_matches_the_masked_form(la, shape):
    B, H, N = shape
    got, (q, k, v) = _run(la, 1300 + N, B, H, N)
    want = oracle.masked_attention(q, k, v, causal=True, feature=oracle.poly2_feature)
    assert_close(got, want, "bf16", f"poly2 out {shape}")


def test_poly2_matches_the_recurrence(la):
    B, H, N = 1, 1, 260
    got, (q, k, v) = _run(la, 1400, B, H, N, scale=0.25)
    want, _, _ = oracle.recurrent_attention(q, k, v, feature=oracle.poly2_feature)
    assert_close(got, want, "bf16", "poly2 out vs the recurrence")


def test_poly2_full_size_sampled_rows(la):
    w = inputs.WORKLOADS["causal_fwdbwd_b4h8n16384d64"]
    g = torch.Generator(device=DEV)
    g.manual_seed(w.seed + 7)
    q, k, v = (inputs.torch_normal(g, (w.B, w.H, w.N, 64), w.scale, w.dtype, DEV) for _ in range(3))
    out = la.la_forward_poly2(q, k, v)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    rows = [0, 1, 127, 128, 129, 5000, w.N - 129, w.N - 1]
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        f = lambda t: t[b, h].float().cpu().numpy().astype("float64")  # noqa: E731
        want = oracle.masked_attention_rows(f(q), f(k), f(v), rows, feature=oracle.poly2_feature)
        assert_close(f(out)[rows], want, "bf16", f"poly2 rows of [{b},{h}]")


def test_poly2_rejects_unsupported_shapes(la):
    q = torch.zeros((1, 1, 8, 32), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(la.LAError):
        la.la_forward_poly2(q, q, q)                            # D = 32
    q = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(la.LAError):
        la.la_forward_poly2(q, q, q, causal=False)              # causal only
    with pytest.raises(la.LAError):
        la.la_forward_poly2(q.float(), q.float(), q.float())    # bf16 only
