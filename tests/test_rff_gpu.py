"""Random Fourier features of the RBF kernel (named by paperlayer.ai summary §5 as the
next feature map; the definition taken is Rahimi and Recht's, phi(x) = sqrt(2/F)
cos(W x + b)) on the CUDA path, against the fp64 oracle run with that feature map:
the explicit masked form (causal and not) on small shapes across tiles and ragged
tails, and sampled rows of the B4 H8 N16384 workload. W (F x D, rows ~ N(0, I), on
the bf16 grid) and b (uniform on [0, 2 pi)) are seeded inputs. For these inputs every
denominator stays above 0.16 per summed token (checked in the oracle's own terms), so
the quotients are well conditioned."""

import numpy as np
import pytest

import oracle
from kernelized_causal_self_gb300 import inputs
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
F = 64


@pytest.fixture(scope="module")
def la():
    from kernelized_causal_self_gb300 import build
    build.build()
    import kernelized_causal_self_gb300 as pkg
    pkg.load_library()
    return pkg


def _draws(seed):
    W = inputs.normal(seed, (F, 64), 1.0, inputs.BF16, 7)
    b = inputs.uniform(seed, (F,), 0.0, 2.0 * np.pi, 8)
    return W, b


def _feature(W, b):
    return lambda x: oracle.random_fourier_feature(x, W, b)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 3, 200), (2, 2, 129), (1, 2, 1000)],
                         ids=lambda s: "b%dh%dn%d" % s)
def test_rff_matches_the_masked_form(la, shape, causal):
    B, H, N = shape
    seed = 1600 + N
    q, k, v = inputs.qkv(seed, B, H, N, 64, 64, 0.125, inputs.BF16)
    W, b = _draws(seed)
    t = lambda x: inputs.to_torch(x, inputs.BF16, DEV)  # noqa: E731
    out = la.la_forward_rff(t(q), t(k), t(v), t(W), torch.from_numpy(b).to(DEV), causal=causal)
    torch.cuda.synchronize()
    want = oracle.masked_attention(q, k, v, causal=causal, feature=_feature(W, b))
    assert_close(out.float().cpu().numpy(), want, "bf16", f"rff out {shape} causal={causal}")


def test_rff_full_size_sampled_rows(la):
    w = inputs.WORKLOADS["causal_fwdbwd_b4h8n16384d64"]
    g = torch.Generator(device=DEV)
    g.manual_seed(w.seed + 11)
    q, k, v = (inputs.torch_normal(g, (w.B, w.H, w.N, 64), w.scale, w.dtype, DEV) for _ in range(3))
    W, b = _draws(1700)
    out = la.la_forward_rff(q, k, v, inputs.to_torch(W, inputs.BF16, DEV), torch.from_numpy(b).to(DEV))
    torch.cuda.synchronize()
    rows = [0, 1, 127, 128, 5000, w.N - 1]
    for bb, h in ((0, 0), (w.B - 1, w.H - 1)):
        f = lambda x: x[bb, h].float().cpu().numpy().astype("float64")  # noqa: E731
        want = oracle.masked_attention_rows(f(q), f(k), f(v), rows, feature=_feature(W, b))
        assert_close(f(out)[rows], want, "bf16", f"rff rows of [{bb},{h}]")


def test_rff_rejects_unsupported_shapes(la):
    q = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16, device=DEV)
    b = torch.zeros((32,), dtype=torch.float32, device=DEV)
    with pytest.raises(la.LAError):   # F = 32
        la.la_forward_rff(q, q, q, torch.zeros((32, 64), dtype=torch.bfloat16, device=DEV), b)
    with pytest.raises(ValueError):   # bias of the wrong length
        la.la_forward_rff(q, q, q, torch.zeros((64, 64), dtype=torch.bfloat16, device=DEV), b)
