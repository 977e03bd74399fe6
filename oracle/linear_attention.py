"""Plain fp64 CPU oracle for kernelized (linear) attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, links or runs
this module; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it. It shares no code with the CUDA library.

Sources (web pages on *Transformers are RNNs: Fast Autoregressive Transformers
with Linear Attention*, Katharopoulos et al., ICML 2020), cited below as:

* [review]  -- "[Paper Review] Transformers are RNNs: ..." (nubint.ai),
               section "Proposed method".
* [summary] -- "Transformers are RNNs: Fast Autoregressive Transformers with
               Linear Attention" (paperlayer.ai); sections numbered as in the
               paper (§3.1, §3.2, §3.2.1, §3.3, §3.3.1, §3.4, App. A).
* [deck]    -- "Transformers are RNNs: ... 解读" (zhengyuhong.cn slide deck);
               slides numbered 1-9 (slide 3: associativity, slide 4: the S/Z
               prefix recurrence).

Notation (row-wise): per (batch, head) Q, K are N x D, V is N x M; Q_i is a
D-vector, V_i an M-vector; phi acts elementwise.

Every function is written for clarity, in float64, with no blocking, chunking
or fusion beyond what the formula states. Arrays may carry leading batch axes
(e.g. [B, H, N, D]); all formulas act on the last two axes.
"""

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# Feature maps
# ---------------------------------------------------------------------------

def elu_plus_one(x):
    """phi(x) = elu(x) + 1 with the standard ELU (alpha = 1).

    [summary §3.2.1] and [deck slide 3] name phi(x) = elu(x) + 1 as the map used
    in the experiments; it keeps every similarity positive. The ELU slope alpha
    is not printed; the standard alpha = 1 is taken, which makes phi equal to
    x + 1 for x > 0 and exp(x) for x <= 0 (continuous, value 1 and slope 1 at 0).
    """
    x = np.asarray(x, dtype=F64)
    return np.where(x > 0.0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def elu_plus_one_grad(x):
    """d phi / dx for phi = elu + 1: 1 for x > 0, exp(x) for x <= 0."""
    x = np.asarray(x, dtype=F64)
    return np.where(x > 0.0, 1.0, np.exp(np.minimum(x, 0.0)))


def poly2_feature(x):
    """Exact finite feature map of the degree-2 polynomial kernel.

    [summary §3.2.1]: the degree-2 polynomial kernel sim(x, y) = (x . y)^2 has an
    exact finite feature map, phi(x) = vec(x x^T) (dimension D^2), since
    vec(x x^T) . vec(y y^T) = (x . y)^2. Used only to check the oracle's own
    associative machinery against an explicit kernel sum.
    """
    x = np.asarray(x, dtype=F64)
    outer = x[..., :, None] * x[..., None, :]
    return outer.reshape(x.shape[:-1] + (x.shape[-1] * x.shape[-1],))


def random_fourier_feature(x, W, b):
    """Random Fourier features of the RBF kernel.

    [summary §5] names random Fourier features, approximating the RBF kernel, as the
    feature map to try next, without a definition. The plainest one, the random
    Fourier features of Rahimi and Recht (2007): with the F rows w_f of W drawn
    i.i.d. N(0, sigma^-2 I) and b_f uniform on [0, 2 pi),
        phi(x) = sqrt(2 / F) [cos(w_1 . x + b_1), ..., cos(w_F . x + b_F)],
    so that E[phi(x) . phi(y)] = exp(-|x - y|^2 / (2 sigma^2)). The draws are inputs:
    W is [F, D], b is [F]; x is [..., D]; returns [..., F].
    """
    x = np.asarray(x, dtype=F64)
    W = np.asarray(W, dtype=F64)
    b = np.asarray(b, dtype=F64)
    F = W.shape[0]
    return np.sqrt(2.0 / F) * np.cos(x @ W.T + b)


# ---------------------------------------------------------------------------
# Forward: three independent forms of the same result
# ---------------------------------------------------------------------------

def masked_attention(q, k, v, causal=True, feature=elu_plus_one):
    """Explicit O(N^2) kernel attention.

    [summary §3.1]: generalized attention replaces the softmax weight by any
    non-negative similarity, V'_i = sum_j sim(Q_i, K_j) V_j / sum_j sim(Q_i, K_j);
    with sim(x, y) = phi(x) . phi(y) ([review], [deck slide 3]).
    [summary §3.3], [deck slide 4]: causal masking lets position i see only
    positions j <= i (inclusive).
    """
    fq = feature(q)
    fk = feature(k)
    v = np.asarray(v, dtype=F64)
    sim = fq @ np.swapaxes(fk, -1, -2)          # [..., N, N], sim[i, j]
    if causal:
        n = sim.shape[-1]
        sim = sim * np.tril(np.ones((n, n), dtype=F64))
    return (sim @ v) / sim.sum(axis=-1, keepdims=True)


def masked_attention_rows(q, k, v, rows, feature=elu_plus_one):
    """The causal masked form of masked_attention at selected query rows only.

    Same definition ([summary §3.1], [summary §3.3]: out_i = sum_{j<=i}
    sim(Q_i, K_j) V_j / sum_{j<=i} sim(Q_i, K_j)), evaluated one row at a time,
    so that long sequences can be checked where the N x N similarity matrix
    would not fit. q, k: [N, D] and v: [N, M] of one sequence; rows: query
    positions. Returns [len(rows), M].
    """
    fk = feature(k)
    v = np.asarray(v, dtype=F64)
    out = []
    for i in rows:
        w = fk[: i + 1] @ feature(q[i])         # sim(Q_i, K_j) for j <= i
        out.append((w @ v[: i + 1]) / w.sum())
    return np.stack(out)


def linearized_attention(q, k, v, feature=elu_plus_one):
    """Non-causal linear attention by associativity.

    [review, "Proposed method"]: V' = phi(Q) (phi(K)^T V) / (phi(Q)^T sum_j
    phi(K_j)), with S = sum_j phi(K_j) V_j^T and Z = sum_j phi(K_j) shared by all
    queries. [deck slide 3]: (phi(Q) phi(K)^T) V = phi(Q) (phi(K)^T V).
    Returns (out, S, Z).
    """
    fq = feature(q)
    fk = feature(k)
    v = np.asarray(v, dtype=F64)
    S = np.swapaxes(fk, -1, -2) @ v             # [..., D, M]
    Z = fk.sum(axis=-2)                         # [..., D]
    num = fq @ S                                # [..., N, M]
    den = fq @ Z[..., :, None]                  # [..., N, 1]
    return num / den, S, Z


def recurrent_attention(q, k, v, S0=None, Z0=None, feature=elu_plus_one):
    """Causal linear attention as the S/Z prefix recurrence.

    [deck slide 4]: S_i = S_{i-1} + phi(K_i) V_i^T, Z_i = Z_{i-1} + phi(K_i), and
    the output at i is phi(Q_i)^T S_i / (phi(Q_i)^T Z_i). [summary §3.3]: each
    step is a constant-time update. S0, Z0 are the state before position 0
    (zero by default). Returns (out, S_N, Z_N).
    """
    fq = feature(q)
    fk = feature(k)
    v = np.asarray(v, dtype=F64)
    lead = fq.shape[:-2]
    n, d = fq.shape[-2], fq.shape[-1]
    m = v.shape[-1]
    S = np.zeros(lead + (d, m), dtype=F64) if S0 is None else np.array(S0, dtype=F64)
    Z = np.zeros(lead + (d,), dtype=F64) if Z0 is None else np.array(Z0, dtype=F64)
    out = np.empty(lead + (n, m), dtype=F64)
    for i in range(n):
        S = S + fk[..., i, :, None] * v[..., i, None, :]
        Z = Z + fk[..., i, :]
        num = np.einsum("...d,...dm->...m", fq[..., i, :], S)
        den = np.einsum("...d,...d->...", fq[..., i, :], Z)
        out[..., i, :] = num / den[..., None]
    return out, S, Z


def forward(q, k, v, causal=True):
    """The operator the library computes: causal or non-causal, phi = elu + 1."""
    if causal:
        return recurrent_attention(q, k, v)[0]
    return linearized_attention(q, k, v)[0]


def prefill(q, k, v):
    """Causal forward that also returns the final state (S_N, Z_N).

    [summary §3.4], [review, "Proposed method"]: the causally masked layer is an
    RNN whose hidden state is the attention memory s and normalizer memory z.
    """
    return recurrent_attention(q, k, v)


def decode_step(q, k, v, S, Z):
    """One autoregressive step on carried state: update, then read out.

    [deck slide 4] and [summary §3.3.2]: inference keeps S, Z and per token first
    adds the new key/value, S <- S + phi(k) v^T, Z <- Z + phi(k), then reads out
    phi(q)^T S / phi(q)^T Z (S_i contains token i). q, k: [..., D]; v: [..., M];
    S: [..., D, M]; Z: [..., D]. Returns (out, S_new, Z_new).
    """
    fq = elu_plus_one(q)
    fk = elu_plus_one(k)
    v = np.asarray(v, dtype=F64)
    S_new = np.asarray(S, dtype=F64) + fk[..., :, None] * v[..., None, :]
    Z_new = np.asarray(Z, dtype=F64) + fk
    num = np.einsum("...d,...dm->...m", fq, S_new)
    den = np.einsum("...d,...d->...", fq, Z_new)
    return num / den[..., None], S_new, Z_new


# ---------------------------------------------------------------------------
# Backward: cumulative-sum gradients
# ---------------------------------------------------------------------------

def backward(q, k, v, dout, causal=True):
    """Gradients (dq, dk, dv) of sum(dout * out) by cumulative sums.

    [summary §3.3.1]: the gradients are computed with cumulative sums, never
    storing every S_i, in linear time and constant memory in N.
    [summary App. A]: the phi(Q) gradient is a forward-direction cumulative sum
    (Q_l only affects output l), the phi(K) and V gradients are cumulative sums
    running in the opposite direction (K_j, V_j affect every output i >= j);
    the denominator is left to autograd there, so its terms are written out
    here by the quotient rule. With G_i = dout_i, den_i = phi(Q_i)^T Z_i and
    out_i = num_i / den_i:

        gN_i  = G_i / den_i                       (gradient w.r.t. num_i)
        gd_i  = -(G_i . out_i) / den_i            (gradient w.r.t. den_i)
        dphiQ_i = S_i gN_i + gd_i Z_i             (forward-direction sums)
        R_j = sum_{i>=j} phi(Q_i) gN_i^T,  r_j = sum_{i>=j} gd_i phi(Q_i)
        dphiK_j = R_j V_j + r_j,  dV_j = R_j^T phi(K_j)   (reverse-direction)

    and the chain rule through phi gives dq = dphiQ * phi'(q), dk = dphiK *
    phi'(k). Non-causal: S, Z are the full sums and R, r the full sums too.
    """
    q = np.asarray(q, dtype=F64)
    k = np.asarray(k, dtype=F64)
    v = np.asarray(v, dtype=F64)
    G = np.asarray(dout, dtype=F64)
    fq = elu_plus_one(q)
    fk = elu_plus_one(k)
    lead = q.shape[:-2]
    n, d = q.shape[-2], q.shape[-1]
    m = v.shape[-1]

    dphiq = np.empty(lead + (n, d), dtype=F64)
    gN = np.empty(lead + (n, m), dtype=F64)
    gd = np.empty(lead + (n,), dtype=F64)

    if causal:
        # forward-direction scan: S_i, Z_i include position i
        S = np.zeros(lead + (d, m), dtype=F64)
        Z = np.zeros(lead + (d,), dtype=F64)
        for i in range(n):
            S = S + fk[..., i, :, None] * v[..., i, None, :]
            Z = Z + fk[..., i, :]
            num = np.einsum("...d,...dm->...m", fq[..., i, :], S)
            den = np.einsum("...d,...d->...", fq[..., i, :], Z)
            out = num / den[..., None]
            gN[..., i, :] = G[..., i, :] / den[..., None]
            gd[..., i] = -np.einsum("...m,...m->...", G[..., i, :], out) / den
            dphiq[..., i, :] = (np.einsum("...dm,...m->...d", S, gN[..., i, :])
                                + gd[..., i, None] * Z)
        # reverse-direction scan: R_j, r_j include position j
        dphik = np.empty(lead + (n, d), dtype=F64)
        dv = np.empty(lead + (n, m), dtype=F64)
        R = np.zeros(lead + (d, m), dtype=F64)
        r = np.zeros(lead + (d,), dtype=F64)
        for j in range(n - 1, -1, -1):
            R = R + fq[..., j, :, None] * gN[..., j, None, :]
            r = r + gd[..., j, None] * fq[..., j, :]
            dphik[..., j, :] = np.einsum("...dm,...m->...d", R, v[..., j, :]) + r
            dv[..., j, :] = np.einsum("...dm,...d->...m", R, fk[..., j, :])
    else:
        S = np.swapaxes(fk, -1, -2) @ v
        Z = fk.sum(axis=-2)
        num = fq @ S
        den = fq @ Z[..., :, None]                           # [..., N, 1]
        out = num / den
        gN[...] = G / den
        gd[...] = -(G * out).sum(axis=-1) / den[..., 0]
        dphiq[...] = gN @ np.swapaxes(S, -1, -2) + gd[..., :, None] * Z[..., None, :]
        R = np.swapaxes(fq, -1, -2) @ gN                     # [..., D, M]
        r = np.einsum("...n,...nd->...d", gd, fq)            # [..., D]
        dphik = v @ np.swapaxes(R, -1, -2) + r[..., None, :]
        dv = fk @ R

    dq = dphiq * elu_plus_one_grad(q)
    dk = dphik * elu_plus_one_grad(k)
    return dq, dk, dv


def denominators(q, k, causal=True):
    """den_i = phi(Q_i)^T Z_i (causal) or phi(Q_i)^T Z (non-causal); [deck slide 4]."""
    fq = elu_plus_one(q)
    fk = elu_plus_one(k)
    Z = np.cumsum(fk, axis=-2) if causal else fk.sum(axis=-2, keepdims=True)
    return (fq * Z).sum(axis=-1)
