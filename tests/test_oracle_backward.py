"""Pins for the oracle's backward and log-sum-exp (no GPU needed).

The pages print no backward; the oracle's is the gradient of the forward's
definition (section 关键源码片段 of the vLLM PR #55629 page: SDPA with the
additive decomposed bias), taken by the chain rule.  It is tied to something
other than itself here:
  * central finite differences of ``L = sum(dout * fused(...))`` with respect to
    every element of every input, on tiny problems;
  * invariants: each row of the bias gradient sums to zero over the keys (the
    softmax is shift-invariant), so every row of ``drel_h`` and of ``drel_w``
    sums to zero;
  * a closed form: with every row of v equal, the output does not depend on
    q, k or the bias, so their gradients vanish and ``dv = P^T dout``;
  * ``lse2`` against scipy's log-sum-exp and the closed form log2(N) for zero
    logits.
Planted mistakes in copies of the backward must each fail the finite
differences.
"""
from __future__ import annotations

import numpy as np
import pytest
import scipy.special

import oracle


def _case(BH=2, H=2, W=3, d=4, seed=5, sig=0.7):
    r = np.random.default_rng(seed)
    N = H * W
    return dict(q=sig * r.standard_normal((BH, N, d)), k=sig * r.standard_normal((BH, N, d)),
                v=r.standard_normal((BH, N, d)), th=sig * r.standard_normal((2 * H - 1, d)),
                tw=sig * r.standard_normal((2 * W - 1, d)), dout=r.standard_normal((BH, N, d)))


def _fd_grads(c, H, W, scale, h=1e-6):
    """Central finite differences of sum(dout * fused(...)) for every input element."""
    names = ["q", "k", "v", "th", "tw"]

    def loss(x):
        return float((c["dout"] * oracle.fused(x["q"], x["k"], x["v"], x["th"], x["tw"], H, W, scale)).sum())

    out = {}
    for nm in names:
        g = np.zeros_like(c[nm])
        it = np.nditer(c[nm], flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            xp = {n: c[n].copy() for n in names}
            xm = {n: c[n].copy() for n in names}
            xp[nm][i] += h
            xm[nm][i] -= h
            g[i] = (loss(xp) - loss(xm)) / (2 * h)
        out[nm] = g
    return out


def _check_grads(grads, fd, what=""):
    for nm, g in zip(["q", "k", "v", "th", "tw"], grads):
        ref = fd[nm]
        err = np.abs(g - ref).max()
        assert err <= 1e-6 * max(1.0, np.abs(ref).max()), f"{what} d{nm}: max error {err:.3e}"


@pytest.mark.parametrize("shape", [(2, 2, 3, 4), (1, 3, 2, 5)])
def test_fused_backward_matches_finite_differences(shape):
    BH, H, W, d = shape
    c = _case(BH, H, W, d)
    scale = d ** -0.5
    grads = oracle.fused_backward(c["q"], c["k"], c["v"], c["th"], c["tw"], H, W, scale, c["dout"])
    _check_grads(grads, _fd_grads(c, H, W, scale), f"shape {shape}")


def test_attention_backward_matches_finite_differences():
    """The compact-bias entry: gradients with respect to q, k, v, rel_h and rel_w."""
    BH, H, W, d = 2, 2, 3, 4
    c = _case(BH, H, W, d, seed=9)
    r = np.random.default_rng(3)
    rh, rw = r.standard_normal((BH, H * W, H)), r.standard_normal((BH, H * W, W))
    scale = 0.3
    x = dict(q=c["q"], k=c["k"], v=c["v"], rh=rh, rw=rw)

    def loss(y):
        return float((c["dout"] * oracle.attention(y["q"], y["k"], y["v"], y["rh"], y["rw"], H, W, scale)).sum())

    got = oracle.attention_backward(c["q"], c["k"], c["v"], rh, rw, H, W, scale, c["dout"])
    for nm, g in zip(["q", "k", "v", "rh", "rw"], got):
        fd = np.zeros_like(x[nm])
        it = np.nditer(x[nm], flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            xp = {n: t.copy() for n, t in x.items()}
            xm = {n: t.copy() for n, t in x.items()}
            xp[nm][i] += 1e-6
            xm[nm][i] -= 1e-6
            fd[i] = (loss(xp) - loss(xm)) / 2e-6
        assert np.abs(g - fd).max() <= 1e-6 * max(1.0, np.abs(fd).max()), nm


def test_bias_gradient_rows_sum_to_zero():
    c = _case(3, 4, 5, 8, seed=11, sig=1.5)
    rh, rw = oracle.project(c["q"], c["th"], c["tw"], 4, 5)
    _, _, _, drh, drw = oracle.attention_backward(c["q"], c["k"], c["v"], rh, rw, 4, 5, 0.35, c["dout"])
    assert np.abs(drh.sum(axis=-1)).max() < 1e-12
    assert np.abs(drw.sum(axis=-1)).max() < 1e-12
    # and the two marginals of the same dZ carry the same total per row
    assert np.abs(drh.sum(axis=-1) - drw.sum(axis=-1)).max() < 1e-12


def test_constant_v_closed_form():
    """Every row of v the same vector: out = that vector whatever the weights, so dq, dk and the
    table gradients vanish and dv = P^T dout with P the softmax of the logits."""
    H, W, d = 3, 3, 4
    c = _case(2, H, W, d, seed=2)
    c["v"][:] = c["v"][:, :1, :]
    scale = 0.5
    dq, dk, dv, dth, dtw = oracle.fused_backward(c["q"], c["k"], c["v"], c["th"], c["tw"], H, W, scale, c["dout"])
    for g in (dq, dk, dth, dtw):
        assert np.abs(g).max() < 1e-12
    rh, rw = oracle.project(c["q"], c["th"], c["tw"], H, W)
    for b in range(2):
        z = scale * c["q"][b] @ c["k"][b].T + oracle.dense_bias(rh[b], rw[b], H, W)
        p = np.exp(z - z.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        assert np.allclose(dv[b], p.T @ c["dout"][b], atol=1e-12)


def test_lse2():
    c = _case(2, 3, 4, 6, seed=4, sig=2.0)
    rh, rw = oracle.project(c["q"], c["th"], c["tw"], 3, 4)
    got = oracle.lse2(c["q"], c["k"], rh, rw, 3, 4, 0.4)
    for b in range(2):
        z = 0.4 * c["q"][b] @ c["k"][b].T + oracle.dense_bias(rh[b], rw[b], 3, 4)
        assert np.allclose(got[b], scipy.special.logsumexp(z, axis=1) / np.log(2.0), atol=1e-12)
    zero = oracle.lse2(np.zeros((1, 12, 4)), np.zeros((1, 12, 4)), np.zeros((1, 12, 3)), np.zeros((1, 12, 4)), 3, 4, 1.0)
    assert np.allclose(zero, np.log2(12.0), atol=1e-14)


# --------------------------------------------------------------------------- planted mistakes
def _mutant_backward(kind):
    def bwd(q, k, v, th, tw, H, W, scale, dout):
        q, k, v, th, tw, dout = (np.asarray(x, float) for x in (q, k, v, th, tw, dout))
        BH, N, d = q.shape
        rh, rw = oracle.project(q, th, tw, H, W)
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        dth, dtw = np.zeros_like(th), np.zeros_like(tw)
        for b in range(BH):
            z = scale * (q[b] @ k[b].T) + oracle.dense_bias(rh[b], rw[b], H, W)
            p = np.exp(z - z.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            o = p @ v[b]
            dv[b] = (p @ dout[b]) if kind == "dv_untransposed" else (p.T @ dout[b])
            dp = dout[b] @ v[b].T
            dd = (dout[b] * o).sum(1)
            dz = p * dp if kind == "no_rowsum" else p * (dp - dd[:, None])
            dq[b] = (dz @ k[b]) if kind == "dq_unscaled" else scale * (dz @ k[b])
            dk[b] = scale * ((dz @ q[b]) if kind == "dk_untransposed" else (dz.T @ q[b]))
            for n in range(N):
                qh, qw = divmod(n, W)
                for m in range(N):
                    kh, kw = divmod(m, W)
                    ih = (kh - qh + H - 1) if kind == "table_index_sign" else (qh - kh + H - 1)
                    iw = qw - kw + W - 1
                    dq[b, n] += dz[n, m] * (th[ih] + tw[iw])
                    dth[ih] += dz[n, m] * q[b, n]
                    if kind != "drop_dtw":
                        dtw[iw] += dz[n, m] * q[b, n]
        return dq, dk, dv, dth, dtw
    return bwd


BW_MUTANTS = ["dv_untransposed", "no_rowsum", "dq_unscaled", "dk_untransposed", "table_index_sign", "drop_dtw"]


def test_backward_mutant_scaffolding_agrees():
    c = _case(2, 2, 3, 4, seed=8)
    a = _mutant_backward("none")(c["q"], c["k"], c["v"], c["th"], c["tw"], 2, 3, 0.5, c["dout"])
    b = oracle.fused_backward(c["q"], c["k"], c["v"], c["th"], c["tw"], 2, 3, 0.5, c["dout"])
    for x, y in zip(a, b):
        assert np.allclose(x, y, atol=1e-12)


@pytest.mark.parametrize("kind", BW_MUTANTS)
def test_backward_planted_mistake_is_caught(kind):
    c = _case(2, 2, 3, 4, seed=8)
    fd = _fd_grads(c, 2, 3, 0.5)
    grads = _mutant_backward(kind)(c["q"], c["k"], c["v"], c["th"], c["tw"], 2, 3, 0.5, c["dout"])
    with pytest.raises(AssertionError):
        _check_grads(grads, fd, kind)
