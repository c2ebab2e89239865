"""Pins for the CPU float64 oracle (no GPU needed).

The oracle is only trusted because these checks tie it to something other
than itself: hand-derived worked examples (tests/golden/hand_worked.json),
a pure-Python brute force on tiny grids, the library SDPA routine that the
vLLM PR #55629 page (section 关键源码片段, key source excerpt) uses to define
the result, and closed forms / invariants of the method.  The last test plants
plausible mistakes in copies of the oracle and checks that every one of them
is caught by at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")
RNG = np.random.default_rng(1234)


# --------------------------------------------------------------------------- helpers
def _rand_case(BH, H, W, d, sig_t=0.5, seed=0):
    r = np.random.default_rng(seed)
    N = H * W
    return dict(q=r.standard_normal((BH, N, d)), k=r.standard_normal((BH, N, d)),
                v=r.standard_normal((BH, N, d)), th=sig_t * r.standard_normal((2 * H - 1, d)),
                tw=sig_t * r.standard_normal((2 * W - 1, d)))


def brute_force(q, k, v, th, tw, H, W, scale):
    """Per-element pure-Python evaluation of the definition (tiny inputs only)."""
    BH, N, d = len(q), len(q[0]), len(q[0][0])
    out = [[[0.0] * len(v[0][0]) for _ in range(N)] for _ in range(BH)]
    for b in range(BH):
        for n in range(N):
            qh, qw = divmod(n, W)
            logits = []
            for m in range(N):
                kh, kw = divmod(m, W)
                s = 0.0
                for c in range(d):
                    s += q[b][n][c] * k[b][m][c]
                bias = 0.0
                for c in range(d):
                    bias += q[b][n][c] * th[qh - kh + H - 1][c]
                    bias += q[b][n][c] * tw[qw - kw + W - 1][c]
                logits.append(scale * s + bias)
            top = max(logits)
            e = [math.exp(x - top) for x in logits]
            z = sum(e)
            for m in range(N):
                for c in range(len(v[0][0])):
                    out[b][n][c] += e[m] / z * v[b][m][c]
    return np.array(out)


# --------------------------------------------------------------------------- pins
# Each pin takes (project_fn, attention_fn) with the oracle's signatures and
# raises AssertionError when the implementation disagrees with what it pins.

def pin_golden(project_fn, attention_fn):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        H, W, s = c["H"], c["W"], c["scale"]
        rh, rw = project_fn(c["q"], c["rel_pos_h"], c["rel_pos_w"], H, W)
        np.testing.assert_allclose(rh, c["rel_h"], atol=1e-12, err_msg=c["name"] + " rel_h")
        np.testing.assert_allclose(rw, c["rel_w"], atol=1e-12, err_msg=c["name"] + " rel_w")
        out = attention_fn(c["q"], c["k"], c["v"], rh, rw, H, W, s)
        np.testing.assert_allclose(out, c["out"], rtol=1e-12, atol=1e-12, err_msg=c["name"] + " out")


def pin_brute_force(project_fn, attention_fn):
    for (H, W, d) in [(1, 1, 1), (1, 4, 4), (3, 1, 4), (2, 3, 1), (2, 3, 4), (4, 4, 4), (3, 5, 2)]:
        c = _rand_case(2, H, W, d, seed=H * 100 + W * 10 + d)
        scale = 0.37
        rh, rw = project_fn(c["q"], c["th"], c["tw"], H, W)
        got = attention_fn(c["q"], c["k"], c["v"], rh, rw, H, W, scale)
        want = brute_force(c["q"].tolist(), c["k"].tolist(), c["v"].tolist(), c["th"].tolist(),
                           c["tw"].tolist(), H, W, scale)
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12, err_msg=f"{H}x{W} d={d}")


def pin_library_sdpa(project_fn, attention_fn):
    """The page defines the result as SDPA with the additive bias (rel_h + rel_w).view(...)."""
    for (H, W, d) in [(3, 5, 8), (4, 4, 16), (5, 2, 8)]:
        c = _rand_case(3, H, W, d, sig_t=1.0, seed=7 + H + W)
        N = H * W
        rh, rw = project_fn(c["q"], c["th"], c["tw"], H, W)
        rh_t = torch.from_numpy(np.asarray(rh)).reshape(3, N, H, 1)
        rw_t = torch.from_numpy(np.asarray(rw)).reshape(3, N, 1, W)
        bias = (rh_t + rw_t).view(3, N, H * W)
        q, k, v = (torch.from_numpy(c[x]) for x in ("q", "k", "v"))
        want = F.scaled_dot_product_attention(q, k, v, attn_mask=bias, scale=d ** -0.5).numpy()
        got = attention_fn(c["q"], c["k"], c["v"], rh, rw, H, W, d ** -0.5)
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def pin_one_hot_tables(project_fn, attention_fn):
    """With rel_pos_h[r] = e_c: rel_h[n, kh] = q_n[c] iff qh - kh + H - 1 == r (same for w)."""
    H, W, d = 3, 4, 5
    q = RNG.standard_normal((2, H * W, d))
    for r in range(2 * H - 1):
        for c in (0, 3):
            th = np.zeros((2 * H - 1, d)); th[r, c] = 1.0
            tw = np.zeros((2 * W - 1, d))
            rh, rw = project_fn(q, th, tw, H, W)
            want = np.zeros((2, H * W, H))
            for n in range(H * W):
                for kh in range(H):
                    if n // W - kh + H - 1 == r:
                        want[:, n, kh] = q[:, n, c]
            np.testing.assert_allclose(rh, want, atol=1e-15)
            np.testing.assert_allclose(rw, 0.0, atol=1e-15)
    for r in range(2 * W - 1):
        tw = np.zeros((2 * W - 1, d)); tw[r, 2] = 1.0
        rh, rw = project_fn(q, np.zeros((2 * H - 1, d)), tw, H, W)
        want = np.zeros((2, H * W, W))
        for n in range(H * W):
            for kw in range(W):
                if n % W - kw + W - 1 == r:
                    want[:, n, kw] = q[:, n, 2]
        np.testing.assert_allclose(rw, want, atol=1e-15)


def pin_shift_identity(project_fn, attention_fn):
    """All q rows equal: Bias[(qh,qw),(kh,kw)] depends only on (qh - kh, qw - kw) (block Toeplitz)."""
    H, W, d = 4, 3, 6
    q = np.tile(RNG.standard_normal((1, 1, d)), (1, H * W, 1))
    th, tw = RNG.standard_normal((2 * H - 1, d)), RNG.standard_normal((2 * W - 1, d))
    rh, rw = project_fn(q, th, tw, H, W)
    rh, rw = np.asarray(rh)[0], np.asarray(rw)[0]
    seen = {}
    for n in range(H * W):
        for m in range(H * W):
            key = (n // W - m // W, n % W - m % W)
            val = rh[n, m // W] + rw[n, m % W]
            if key in seen:
                assert abs(seen[key] - val) < 1e-12, key
            else:
                seen[key] = val
    assert len(seen) == (2 * H - 1) * (2 * W - 1)
    # distinct offsets read distinct table rows, so the values differ
    vals = np.array(sorted(seen.values()))
    assert np.min(np.diff(vals)) > 1e-9


def pin_rows_sum_to_one(project_fn, attention_fn):
    H, W, d = 3, 4, 8
    c = _rand_case(2, H, W, d, sig_t=2.0, seed=5)
    rh, rw = project_fn(c["q"], c["th"], c["tw"], H, W)
    out = attention_fn(c["q"], c["k"], np.ones_like(c["v"]), rh, rw, H, W, 0.5)
    np.testing.assert_allclose(out, 1.0, atol=1e-13)


def pin_zero_tables(project_fn, attention_fn):
    """Zero tables reduce the method to textbook attention (the page's use_rel_pos=False branch)."""
    H, W, d = 4, 5, 8
    c = _rand_case(2, H, W, d, seed=9)
    z_h, z_w = np.zeros((2 * H - 1, d)), np.zeros((2 * W - 1, d))
    rh, rw = project_fn(c["q"], z_h, z_w, H, W)
    got = attention_fn(c["q"], c["k"], c["v"], rh, rw, H, W, d ** -0.5)
    q, k, v = (torch.from_numpy(c[x]) for x in ("q", "k", "v"))
    want = F.scaled_dot_product_attention(q, k, v).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def pin_zero_query(project_fn, attention_fn):
    """q = 0: every logit is 0, so each output row is the mean of v."""
    H, W, d = 3, 3, 4
    c = _rand_case(2, H, W, d, seed=11)
    q = np.zeros_like(c["q"])
    rh, rw = project_fn(q, c["th"], c["tw"], H, W)
    out = attention_fn(q, c["k"], c["v"], rh, rw, H, W, 0.125)
    np.testing.assert_allclose(out, np.broadcast_to(c["v"].mean(axis=1, keepdims=True), out.shape), atol=1e-14)


def pin_separable_closed_form(project_fn, attention_fn):
    """k = 0: p[n, (kh, kw)] = softmax(rel_h[n])[kh] * softmax(rel_w[n])[kw]."""
    H, W, d = 3, 5, 4
    c = _rand_case(1, H, W, d, sig_t=1.0, seed=13)
    k = np.zeros_like(c["k"])
    rh, rw = project_fn(c["q"], c["th"], c["tw"], H, W)
    rh, rw = np.asarray(rh), np.asarray(rw)
    out = attention_fn(c["q"], k, c["v"], rh, rw, H, W, 0.125)
    ph = np.exp(rh[0] - rh[0].max(1, keepdims=True)); ph /= ph.sum(1, keepdims=True)
    pw = np.exp(rw[0] - rw[0].max(1, keepdims=True)); pw /= pw.sum(1, keepdims=True)
    v = c["v"][0].reshape(H, W, d)
    want = np.einsum("nh,nw,hwc->nc", ph, pw, v)
    np.testing.assert_allclose(out[0], want, rtol=1e-11, atol=1e-12)
    # the projection itself on this case, by direct dot products
    q = c["q"][0]
    for n in range(H * W):
        qh, qw = divmod(n, W)
        for kh in range(H):
            assert abs(rh[0, n, kh] - q[n] @ c["th"][qh - kh + H - 1]) < 1e-12
        for kw in range(W):
            assert abs(rw[0, n, kw] - q[n] @ c["tw"][qw - kw + W - 1]) < 1e-12


PINS = [pin_golden, pin_brute_force, pin_library_sdpa, pin_one_hot_tables, pin_shift_identity,
        pin_rows_sum_to_one, pin_zero_tables, pin_zero_query, pin_separable_closed_form]


# --------------------------------------------------------------------------- tests
@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.project, oracle.attention)


def test_fused_is_project_then_attention():
    H, W, d = 3, 4, 8
    c = _rand_case(2, H, W, d, seed=21)
    rh, rw = oracle.project(c["q"], c["th"], c["tw"], H, W)
    a = oracle.attention(c["q"], c["k"], c["v"], rh, rw, H, W, 0.2)
    b = oracle.fused(c["q"], c["k"], c["v"], c["th"], c["tw"], H, W, 0.2)
    np.testing.assert_array_equal(a, b)


def test_row_variants_match_full():
    H, W, d = 5, 7, 8
    c = _rand_case(3, H, W, d, sig_t=1.0, seed=3)
    full = oracle.fused(c["q"], c["k"], c["v"], c["th"], c["tw"], H, W, 0.125)
    rh, rw = oracle.project(c["q"], c["th"], c["tw"], H, W)
    rows = np.array([0, 6, 7, 20, 34])
    for b in range(3):
        prh, prw = oracle.project_rows(c["q"][b][rows], rows, c["th"], c["tw"], H, W)
        np.testing.assert_allclose(prh, rh[b][rows], atol=1e-13)
        np.testing.assert_allclose(prw, rw[b][rows], atol=1e-13)
        got = oracle.fused_rows(c["q"], c["k"], c["v"], c["th"], c["tw"], b, rows, H, W, 0.125)
        np.testing.assert_allclose(got, full[b][rows], rtol=1e-12, atol=1e-13)
        got2 = oracle.attention_rows(c["q"], c["k"], c["v"], rh[b][rows], rw[b][rows], b, rows, H, W, 0.125)
        np.testing.assert_allclose(got2, full[b][rows], rtol=1e-12, atol=1e-13)


def test_bad_shapes_rejected():
    with pytest.raises(ValueError):
        oracle.project(np.zeros((1, 6, 4)), np.zeros((3, 4)), np.zeros((5, 4)), 2, 4)
    with pytest.raises(ValueError):
        oracle.project(np.zeros((1, 6, 4)), np.zeros((4, 4)), np.zeros((5, 4)), 2, 3)


# --------------------------------------------------------------------------- planted mistakes
def _mutant_project(kind):
    def proj(q, th, tw, H, W):
        q, th, tw = np.asarray(q, float), np.asarray(th, float), np.asarray(tw, float)
        BH, N, d = q.shape
        rh, rw = np.zeros((BH, N, H)), np.zeros((BH, N, W))
        for n in range(N):
            qh, qw = divmod(n, W)
            for kh in range(H):
                r = (kh - qh + H - 1) if kind == "sign_h" else (qh - kh + H - 1)
                rh[:, n, kh] = q[:, n] @ th[r]
            for kw in range(W):
                r = (kw - qw + W - 1) if kind == "sign_w" else (qw - kw + W - 1)
                rw[:, n, kw] = q[:, n] @ tw[r]
        if kind == "drop_w":
            rw[:] = 0.0
        if kind == "swap_tables" and H == W:
            rh, rw = rw, rh
        return rh, rw
    return proj


def _mutant_attention(kind):
    def attn(q, k, v, rh, rw, H, W, scale):
        q, k, v, rh, rw = (np.asarray(x, float) for x in (q, k, v, rh, rw))
        BH, N, _ = q.shape
        out = np.empty((BH, N, v.shape[2]))
        for b in range(BH):
            if kind == "key_transposed":
                bias = (rh[b][:, None, :] + rw[b][:, :, None]).reshape(N, N)
            else:
                bias = (rh[b][:, :, None] + rw[b][:, None, :]).reshape(N, N)
            s = q[b] @ k[b].T
            if kind == "bias_scaled":
                logits = scale * (s + bias)
            elif kind == "unscaled_qk":
                logits = s + bias
            else:
                logits = scale * s + bias
            logits -= logits.max(1, keepdims=True)
            p = np.exp(logits)
            if kind == "no_normalise":
                out[b] = p @ v[b]
            else:
                out[b] = (p / p.sum(1, keepdims=True)) @ v[b]
        return out
    return attn


MUTANTS = {
    "sign_h": (_mutant_project("sign_h"), oracle.attention),
    "sign_w": (_mutant_project("sign_w"), oracle.attention),
    "drop_w": (_mutant_project("drop_w"), oracle.attention),
    "key_transposed": (oracle.project, _mutant_attention("key_transposed")),
    "bias_scaled": (oracle.project, _mutant_attention("bias_scaled")),
    "unscaled_qk": (oracle.project, _mutant_attention("unscaled_qk")),
    "no_normalise": (oracle.project, _mutant_attention("no_normalise")),
}


def test_reference_mutant_is_equivalent():
    """The loop-based mutant scaffolding with no mistake planted agrees with the oracle."""
    for pin in PINS:
        pin(_mutant_project("none"), _mutant_attention("none"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    proj, attn = MUTANTS[name]
    caught = []
    for pin in PINS:
        try:
            pin(proj, attn)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
