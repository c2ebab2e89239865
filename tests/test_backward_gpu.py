"""The backward (dera_relpos_fused_backward) and the training forward (dera_relpos_fused_lse)
against the CPU float64 oracle's chain-rule gradient.

Tolerance (derived, then confirmed by the margins printed at the end of the run): P and dZ enter
the tensor-core products rounded to the input dtype (relative 2^-9 for bf16, 2^-11 for fp16) with
fp32 accumulation, so each gradient carries a relative rounding error of that order, amplified where
a sum cancels.  The checks are rel-L2 <= 1e-2 (bf16) / 4e-3 (fp16) and a max-abs error of at most
3e-2 (bf16) / 1e-2 (fp16) of the largest reference value, per gradient.  The table gradients sum
over every row of every head, in fp32.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import relative_position_bias_gb300 as rpb
from conftest import record_margin
from relative_position_bias_gb300 import build as rbuild
from relative_position_bias_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: (1e-2, 3e-2), torch.float16: (4e-3, 1e-2)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    rbuild.build()
    rpb.load_library()
    yield
    assert rpb.device_status() == 0, "a kernel hit its bounded-wait budget"


def make_case(BH, H, W, dtype, sq=1.0, sk=1.0, sv=1.0, st=0.5, seed=0):
    g = torch.Generator().manual_seed(seed)
    N = H * W
    x = {"q": sq * torch.randn(BH, N, 64, generator=g), "k": sk * torch.randn(BH, N, 64, generator=g),
         "v": sv * torch.randn(BH, N, 64, generator=g), "rel_pos_h": st * torch.randn(2 * H - 1, 64, generator=g),
         "rel_pos_w": st * torch.randn(2 * W - 1, 64, generator=g), "dout": torch.randn(BH, N, 64, generator=g)}
    return {n: t.to(dtype) for n, t in x.items()}


CASES = {
    # name: (BH, H, W, dtype, sigma_q, sigma_k)
    "grid16-bf16": (2, 16, 16, torch.bfloat16, 1.0, 1.0),
    "global64-bf16": (2, 64, 64, torch.bfloat16, 0.5, 0.5),
    "ragged40-f16": (3, 40, 40, torch.float16, 2.0, 2.0),
    "window14-bf16": (6, 14, 14, torch.bfloat16, 1.0, 1.0),
    "odd7x30-f16": (2, 7, 30, torch.float16, 1.0, 1.0),
    "tall33x9-bf16": (2, 33, 9, torch.bfloat16, 1.0, 1.0),
    "tiny3x5-f16": (3, 3, 5, torch.float16, 1.0, 1.0),       # one partial query tile, one key tile
    "single1x1-bf16": (2, 1, 1, torch.bfloat16, 1.0, 1.0),   # one token: dq = dk = 0, dv = dout
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_matches_oracle(name):
    BH, H, W, dtype, sq, sk = CASES[name]
    x = make_case(BH, H, W, dtype, sq=sq, sk=sk, seed=sorted(CASES).index(name))
    d = {n: t.cuda() for n, t in x.items()}
    scale = 0.125
    out, lse = rpb.fused_lse(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], H, W, scale,
                             out_dtype=torch.float32)
    grads = rpb.fused_backward(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], out, lse, d["dout"], H, W,
                               scale)
    torch.cuda.synchronize()
    f = {n: I.to_f64(t) for n, t in x.items()}
    want = oracle.fused_backward(f["q"], f["k"], f["v"], f["rel_pos_h"], f["rel_pos_w"], H, W, scale, f["dout"])
    rl2_tol, max_tol = TOL[dtype]
    for gname, got, ref in zip(["dq", "dk", "dv", "drel_pos_h", "drel_pos_w"], grads, want):
        g = got.double().cpu().numpy()
        assert np.isfinite(g).all(), gname
        err = np.abs(g - ref).max()
        # a gradient that vanishes (one token: dq = dk = 0) is measured against the O(1) scale
        # of the inputs instead of its own zero norm
        scale_ref = max(np.abs(ref).max(), 1e-2)
        rl2 = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-2 * math.sqrt(ref.size))
        record_margin(f"backward {name} {gname} (max-abs / max|ref|)", err / scale_ref, rl2,
                      f"{max_tol:g} / {rl2_tol:g}")
        assert rl2 <= rl2_tol, f"{gname}: rel-L2 {rl2:.3e}"
        assert err <= max_tol * scale_ref, f"{gname}: max-abs {err:.3e} of max {scale_ref:.3e}"


@pytest.mark.parametrize("name", ["grid16-bf16", "ragged40-f16", "window14-bf16"])
def test_forward_lse(name):
    """The training forward's out is the plain forward's, bit for bit, and lse is the oracle's."""
    BH, H, W, dtype, sq, sk = CASES[name]
    x = make_case(BH, H, W, dtype, sq=sq, sk=sk, seed=3)
    d = {n: t.cuda() for n, t in x.items()}
    scale = 0.125
    out, lse = rpb.fused_lse(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], H, W, scale,
                             out_dtype=torch.float32)
    plain = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], H, W, scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(out, plain)
    f = {n: I.to_f64(t) for n, t in x.items()}
    rh, rw = oracle.project(f["q"], f["rel_pos_h"], f["rel_pos_w"], H, W)
    want = oracle.lse2(f["q"], f["k"], rh, rw, H, W, scale)
    err = np.abs(lse.double().cpu().numpy() - want).max()
    record_margin(f"forward lse {name}", err, 0.0, "1e-3 (base 2)")
    assert err <= 1e-3, f"lse max-abs {err:.3e}"


def test_backward_is_deterministic():
    """No atomics: two calls give bit-identical gradients."""
    BH, H, W, dtype, sq, sk = CASES["global64-bf16"]
    x = make_case(BH, H, W, dtype, sq=sq, sk=sk, seed=5)
    d = {n: t.cuda() for n, t in x.items()}
    out, lse = rpb.fused_lse(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], H, W, 0.125)
    a = rpb.fused_backward(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], out, lse, d["dout"], H, W, 0.125,
                           grad_dtype=torch.bfloat16)
    b = rpb.fused_backward(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], out, lse, d["dout"], H, W, 0.125,
                           grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    for x1, x2 in zip(a, b):
        assert torch.equal(x1, x2)
    # a bf16 gradient is the fp32 one rounded
    c = rpb.fused_backward(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], out, lse, d["dout"], H, W, 0.125)
    torch.cuda.synchronize()
    for x16, x32 in zip(a[:3], c[:3]):
        assert torch.equal(x16, x32.to(torch.bfloat16))


def test_backward_on_another_stream():
    """A call on a stream other than the current one (its scratch is recorded on that stream)
    gives the same gradients, bit for bit."""
    BH, H, W, dtype, sq, sk = CASES["grid16-bf16"]
    x = make_case(BH, H, W, dtype, sq=sq, sk=sk, seed=7)
    d = {n: t.cuda() for n, t in x.items()}
    out, lse = rpb.fused_lse(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], H, W, 0.125)
    args = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], out, lse, d["dout"], H, W, 0.125)
    a = rpb.fused_backward(*args)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    b = rpb.fused_backward(*args, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for x1, x2 in zip(a, b):
        assert torch.equal(x1, x2)


def test_backward_empty_batch():
    """BH = 0: nothing to compute; the table gradients are zero."""
    H, W = 4, 4
    e = torch.empty(0, H * W, 64, dtype=torch.bfloat16, device="cuda")
    th = torch.randn(2 * H - 1, 64).to(torch.bfloat16).cuda()
    tw = torch.randn(2 * W - 1, 64).to(torch.bfloat16).cuda()
    lse = torch.empty(0, H * W, dtype=torch.float32, device="cuda")
    dq, dk, dv, dth, dtw = rpb.fused_backward(e, e, e, th, tw, e.float(), lse, e, H, W, 0.125)
    torch.cuda.synchronize()
    assert dq.shape == (0, H * W, 64) and dk.shape == dq.shape and dv.shape == dq.shape
    assert torch.count_nonzero(dth) == 0 and torch.count_nonzero(dtw) == 0


def _bench_case(name):
    """A workload exactly as `bench.py --entry backward` times it: the seeded inputs, dout from
    seed 1000, the training forward's out and lse in the input dtype, gradients in the input
    dtype."""
    w = I.WORKLOADS[name]
    x = I.make_inputs(w, seed=0)
    d = {n: t.cuda() for n, t in x.items()}
    g = torch.Generator().manual_seed(1000)
    dout = torch.randn(w.BH, w.N, w.d, generator=g).to(w.torch_dtype)
    out, lse = rpb.fused_lse(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
    grads = rpb.fused_backward(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], out, lse, dout.cuda(), w.H,
                               w.W, w.scale, grad_dtype=w.torch_dtype)
    torch.cuda.synchronize()
    return w, x, d, dout, out, lse, grads


def _check(label, got, ref, dtype):
    rl2_tol, max_tol = TOL[dtype]
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    assert np.isfinite(g).all(), label
    err = np.abs(g - ref).max()
    scale_ref = max(np.abs(ref).max(), 1e-2)
    rl2 = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-2 * math.sqrt(ref.size))
    record_margin(f"backward {label} (max-abs / max|ref|)", err / scale_ref, rl2, f"{max_tol:g} / {rl2_tol:g}")
    assert rl2 <= rl2_tol, f"{label}: rel-L2 {rl2:.3e}"
    assert err <= max_tol * scale_ref, f"{label}: max-abs {err:.3e} of max {scale_ref:.3e}"


@pytest.mark.parametrize("name", ["global64", "batched64", "wide64", "ragged40", "window14"])
def test_backward_full_size(name):
    """The bench's call on each workload at its full size (input-dtype out and gradients), every
    gradient element against the oracle, which takes the heads one at a time."""
    w, x, _, dout, _, _, grads = _bench_case(name)
    f = {n: I.to_f64(t) for n, t in x.items()}
    want = oracle.fused_backward(f["q"], f["k"], f["v"], f["rel_pos_h"], f["rel_pos_w"], w.H, w.W, w.scale,
                                 I.to_f64(dout))
    for gname, got, ref in zip(["dq", "dk", "dv", "drel_pos_h", "drel_pos_w"], grads, want):
        _check(f"{name} full {gname}", got, ref, w.torch_dtype)
