"""Softmax range handling of the attention kernel, against the CPU float64 oracle.

The kernel exponentiates each key tile against a running row maximum and stores P in fp16 for the
P.V product (section 风险与影响 of the vLLM PR #55629 page fixes exp2 and fp32 accumulation; the
fp16 P is this library's reading).  fp16 has a narrow exponent range: a p below 2^-24 flushes to
zero and one below 2^-14 keeps only part of its mantissa.  So the kernel must never let the
maximum it uses sit far above the row's true maximum while most of the row's mass lies in keys
well below it: that mass would be lost from P.V but still counted in the fp32 row sum.  The page
lists stability under extreme inputs as the path's first risk.

`test_start_maximum_overshoot` builds exactly that row: the true maximum is one key of the first
key tile, the row's largest rel_h term sits on grid rows whose keys score very low, and thousands
of keys sit about 13 (base 2) below the maximum.  A starting maximum estimated from "best score +
largest rel_h" overshoots the true maximum by 12 there.

`test_rows_sum_to_one` uses V = 1, for which every output is exactly 1 at any size, and checks it
on every row of every workload, for both entries.

`test_rel_h_patterns` moves the row maximum by large steps between key tiles through the rel_h
term alone (rising, falling, and jumping on every other tile), which drives the kernel's
decisions per tile: take a tile exact at once, exponentiate it speculatively, or start a warp at
the safe cap."""
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

ABS_TOL = 4e-3
RL2_TOL = 1e-2
LOG2E = 1.0 / math.log(2.0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    rbuild.build()
    rpb.load_library()
    yield
    assert rpb.device_status() == 0, "a kernel hit its bounded-wait budget"


def overshoot_case(H: int, W: int, heads: int, dtype: torch.dtype, seed: int = 7):
    """q, k, v, tables and the compact bias of the overshoot row pattern, the same for every head
    (the heads only spread the work over the device so that the schedule cuts units).

    q = a*e0 for every token, so scale*q.k = a*scale*b_m with k_m = b_m*e0.  In base-2 units:
      key (kh=0, kw=5): 0                      (the row's true maximum)
      other keys of grid rows 0, 1: about -40
      grid rows 2 .. H-3: about -13.1          (the bulk: thousands of keys)
      grid rows H-2, H-1: about -40 + 16        (low scores on the largest rel_h term)
    rel_h is 16 (base 2) on grid rows H-2, H-1 and 0 elsewhere; rel_w is 0.  The fused entry
    gets that rel_h from rel_pos_h rows 0 and 1 (for query grid rows 0 and 1 only), the compact
    entry gets it directly for every row."""
    a = 2.0
    scale = 0.125
    sl2 = a * scale * LOG2E
    N = H * W
    b = np.full((H, W), -40.0 / sl2)
    b[2:H - 2, :] = -13.1 / sl2
    b[0, 5] = 0.0
    q = torch.zeros(heads, N, 64)
    q[..., 0] = a
    k = torch.zeros(heads, N, 64)
    k[..., 0] = torch.from_numpy(b.reshape(-1)).float()
    g = torch.Generator().manual_seed(seed)
    v = (1.0 + 0.5 * torch.randn(N, 64, generator=g)).expand(heads, N, 64).contiguous()  # mean 1
    hb = 16.0 / LOG2E
    th = torch.zeros(2 * H - 1, 64)
    th[0:2, 0] = hb / a
    tw = torch.zeros(2 * W - 1, 64)
    x = {"q": q, "k": k, "v": v, "rel_pos_h": th, "rel_pos_w": tw}
    x = {n: t.to(dtype) for n, t in x.items()}
    rel_h = torch.zeros(heads, N, H)
    rel_h[:, :, H - 2:] = hb
    rel_w = torch.zeros(heads, N, W)
    return x, rel_h, rel_w, scale


@pytest.mark.parametrize("workspace", [None, False], ids=["workspace", "no-workspace"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("grid", [(64, 64, 12), (40, 40, 24)], ids=["64x64", "40x40"])
@pytest.mark.parametrize("entry", ["fused", "attention"])
def test_start_maximum_overshoot(entry, grid, dtype, workspace):
    H, W, heads = grid
    x, rel_h, rel_w, scale = overshoot_case(H, W, heads, dtype)
    d = {n: t.cuda() for n, t in x.items()}
    f = {n: I.to_f64(t) for n, t in x.items()}
    if entry == "fused":
        out = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], H, W, scale,
                        out_dtype=torch.float32, workspace=workspace)
        want = oracle.fused(f["q"][:1], f["k"][:1], f["v"][:1], f["rel_pos_h"], f["rel_pos_w"], H, W, scale)
    else:
        out = rpb.attention(d["q"], d["k"], d["v"], rel_h.cuda(), rel_w.cuda(), H, W, scale,
                            out_dtype=torch.float32, workspace=workspace)
        want = oracle.attention(f["q"][:1], f["k"][:1], f["v"][:1], rel_h[:1].double().numpy(),
                                rel_w[:1].double().numpy(), H, W, scale)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - want)          # every head against the one oracle head (same problem)
    rl2 = np.linalg.norm(got - want) / (np.linalg.norm(want) * math.sqrt(heads))
    what = f"overshoot {entry} {H}x{W} {str(dtype)[6:]} {'workspace' if workspace is None else 'no-workspace'}"
    record_margin(what, err.max(), rl2)
    assert err.max() <= ABS_TOL, f"{what}: max-abs {err.max():.3e}"
    assert rl2 <= RL2_TOL


@pytest.mark.parametrize("entry", ["fused", "two_step"])
@pytest.mark.parametrize("name", list(I.WORKLOADS))
def test_rows_sum_to_one(name, entry):
    """V = 1 on the full workload: out = sum_m p_m / sum_m p_m = 1 on every row, whatever q, k and
    the tables are.  The kernel's P (fp16) feeds the numerator and its fp32 row sums the
    denominator, so this bounds their disagreement on every row of every head."""
    w = I.WORKLOADS[name]
    x = I.make_inputs(w)
    d = {n: t.cuda() for n, t in x.items()}
    d["v"] = torch.ones_like(d["v"])
    if entry == "fused":
        out = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale,
                        out_dtype=torch.float32)
    else:
        rh, rw = rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W)
        out = rpb.attention(d["q"], d["k"], d["v"], rh, rw, w.H, w.W, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    dev = (out.double() - 1.0).abs()
    err = float(dev.max())
    rl2 = float(torch.linalg.vector_norm(out.double() - 1.0) / math.sqrt(out.numel()))
    record_margin(f"rows sum to 1: {entry} {name} (all rows)", err, rl2, "2e-3 / 1e-2")
    assert bool(torch.isfinite(out).all())
    assert err <= 2e-3, f"{entry} {name}: max |out - 1| = {err:.3e}"


def ramp_case(H: int, W: int, heads: int, dtype: torch.dtype, pattern: str, seed: int = 11):
    """A rel_h term that moves the row maximum by a fixed pattern across the key grid rows, the
    same problem for every head.  q = a*e0 + small noise, T_h[i, 0] = f(i) / a, so
    rel_h[n, kh] = f(qh - kh + H - 1) (natural units), and the scores and rel_w stay small:
      "rise": f falls by 8 (base 2) per table row, so rel_h rises by 8 per key grid row and every
              key tile lifts the row maximum by about 16: each tile is taken exact at once, and
              the rel_h spread makes every warp start from the safe cap;
      "fall": the mirror image: the first key tile holds the maximum and later tiles sit far below;
      "zigzag": f is 24 (base 2) on pairs of table rows and 0 on the pairs between, so the
              maximum jumps on every other key tile."""
    a = 2.0
    scale = 0.125
    N = H * W
    g = torch.Generator().manual_seed(seed)
    q = 0.05 * torch.randn(N, 64, generator=g)
    q[:, 0] = a
    k = 0.5 * torch.randn(N, 64, generator=g)
    k[:, 0] = 0.0
    v = torch.randn(N, 64, generator=g)
    i = torch.arange(2 * H - 1, dtype=torch.float32)
    if pattern == "rise":
        f = -8.0 * i
    elif pattern == "fall":
        f = 8.0 * i
    else:
        f = torch.where((torch.div(i, 2, rounding_mode="floor") % 2) == 0, torch.tensor(24.0), torch.tensor(0.0))
    th = 0.1 * torch.randn(2 * H - 1, 64, generator=g)
    th[:, 0] = f / LOG2E / a
    tw = 0.1 * torch.randn(2 * W - 1, 64, generator=g)
    x = {"q": q, "k": k, "v": v, "rel_pos_h": th, "rel_pos_w": tw}
    x = {n: t.to(dtype) for n, t in x.items()}
    for n in ("q", "k", "v"):
        x[n] = x[n].expand(heads, N, 64).contiguous()
    return x, scale


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("grid", [(64, 64, 12), (40, 40, 24)], ids=["64x64", "40x40"])
@pytest.mark.parametrize("pattern", ["rise", "fall", "zigzag"])
@pytest.mark.parametrize("entry", ["fused", "attention"])
def test_rel_h_patterns(entry, pattern, grid, dtype):
    """Row maxima that move by large steps between key tiles: the tiles the kernel takes exact
    at once, the ones it exponentiates speculatively and the safe starting cap all meet here."""
    H, W, heads = grid
    x, scale = ramp_case(H, W, heads, dtype, pattern)
    d = {n: t.cuda() for n, t in x.items()}
    f = {n: I.to_f64(t) for n, t in x.items()}
    if entry == "fused":
        out = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], H, W, scale,
                        out_dtype=torch.float32)
    else:
        rh, rw = rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], H, W)
        out = rpb.attention(d["q"], d["k"], d["v"], rh, rw, H, W, scale, out_dtype=torch.float32)
    want = oracle.fused(f["q"][:1], f["k"][:1], f["v"][:1], f["rel_pos_h"], f["rel_pos_w"], H, W, scale)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - want)
    rl2 = np.linalg.norm(got - want) / (np.linalg.norm(want) * math.sqrt(heads))
    what = f"rel_h {pattern} {entry} {H}x{W} {str(dtype)[6:]}"
    record_margin(what, err.max(), rl2)
    assert err.max() <= ABS_TOL, f"{what}: max-abs {err.max():.3e}"
    assert rl2 <= RL2_TOL
