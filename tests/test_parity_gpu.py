"""GPU parity of the CUDA path against the CPU float64 oracle.

Inputs come from the seeded generator (relative_position_bias_gb300.inputs)
and are rounded to the workload dtype once; the same bytes go to the GPU and,
widened exactly to float64, to the oracle.

Tolerances (from the target stated for this method: max-abs 4e-3 and
relative L2 1e-2 against the float64 oracle):
  * fp32 output mode: |out - oracle| <= 4e-3 everywhere, rel-L2 <= 1e-2.
  * 16-bit output: the kernel's only extra step is the final round-to-nearest,
    which alone can move a value by half an ulp of the output dtype (for bf16
    and |out| in [2, 4) that is 7.8e-3, above 4e-3).  So a 16-bit output must
    be bit-equal to the rounded fp32-mode output of the same call, and within
    4e-3 + ulp/2 of the oracle, and rel-L2 <= 1e-2.
  * projection: fp32 accumulation of 64 exact products; |err| <= 2e-4 * (1 + |x|).
"""
from __future__ import annotations

import re
from pathlib import Path

from dataclasses import replace

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
MANT_BITS = {torch.bfloat16: 7, torch.float16: 10}


@pytest.fixture(scope="module", autouse=True)
def _built():
    rbuild.build()
    rpb.load_library()
    yield
    assert rpb.device_status() == 0, "a kernel hit its bounded-wait budget"


def _dev(x: dict) -> dict:
    return {k: t.cuda() for k, t in x.items()}


def _f64(x: dict) -> dict:
    return {k: I.to_f64(t) for k, t in x.items()}


def half_ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return 0.5 * 2.0 ** (np.floor(np.log2(ax)) - MANT_BITS[dtype])


def check_out(got32: torch.Tensor, want: np.ndarray, got16: torch.Tensor | None = None, what: str = ""):
    g = got32.double().cpu().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - want)
    rl2 = np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-300)
    record_margin(what, err.max(), rl2)
    assert err.max() <= ABS_TOL, f"{what}: max-abs {err.max():.3e}"
    assert rl2 <= RL2_TOL, f"{what}: rel-L2 {rl2:.3e}"
    if got16 is not None:
        rounded = got32.to(got16.dtype)
        assert torch.equal(got16.view(torch.int16), rounded.view(torch.int16)), f"{what}: 16-bit != RN(fp32 mode)"
        g16 = got16.double().cpu().numpy()
        assert (np.abs(g16 - want) <= ABS_TOL + half_ulp(want, got16.dtype)).all(), f"{what}: 16-bit bound"
        assert np.linalg.norm(g16 - want) / np.linalg.norm(want) <= RL2_TOL
    return float(err.max()), float(rl2)


_ATTN_SRC = Path(__file__).resolve().parents[1] / "relative_position_bias_gb300" / "csrc" / "attention.cuh"


def query_tiles_per_unit() -> int:
    """Query tiles (of 128 rows) in one work unit of the attention kernel's schedule."""
    m = re.search(r"constexpr int kTilesPerUnit = (\d+);", _ATTN_SRC.read_text())
    assert m, "kTilesPerUnit not found"
    return int(m.group(1))


def default_plan(w: I.Workload) -> tuple[bool, int, int]:
    """(split, units, units per head) of the default (workspace) schedule, restated from the host
    plan: units are groups of query tiles of one head; the work is split when the units do not
    fill whole waves of one CTA per SM and a unit spans at least 4 key tiles (whole grid rows of
    the padded width 16, 32, 40 or 64 per tile, fewer rows with head_dim 128)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per = query_tiles_per_unit()
    units_per_head = (-(-w.N // 128) + per - 1) // per
    U = w.BH * units_per_head
    wp = next(x for x in (16, 32, 40, 64) if x >= w.W)
    kht = {16: 8, 32: 4, 40: 3, 64: 2}[wp] if w.d == 64 else {16: 4, 32: 2, 40: 2, 64: 1}[wp]
    n_kv = -(-w.H // kht)
    return (n_kv >= 4 and U > sms and U % sms != 0), U, units_per_head


def tail_heads(w: I.Workload) -> set[int]:
    """Heads with a unit in the stream-K tail of the default schedule: the last one and a fraction
    waves of units when the work is split.  Cut units only occur there."""
    split, U, units_per_head = default_plan(w)
    if not split:
        return set()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    first_tail = max(U // sms - 1, 0) * sms
    return {u // units_per_head for u in range(first_tail, U)}


def dense_heads(w: I.Workload, at_least: int = 16, seed: int = 0) -> list[int]:
    """Heads checked on every row: the first and last heads, every head holding a tail (possibly
    cut) unit, and random others up to `at_least`."""
    r = np.random.default_rng(seed)
    heads = {0, 1, w.BH - 1} | tail_heads(w)
    heads = {h for h in heads if 0 <= h < w.BH}
    rest = [h for h in r.permutation(w.BH).tolist() if h not in heads]
    heads |= set(rest[:max(0, at_least - len(heads))])
    return sorted(heads)


# --------------------------------------------------------------------------- projection
@pytest.mark.parametrize("name", list(I.WORKLOADS))
def test_project_parity(name):
    w = I.WORKLOADS[name]
    x = I.make_inputs(w)
    d = _dev(x)
    rh, rw = rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W)
    torch.cuda.synchronize()
    f = _f64(x)
    want_h, want_w = oracle.project(f["q"], f["rel_pos_h"], f["rel_pos_w"], w.H, w.W)
    for got, want in ((rh, want_h), (rw, want_w)):
        g = got.double().cpu().numpy()
        assert (np.abs(g - want) <= 2e-4 * (1 + np.abs(want))).all(), np.abs(g - want).max()


@pytest.mark.parametrize("bias_dtype", [torch.bfloat16, torch.float16])
def test_project_16bit_bias(bias_dtype):
    w = I.WORKLOADS["global64"].with_grid(24, 40, B=1, heads=3)
    x = I.make_inputs(w, seed=3)
    d = _dev(x)
    rh32, rw32 = rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W)
    rh, rw = rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, bias_dtype=bias_dtype)
    torch.cuda.synchronize()
    assert torch.equal(rh, rh32.to(bias_dtype)) and torch.equal(rw, rw32.to(bias_dtype))


# --------------------------------------------------------------------------- full workloads
_ORACLE_CACHE: dict = {}


def _oracle_full_or_heads(w, f, entry, rel=None, cache_key=None):
    """The whole oracle output: every head of every workload up to batched64's size (the oracle
    takes the heads one at a time; batched64's 96 heads take seconds), else every row of the
    heads `dense_heads` picks.  With `cache_key`, a result is kept for the next test that asks
    for the same output."""
    if cache_key is not None and cache_key in _ORACLE_CACHE:
        return _ORACLE_CACHE[cache_key]
    heads = None if w.BH * w.N * w.N <= 96 * 4096 * 4096 else dense_heads(w)
    sel = (lambda a: a) if heads is None else (lambda a: a[heads])
    if entry == "fused":
        want = oracle.fused(sel(f["q"]), sel(f["k"]), sel(f["v"]), f["rel_pos_h"], f["rel_pos_w"], w.H, w.W, w.scale)
    else:
        want = oracle.attention(sel(f["q"]), sel(f["k"]), sel(f["v"]), sel(rel[0]), sel(rel[1]), w.H, w.W, w.scale)
    if cache_key is not None:
        _ORACLE_CACHE[cache_key] = (heads, want)
    return heads, want


def _select(t: torch.Tensor, heads):
    return t if heads is None else t[heads]


@pytest.mark.parametrize("split", [True, False], ids=["workspace", "no-workspace"])
@pytest.mark.parametrize("name", list(I.WORKLOADS))
def test_fused_parity(name, split):
    """Default call (scratch workspace: units split across CTAs where that evens
    the load) and the one-CTA-per-unit schedule, both against the oracle."""
    w = I.WORKLOADS[name]
    x = I.make_inputs(w)
    d = _dev(x)
    args = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
    ws = None if split else False
    o32 = rpb.fused(*args, out_dtype=torch.float32, workspace=ws)
    o16 = rpb.fused(*args, workspace=ws)
    torch.cuda.synchronize()
    # every row, not only the sampled ones, must be finite
    assert bool(torch.isfinite(o32).all()) and bool(torch.isfinite(o16).all()), f"fused {name}: non-finite output"
    heads, want = _oracle_full_or_heads(w, _f64(x), "fused", cache_key=("fused", name))
    check_out(_select(o32, heads), want, _select(o16, heads),
              what=f"fused {name} {'workspace' if split else 'no-workspace'}" + ("" if heads is None else f" ({len(heads)} heads)"))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", ["inf", "clamp", "raise"])
@pytest.mark.parametrize("entry", ["fused", "attention"])
def test_late_large_scores(entry, case, dtype):
    """Scores in a late key tile far above everything before them in the row.

    The kernel exponentiates each tile against the row maximum it has seen so
    far and stores P in fp16, so these rows exercise its overflow handling:
    "inf": one key 150 (base-2 units) above the rest, whose 2^x overflows even
    fp32; "clamp": one key about 18 above the running maximum (p beyond the
    fp16 range); "raise": a whole tile about 12 above it (the row sum passes
    the kernel's bound with every p still in range).  All must match the oracle."""
    base = I.WORKLOADS["grid16"] if dtype == "bf16" else I.WORKLOADS["ragged40"]
    w = base.with_grid(32, 32, B=1, heads=2)
    x = I.make_inputs(w, seed=11)
    tdt = x["q"].dtype
    q, k = x["q"].float(), x["k"].float()
    q[..., 0] = 2.0
    if case == "inf":
        k[:, 677, :] = 0.0
        k[:, 677, 0] = 416.0   # q.k = 832: 150 in base-2 units after scale * log2(e)
    elif case == "clamp":
        k[:, 677, :] = 0.0
        k[:, 677, 0] = 60.0    # about 21.6 in base-2 units
    else:
        k[:, 640:768, 0] += 33.0  # about +11.9 for the whole key tile 5
    x["q"], x["k"] = q.to(tdt), k.to(tdt)
    x["rel_pos_h"] = (x["rel_pos_h"].float() * 0.1).to(tdt)
    x["rel_pos_w"] = (x["rel_pos_w"].float() * 0.1).to(tdt)
    d, f = _dev(x), _f64(x)
    if entry == "fused":
        args = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
        o32 = rpb.fused(*args, out_dtype=torch.float32)
        o16 = rpb.fused(*args)
        torch.cuda.synchronize()
        want = oracle.fused(f["q"], f["k"], f["v"], f["rel_pos_h"], f["rel_pos_w"], w.H, w.W, w.scale)
    else:
        rh, rw = oracle.project(f["q"], f["rel_pos_h"], f["rel_pos_w"], w.H, w.W)
        rh32, rw32 = torch.from_numpy(rh).float(), torch.from_numpy(rw).float()
        args = (d["q"], d["k"], d["v"], rh32.cuda(), rw32.cuda(), w.H, w.W, w.scale)
        o32 = rpb.attention(*args, out_dtype=torch.float32)
        o16 = rpb.attention(*args)
        torch.cuda.synchronize()
        want = oracle.attention(f["q"], f["k"], f["v"], rh32.double().numpy(), rw32.double().numpy(), w.H, w.W,
                                w.scale)
    check_out(o32, want, o16, what=f"late large scores {entry} {case} {dtype}")


@pytest.mark.parametrize("entry", ["fused", "attention"])
@pytest.mark.parametrize("BH", [None, 1, 2, 3], ids=["sms+1", "sms+sms/2", "2sms+1", "3sms-1"])
def test_split_schedule_ragged(entry, BH):
    """Unit counts just past whole waves of the device, on a ragged 40x40 grid
    (13 query tiles per head), so most units are cut between two CTAs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_head = (-(-1600 // 128) + query_tiles_per_unit() - 1) // query_tiles_per_unit()
    units = {None: sms + 1, 1: sms + sms // 2, 2: 2 * sms + 1, 3: 3 * sms - 1}[BH]
    heads = -(-units // per_head)
    w = I.WORKLOADS["ragged40"].with_grid(40, 40, B=1, heads=heads)
    assert rpb.workspace_size(w.BH, w.H, w.W, w.d) > 0
    x = I.make_inputs(w, seed=heads)
    d = _dev(x)
    f = _f64(x)
    if entry == "fused":
        o32 = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale,
                        out_dtype=torch.float32)
        torch.cuda.synchronize()
        heads_s, want = _oracle_full_or_heads(w, f, "fused")
    else:
        rh, rw = oracle.project(f["q"], f["rel_pos_h"], f["rel_pos_w"], w.H, w.W)
        rh32, rw32 = torch.from_numpy(rh).float(), torch.from_numpy(rw).float()
        o32 = rpb.attention(d["q"], d["k"], d["v"], rh32.cuda(), rw32.cuda(), w.H, w.W, w.scale,
                            out_dtype=torch.float32)
        torch.cuda.synchronize()
        heads_s, want = _oracle_full_or_heads(w, f, "attention", (rh32.double().numpy(), rw32.double().numpy()))
    check_out(_select(o32, heads_s), want, what=f"split {entry} {w.BH} heads")


@pytest.mark.parametrize("name", list(I.WORKLOADS))
def test_workspace_size_formula(name):
    """The reported scratch is the documented layout: an 8-byte counter per query tile of each
    unit (256-byte aligned), then two 66-float-per-row slots per CTA and query tile of a unit;
    zero when the units fill whole waves of one CTA per SM or span fewer than 4 key tiles."""
    w = I.WORKLOADS[name]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per = query_tiles_per_unit()
    split, units, _ = default_plan(w)
    want = ((8 * per * units + 255) // 256 * 256 + 2 * sms * per * 128 * (w.d + 2) * 4) if split else 0
    assert rpb.workspace_size(w.BH, w.H, w.W, w.d) == want


def test_caller_workspace_and_reuse():
    """A caller-owned workspace gives the same bytes as the cached one, call after call."""
    w = I.WORKLOADS["global64"]
    d = _dev(I.make_inputs(w))
    args = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
    ref = rpb.fused(*args)
    ws = torch.empty(rpb.workspace_size(w.BH, w.H, w.W, w.d), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        again = rpb.fused(*args, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(again, ref)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")          # too small: one CTA per unit
    alt = rpb.fused(*args, out_dtype=torch.float32, workspace=small)
    torch.cuda.synchronize()
    f = _f64(I.make_inputs(w))
    check_out(alt, oracle.fused(f["q"], f["k"], f["v"], f["rel_pos_h"], f["rel_pos_w"], w.H, w.W, w.scale),
              what="fused global64 workspace too small")


def test_default_workspace_per_stream():
    """Calls on two streams that overlap on the GPU each get their own cached scratch, so both
    match a serial call bit for bit."""
    w = I.WORKLOADS["global64"]
    assert rpb.workspace_size(w.BH, w.H, w.W, w.d) > 0, "this workload must use the split schedule"
    d = _dev(I.make_inputs(w))
    d2 = _dev(I.make_inputs(w, seed=1))
    ref1 = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
    ref2 = rpb.fused(d2["q"], d2["k"], d2["v"], d2["rel_pos_h"], d2["rel_pos_w"], w.H, w.W, w.scale)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            a = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
        with torch.cuda.stream(s2):
            b = rpb.fused(d2["q"], d2["k"], d2["v"], d2["rel_pos_h"], d2["rel_pos_w"], w.H, w.W, w.scale)
        outs.append((a, b))
    torch.cuda.synchronize()
    for a, b in outs:
        assert torch.equal(a, ref1) and torch.equal(b, ref2)


@pytest.mark.parametrize("entry", ["fused", "attention"])
@pytest.mark.parametrize("name", ["global64", "ragged40"])
def test_workspace_contents_are_ignored(name, entry):
    """The split schedule's counters carry a per-launch tag, so a workspace
    full of arbitrary bytes (never cleared) gives the same result as the
    library's own workspace, call after call."""
    w = I.WORKLOADS[name]
    assert rpb.workspace_size(w.BH, w.H, w.W, w.d) > 0, "this workload must use the split schedule"
    d = _dev(I.make_inputs(w))
    if entry == "fused":
        args = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
        call = rpb.fused
    else:
        rh, rw = rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W)
        args = (d["q"], d["k"], d["v"], rh, rw, w.H, w.W, w.scale)
        call = rpb.attention
    ref = call(*args)
    ws = torch.empty(rpb.workspace_size(w.BH, w.H, w.W, w.d), dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(11)
    for trial in range(4):
        if trial < 3:
            ws.random_(0, 256, generator=g)   # the last call reuses what the previous one left
        got = call(*args, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"trial {trial}"


@pytest.mark.parametrize("name", list(I.WORKLOADS))
def test_attention_parity_f32_bias(name):
    """Compact-bias entry fed the oracle's projection (rounded to fp32); the
    oracle consumes exactly those fp32 values."""
    w = I.WORKLOADS[name]
    x = I.make_inputs(w)
    f = _f64(x)
    rh, rw = oracle.project(f["q"], f["rel_pos_h"], f["rel_pos_w"], w.H, w.W)
    rh32, rw32 = torch.from_numpy(rh).float(), torch.from_numpy(rw).float()
    d = _dev(x)
    o32 = rpb.attention(d["q"], d["k"], d["v"], rh32.cuda(), rw32.cuda(), w.H, w.W, w.scale,
                        out_dtype=torch.float32)
    o16 = rpb.attention(d["q"], d["k"], d["v"], rh32.cuda(), rw32.cuda(), w.H, w.W, w.scale)
    torch.cuda.synchronize()
    rel = (rh32.double().numpy(), rw32.double().numpy())
    heads, want = _oracle_full_or_heads(w, f, "attention", rel)
    check_out(_select(o32, heads), want, _select(o16, heads),
              what=f"attention {name}" + ("" if heads is None else f" ({len(heads)} heads)"))


@pytest.mark.parametrize("bias_dtype", [torch.bfloat16, torch.float16])
def test_attention_16bit_bias(bias_dtype):
    """A 16-bit compact bias: the oracle consumes the same rounded values."""
    w = I.WORKLOADS["grid16"].with_grid(24, 24, B=2, heads=3)
    x = I.make_inputs(w, seed=5)
    f = _f64(x)
    rh, rw = oracle.project(f["q"], f["rel_pos_h"], f["rel_pos_w"], w.H, w.W)
    rh16, rw16 = torch.from_numpy(rh).to(bias_dtype), torch.from_numpy(rw).to(bias_dtype)
    d = _dev(x)
    o32 = rpb.attention(d["q"], d["k"], d["v"], rh16.cuda(), rw16.cuda(), w.H, w.W, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    want = oracle.attention(f["q"], f["k"], f["v"], rh16.double().numpy(), rw16.double().numpy(), w.H, w.W, w.scale)
    check_out(o32, want, what="attention 16-bit bias")


def test_two_step_matches_oracle():
    """dera_relpos_project then dera_relpos_attention against the oracle's fused result."""
    w = I.WORKLOADS["global64"]
    x = I.make_inputs(w)
    d = _dev(x)
    rh, rw = rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W)
    o32 = rpb.attention(d["q"], d["k"], d["v"], rh, rw, w.H, w.W, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    f = _f64(x)
    want = oracle.fused(f["q"], f["k"], f["v"], f["rel_pos_h"], f["rel_pos_w"], w.H, w.W, w.scale)
    check_out(o32, want, what="two-step global64")


# --------------------------------------------------------------------------- edge grids
EDGE_GRIDS = [(1, 1), (1, 2), (2, 1), (3, 5), (5, 3), (17, 13), (1, 64), (64, 1), (7, 40), (33, 33), (20, 48),
              (64, 17), (5, 64), (2, 16), (9, 16), (16, 9), (40, 40), (63, 63), (11, 37), (64, 33)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("grid", EDGE_GRIDS, ids=lambda g: f"{g[0]}x{g[1]}")
def test_edge_grids(grid, dtype):
    H, W = grid
    base = I.WORKLOADS["ragged40"] if dtype == "f16" else I.WORKLOADS["grid16"]
    w = base.with_grid(H, W, B=1, heads=3)
    x = I.make_inputs(w, seed=H * 97 + W)
    d = _dev(x)
    f = _f64(x)
    o32 = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], H, W, w.scale, out_dtype=torch.float32)
    rh, rw = rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], H, W)
    a32 = rpb.attention(d["q"], d["k"], d["v"], rh, rw, H, W, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    want = oracle.fused(f["q"], f["k"], f["v"], f["rel_pos_h"], f["rel_pos_w"], H, W, w.scale)
    check_out(o32, want, what=f"fused {H}x{W} {dtype}")
    check_out(a32, want, what=f"two-step {H}x{W} {dtype}")


EDGE_GRIDS_D128 = [(1, 1), (3, 5), (17, 13), (64, 1), (7, 40), (33, 33), (20, 48), (2, 16), (40, 40), (64, 33),
                   (11, 37), (64, 64)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("grid", EDGE_GRIDS_D128, ids=lambda g: f"{g[0]}x{g[1]}")
def test_edge_grids_head_dim_128(grid, dtype):
    """head_dim 128 on every padded width (16, 32, 40, 64: key tiles of 4, 2, 2 and 1 grid rows),
    ragged tails and single rows or columns, fused and two-step, against the oracle."""
    H, W = grid
    base = I.WORKLOADS["ragged40"] if dtype == "f16" else I.WORKLOADS["global64d128"]
    w = replace(base.with_grid(H, W, B=1, heads=3), d=128, scale=128 ** -0.5)
    x = I.make_inputs(w, seed=H * 89 + W)
    d = _dev(x)
    f = _f64(x)
    o32 = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], H, W, w.scale, out_dtype=torch.float32)
    o16 = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], H, W, w.scale)
    rh, rw = rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], H, W)
    a32 = rpb.attention(d["q"], d["k"], d["v"], rh, rw, H, W, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    want_h, want_w = oracle.project(f["q"], f["rel_pos_h"], f["rel_pos_w"], H, W)
    assert np.abs(rh.double().cpu().numpy() - want_h).max() <= 2e-4 * (1 + np.abs(want_h).max())
    assert np.abs(rw.double().cpu().numpy() - want_w).max() <= 2e-4 * (1 + np.abs(want_w).max())
    want = oracle.fused(f["q"], f["k"], f["v"], f["rel_pos_h"], f["rel_pos_w"], H, W, w.scale)
    check_out(o32, want, o16, what=f"fused d128 {H}x{W} {dtype}")
    check_out(a32, want, what=f"two-step d128 {H}x{W} {dtype}")


def test_empty_batch_is_a_noop():
    w = I.WORKLOADS["grid16"]
    q = torch.empty(0, w.N, 64, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(2 * w.H - 1, 64, dtype=torch.bfloat16, device="cuda")
    out = rpb.fused(q, q, q, t, t, w.H, w.W, w.scale)
    assert out.shape == (0, w.N, 64)


# --------------------------------------------------------------------------- properties of the call
def test_deterministic_and_graph_capturable():
    w = I.WORKLOADS["global64"]
    d = _dev(I.make_inputs(w))
    args = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
    a = rpb.fused(*args)
    b = rpb.fused(*args)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    out = torch.empty_like(a)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rpb.fused(*args, out=out)          # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        rpb.fused(*args, out=out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, a)


def test_no_device_allocation_in_calls():
    w = I.WORKLOADS["global64"]
    x = I.make_inputs(w)
    d = _dev(x)
    out = torch.empty(w.BH, w.N, 64, dtype=torch.bfloat16, device="cuda")
    rh = torch.empty(w.BH, w.N, w.H, device="cuda")
    rw = torch.empty(w.BH, w.N, w.W, device="cuda")
    args = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
    rpb.fused(*args, out=out)
    rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, rel_h=rh, rel_w=rw)
    rpb.attention(d["q"], d["k"], d["v"], rh, rw, w.H, w.W, w.scale, out=out)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        rpb.fused(*args, out=out)
        rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, rel_h=rh, rel_w=rw)
        rpb.attention(d["q"], d["k"], d["v"], rh, rw, w.H, w.W, w.scale, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.max_memory_allocated() == alloc0
    assert free1 == free0


def test_rejects_host_and_misaligned_pointers():
    w = I.WORKLOADS["grid16"]
    x = I.make_inputs(w)
    d = _dev(x)
    with pytest.raises(rpb.DeraError) as ei:
        rpb.fused(x["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W)
    assert ei.value.status == 6
    pinned = x["v"].pin_memory()
    with pytest.raises(rpb.DeraError) as ei:
        rpb.fused(d["q"], d["k"], pinned, d["rel_pos_h"], d["rel_pos_w"], w.H, w.W)
    assert ei.value.status == 6
    buf = torch.empty(w.BH * w.N * 64 + 8, dtype=torch.bfloat16, device="cuda")
    qm = buf[1:1 + w.BH * w.N * 64].view(w.BH, w.N, 64)      # 2-byte offset
    with pytest.raises(rpb.DeraError) as ei:
        rpb.fused(qm, d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W)
    assert ei.value.status == 5


def test_bounded_wait_reports_timeout_and_context_survives():
    assert rpb.device_status(reset=True) == 0
    rpb.selftest_wait_timeout(budget_cycles=2_000_000)
    assert rpb.device_status(reset=True) == 7
    assert rpb.device_status(reset=False) == 0
    # the context is still usable
    w = I.WORKLOADS["grid16"]
    x = I.make_inputs(w)
    d = _dev(x)
    out = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    f = _f64(x)
    check_out(out, oracle.fused(f["q"], f["k"], f["v"], f["rel_pos_h"], f["rel_pos_w"], w.H, w.W, w.scale),
              what="fused grid16 after a timed-out wait")
