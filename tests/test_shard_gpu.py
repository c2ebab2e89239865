"""The BH-range split of one call (relative_position_bias_gb300.shard) on the GPU.

Each rank of a world runs the fused entry on its contiguous (batch, head) range; nothing is
exchanged while computing.  On one GPU the ranks' slices are computed one after another in this
process (no collective), and their concatenation must match the whole call within the parity
tolerance: the slices' schedules cut units at other places than the whole call's, so the
results need not be bit-identical, only equally close to the exact attention.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import relative_position_bias_gb300 as rpb
from relative_position_bias_gb300 import build as rbuild
from relative_position_bias_gb300 import inputs as I
from relative_position_bias_gb300 import shard

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    rbuild.build()
    rpb.load_library()
    yield
    assert rpb.device_status() == 0


@pytest.mark.parametrize("world", [2, 3, 5])
@pytest.mark.parametrize("name", ["global64", "ragged40"])
def test_rank_slices_concatenate_to_the_whole_call(name, world):
    w = I.WORKLOADS[name]
    x = I.make_inputs(w)
    d = {k: t.cuda() for k, t in x.items()}
    args = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
    whole = rpb.fused(*args, out_dtype=torch.float32)
    parts = [shard.fused_shard(*args, rank=r, world=world, out_dtype=torch.float32) for r in range(world)]
    torch.cuda.synchronize()
    for r, p in enumerate(parts):
        lo, hi = shard.bh_range(w.BH, r, world)
        assert tuple(p.shape) == (hi - lo, w.N, w.d)
    got = torch.cat(parts).double().cpu().numpy()
    want = whole.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - want)
    # both are within 4e-3 of the float64 oracle (the parity tests), so within 8e-3 of each other
    assert err.max() <= 8e-3, f"max-abs {err.max():.3e}"
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 1e-2


@pytest.mark.parametrize("world", [2, 3])
def test_backward_rank_slices(world):
    """The backward's dq, dk, dv for a rank's BH range are exactly the whole call's rows (every
    CTA works within one (batch, head)); the ranks' table-gradient partials add up to the whole
    call's table gradients."""
    w = I.WORKLOADS["global64"]
    x = I.make_inputs(w)
    d = {k: t.cuda() for k, t in x.items()}
    fargs = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
    out, lse = rpb.fused_lse(*fargs, out_dtype=torch.float32)
    dout = torch.randn(w.BH, w.N, w.d, generator=torch.Generator().manual_seed(4)).to(w.torch_dtype).cuda()
    whole = rpb.fused_backward(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], out, lse, dout, w.H, w.W,
                               w.scale)
    parts = [shard.fused_backward_shard(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], out, lse, dout,
                                        w.H, w.W, w.scale, rank=r, world=world, reduce_tables=False)
             for r in range(world)]
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(torch.cat([p[i] for p in parts]), whole[i])
    for i in (3, 4):
        total = sum(p[i].double() for p in parts)
        ref = whole[i].double()
        assert float((total - ref).abs().max()) <= 1e-4 * float(ref.abs().max())
