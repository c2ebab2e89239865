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
