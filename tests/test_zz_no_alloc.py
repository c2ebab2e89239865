"""The allocation-free fused entry point, dera_relpos_fused_noalloc.

Some callers of this library cannot allocate device memory at all (a plug-in
inside a host engine that owns all device memory, or code that must never
trigger the synchronisation an allocation can cause), so they cannot supply
the scratch workspace that dera_relpos_fused uses when it splits work units
between CTAs.  dera_relpos_fused_noalloc takes that scratch from a buffer
compiled into the library instead.  This test calls it through the C ABI
(ctypes, no binding helper) twice in a row on workloads whose schedule does
split units (head_dim 64 and 128), and compares each result with dera_relpos_fused's, within the
tolerance the parity tests use (max-abs 4e-3, relative L2 1e-2).  It lives in
its own file, collected last, and passes alone or after the other tests.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import relative_position_bias_gb300 as rpb
from relative_position_bias_gb300 import build as rbuild
from relative_position_bias_gb300 import inputs as I

pytestmark = pytest.mark.gpu

ABS_TOL = 4e-3
RL2_TOL = 1e-2
DERA_F32, DERA_BF16 = 2, 1
DERA_ERR_SCRATCH = 9


def _noalloc(lib):
    fn = lib.dera_relpos_fused_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, i, i, vp]
    fn.restype = i
    return fn


@pytest.mark.parametrize("name", ["global64", "global64d128"])
def test_noalloc_matches_fused_on_two_calls(name):
    rbuild.build()
    lib = rpb.load_library()
    fn = _noalloc(lib)
    w = I.WORKLOADS[name]
    assert rpb.workspace_size(w.BH, w.H, w.W, w.d) > 0, "this workload must use the split schedule"
    x = I.make_inputs(w)
    d = {k: t.cuda() for k, t in x.items()}
    ref = rpb.fused(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale,
                    out_dtype=torch.float32)
    torch.cuda.synchronize()
    refn = ref.double().cpu().numpy()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((w.BH, w.N, w.d), float("nan"), dtype=torch.float32, device="cuda")
        st = fn(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["rel_pos_h"].data_ptr(),
                d["rel_pos_w"].data_ptr(), out.data_ptr(), w.BH, w.H, w.W, w.d, w.scale, DERA_BF16, DERA_F32,
                stream)
        assert st == 0, lib.dera_status_string(st).decode()
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        err = np.abs(got - refn)
        assert np.isfinite(got).all(), f"call {call}: unwritten output"
        assert err.max() <= ABS_TOL, f"call {call}: max-abs {err.max():.3e} vs dera_relpos_fused"
        assert np.linalg.norm(got - refn) / np.linalg.norm(refn) <= RL2_TOL
    assert rpb.device_status() == 0


def test_noalloc_rejects_problems_beyond_its_buffer():
    rbuild.build()
    lib = rpb.load_library()
    fn = _noalloc(lib)
    # A head count whose unit counters alone exceed the 48 MiB buffer: refused before anything
    # is enqueued.  The pointers are 16-byte aligned pinned HOST memory, so even if the size
    # check ever stopped firing, the device-memory check would still refuse the call
    # (DERA_ERR_DEVICE) and nothing could be launched on them.
    BH = 9_000_001   # 64x64 grid: millions of units
    need = rpb.workspace_size(BH, 64, 64)
    if need == 0:    # whole waves on this device: nudge the count so the split schedule applies
        BH += 1
        need = rpb.workspace_size(BH, 64, 64)
    assert need > 48 * 1024 * 1024
    t = torch.zeros(64, dtype=torch.bfloat16).pin_memory()
    p = t.data_ptr()
    assert p % 16 == 0
    st = fn(p, p, p, p, p, p, BH, 64, 64, 64, 0.125, DERA_BF16, DERA_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == DERA_ERR_SCRATCH, lib.dera_status_string(st).decode()
    assert "scratch" in lib.dera_status_string(st).decode()
