"""C-ABI boundary checks that need no GPU: the library builds and loads,
exports every entry point that include/dera_relpos.h declares, and rejects
bad arguments on the host before touching CUDA."""
from __future__ import annotations

import ctypes
import subprocess

import pytest
import torch

import relative_position_bias_gb300 as rpb
from relative_position_bias_gb300 import api
from relative_position_bias_gb300 import build as rbuild

EXPECTED = {"dera_relpos_project", "dera_relpos_attention", "dera_relpos_fused", "dera_status_string",
            "dera_relpos_device_status", "dera_relpos_selftest_wait_timeout", "dera_relpos_abi_version",
            "dera_relpos_workspace_size", "dera_relpos_fused_noalloc", "dera_relpos_fused_lse",
            "dera_relpos_backward_workspace_size", "dera_relpos_fused_backward"}

FAKE = 0x10000          # aligned, never dereferenced: every call below fails before any CUDA work
FAKE_MISALIGNED = 0x10008


@pytest.fixture(scope="module")
def lib():
    rbuild.build()
    return rpb.load_library()


def test_header_declares_the_entry_points():
    assert set(rpb.declared_entry_points()) == EXPECTED


def test_library_exports_every_declared_symbol(lib):
    for name in rpb.declared_entry_points():
        assert getattr(lib, name) is not None
    out = subprocess.run(["nm", "-D", "--defined-only", rbuild.LIB], capture_output=True, text=True, check=True)
    exported = {line.split()[-1] for line in out.stdout.splitlines() if " T " in line}
    assert EXPECTED <= exported
    # nothing else of ours leaks out of the shared object
    assert not {s for s in exported if s.startswith("_ZN4dera")}


def test_abi_version_and_status_strings(lib):
    assert lib.dera_relpos_abi_version() == 3
    for code, name in api.STATUS_NAMES.items():
        assert lib.dera_status_string(code).decode().startswith(name)
    assert lib.dera_status_string(99).decode() == "DERA_ERR_UNKNOWN"


def _fused(lib, *, ptrs=(FAKE,) * 6, BH=1, H=4, W=4, d=64, in_dt=1, out_dt=2):
    return lib.dera_relpos_fused(*ptrs, BH, H, W, d, 0.125, in_dt, out_dt, None, 0, None)


def _attn(lib, *, ptrs=(FAKE,) * 6, BH=1, H=4, W=4, d=64, in_dt=1, bias_dt=2, out_dt=2):
    return lib.dera_relpos_attention(*ptrs, BH, H, W, d, 0.125, in_dt, bias_dt, out_dt, None, 0, None)


def _proj(lib, *, ptrs=(FAKE,) * 5, BH=1, H=4, W=4, d=64, in_dt=1, bias_dt=2):
    return lib.dera_relpos_project(*ptrs, BH, H, W, d, in_dt, bias_dt, None)


@pytest.mark.parametrize("call", [_fused, _attn, _proj])
def test_host_validation(lib, call):
    assert call(lib, d=256) == 4                      # head_dim: 64 or 128
    assert call(lib, d=32) == 4
    assert call(lib, d=63) == 4
    assert call(lib, H=0) == 2                        # shape
    assert call(lib, W=65) == 2
    assert call(lib, BH=-1) == 2
    assert call(lib, in_dt=2) == 3                    # fp32 inputs are not a fast-path dtype
    assert call(lib, in_dt=7) == 3
    n = 5 if call is _proj else 6
    for i in range(n):
        ptrs = [FAKE] * n
        ptrs[i] = None
        assert call(lib, ptrs=tuple(ptrs)) == 1       # null
        ptrs[i] = FAKE_MISALIGNED
        assert call(lib, ptrs=tuple(ptrs)) == 5       # alignment
    assert call(lib, BH=0) == 0                       # empty batch: no work, no CUDA call
    assert call(lib, BH=0, ptrs=(None,) * n) == 0     # ... and no pointer is looked at


def test_workspace_size_validation(lib):
    n = ctypes.c_size_t(123)
    assert lib.dera_relpos_workspace_size(1, 4, 4, 64, None) == 1
    assert lib.dera_relpos_workspace_size(1, 4, 4, 32, ctypes.byref(n)) == 4
    assert lib.dera_relpos_workspace_size(1, 0, 4, 64, ctypes.byref(n)) == 2
    assert lib.dera_relpos_workspace_size(0, 4, 4, 64, ctypes.byref(n)) == 0 and n.value == 0


def test_dtype_rules(lib):
    assert _attn(lib, bias_dt=5) == 3
    assert _attn(lib, in_dt=1, out_dt=0) == 3         # out must be f32 or the input dtype
    assert _fused(lib, in_dt=0, out_dt=1) == 3
    assert _proj(lib, bias_dt=9) == 3


def test_binding_checks_shapes_before_calling():
    q = torch.zeros(2, 12, 64, dtype=torch.bfloat16)
    th, tw = torch.zeros(5, 64, dtype=torch.bfloat16), torch.zeros(7, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        rpb.project(q, th, tw, 3, 5)                  # N != H*W
    with pytest.raises(ValueError):
        rpb.project(q, th[:4], tw, 3, 4)              # table length != 2H-1
    with pytest.raises(ValueError):
        rpb.fused(q, q, q.transpose(0, 1).contiguous().transpose(0, 1), th, tw, 3, 4)  # not contiguous
    with pytest.raises(TypeError):
        rpb.fused(q, q.half(), q, th, tw, 3, 4)


def test_binding_raises_on_library_errors():
    # CPU tensors are not device memory: the library refuses them (or, with no
    # CUDA device at all, reports the failed device query); it never computes.
    q = torch.zeros(1, 16, 64, dtype=torch.bfloat16)
    th = torch.zeros(7, 64, dtype=torch.bfloat16)
    with pytest.raises(rpb.DeraError) as ei:
        rpb.fused(q, q, q, th, th, 4, 4, out_dtype=torch.float32)
    assert ei.value.status in (6, 8)


def _bwd(lib, *, ptrs=(FAKE,) * 13, BH=1, H=4, W=4, d=64, in_dt=1, out_dt=2, grad_dt=2, ws=FAKE, ws_bytes=1 << 30):
    return lib.dera_relpos_fused_backward(*ptrs, BH, H, W, d, 0.125, in_dt, out_dt, grad_dt, ws, ws_bytes, None)


def test_backward_rejects_before_any_cuda_work(lib):
    """Shape, head_dim, dtype, null and alignment errors of the backward entry, all decided on the host."""
    codes = {n: c for c, n in api.STATUS_NAMES.items()}
    assert _bwd(lib, d=128) == codes["DERA_ERR_HEAD_DIM"]
    assert _bwd(lib, H=65) == codes["DERA_ERR_SHAPE"]
    assert _bwd(lib, in_dt=2) == codes["DERA_ERR_DTYPE"]           # fp32 inputs
    assert _bwd(lib, out_dt=0) == codes["DERA_ERR_DTYPE"]          # fp16 out with bf16 inputs
    assert _bwd(lib, grad_dt=0) == codes["DERA_ERR_DTYPE"]
    assert _bwd(lib, ptrs=(FAKE,) * 12 + (None,)) == codes["DERA_ERR_NULL"]
    assert _bwd(lib, ptrs=(FAKE_MISALIGNED,) + (FAKE,) * 12) == codes["DERA_ERR_ALIGN"]
    lse = lib.dera_relpos_fused_lse(*(FAKE,) * 7, 1, 4, 4, 64, 0.125, 1, 2, None, 0, None)
    assert lse == codes["DERA_OK"] or lse in (codes["DERA_ERR_CUDA"], codes["DERA_ERR_DEVICE"])
    assert lib.dera_relpos_fused_lse(*(FAKE,) * 6, None, 1, 4, 4, 64, 0.125, 1, 2, None, 0, None) == codes["DERA_ERR_NULL"]


def test_backward_workspace_size_formula(lib):
    """fp32 regions, each 256-byte aligned: rel_h, rel_w, D, the exponent's rel_h term by key grid
    row over whole query tiles, per-query-tile table-gradient partials."""
    def a256(x):
        return (x + 255) // 256 * 256
    for BH, H, W in [(1, 4, 4), (12, 64, 64), (3, 40, 40), (2, 14, 14), (5, 7, 30)]:
        rows, nq = BH * H * W, -(-(H * W) // 128)
        want = (a256(4 * rows * H) + a256(4 * rows * W) + a256(4 * rows) + a256(4 * BH * H * nq * 128)
                + a256(4 * BH * nq * (2 * H - 1 + 2 * W - 1) * 64))
        assert rpb.backward_workspace_size(BH, H, W, 64) == want
    with pytest.raises(rpb.DeraError):
        rpb.backward_workspace_size(1, 4, 4, 128)
