"""GB300-native global attention with decomposed relative-position bias.

The computation lives in ``libdera_relpos.so`` (hand-written sm_103a CUDA
behind a C ABI, declared in ``include/dera_relpos.h``); this package is its
thin Python binding.  Entry points: :func:`project`, :func:`attention`,
:func:`fused`; for training, :func:`fused_lse` and :func:`fused_backward`.
"""
from .api import (DERA_BF16, DERA_F16, DERA_F32, DeraError, attention, backward_workspace_size, declared_entry_points,
                  device_status, fused, fused_backward, fused_lse, load_library, project, selftest_wait_timeout,
                  workspace_size)

__all__ = ["DERA_BF16", "DERA_F16", "DERA_F32", "DeraError", "attention", "backward_workspace_size",
           "declared_entry_points", "device_status", "fused", "fused_backward", "fused_lse", "load_library", "project",
           "selftest_wait_timeout", "workspace_size"]
