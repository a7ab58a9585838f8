"""int4_weight_only_w4_gb300 -- weight-only INT4 (group 128) GEMV for GB300.

The compute path is the C-ABI library ``libw4.so`` (hand-written CUDA for
sm_103a, built in-tree by ``__graft_entry__.build()``).  ``w4`` is the thin
ctypes binding to it; ``synthetic`` draws seeded inputs.  The binding is loaded
on first use and raises if the CUDA library is missing: there is no CPU
fallback.
"""
from __future__ import annotations

import importlib

_BINDING_NAMES = {
    "W4Error", "Status", "repacked_sizes", "repack", "dequant", "gemv", "gemv_f32",
    "PackedWeight", "pack", "status_string", "library_path", "check_header",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        mod = importlib.import_module(".w4", __name__)
        return getattr(mod, name)
    raise AttributeError(name)
