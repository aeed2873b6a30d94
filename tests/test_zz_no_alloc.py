"""The forward entry point that allocates nothing (loglinear_fwd_static_workspace).

Some callers may not allocate device memory while they run: a plugin whose host
application owns every device allocation, or code that shares the CUDA context with a
caching allocator it must not disturb.  For them the library keeps a fixed 32 MiB device
array as the forward's workspace.  These tests call that entry point through the C ABI
twice in a row and compare each result with loglinear_fwd (caller-provided workspace)
within the parity tolerance used everywhere else; the first call on the device also
performs the one-time address lookup of the array.

This file is collected last on purpose, so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from parity_util import assert_parity
from structured_mask_linear_gb300.inputs import levels_for, make_inputs, workload


def test_static_workspace_rejects_oversized_shapes():
    """Shapes whose workspace exceeds the fixed array fail with LL_ERR_WORKSPACE before
    anything is enqueued (no GPU needed: the check is on the host)."""
    import structured_mask_linear_gb300 as sml
    from structured_mask_linear_gb300 import _build

    _build.build()
    L = sml.lib()
    s = sml.make_shape(4, 8192, 48, 2, 128, 64, 64, 14, sml.LL_BF16)
    assert L.loglinear_fwd_workspace_bytes(ctypes.byref(s)) > sml.STATIC_WORKSPACE_BYTES
    fake = 0x10000
    st = L.loglinear_fwd_static_workspace(ctypes.byref(s), *([fake] * 6), None, None, 0, None)
    assert st == 5  # LL_ERR_WORKSPACE
    bad = sml.make_shape(4, 8001, 48, 2, 128, 64, 64, 14, sml.LL_BF16)  # T % chunk != 0
    st = L.loglinear_fwd_static_workspace(ctypes.byref(bad), *([fake] * 6), None, None, 0, None)
    assert st == 2  # LL_ERR_SHAPE


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [
    dict(name="small", batch=1, heads=4, T=1024),                      # tensor-core path
    dict(name="tiny"),                                                 # generic path, fp32
])
def test_static_workspace_matches_caller_workspace(cfg):
    import structured_mask_linear_gb300 as sml

    name = cfg.pop("name")
    if "T" in cfg:
        cfg["levels"] = levels_for(cfg["T"])
    w = workload(name, **cfg)
    dev = "cuda:0"
    shape = sml.make_shape(w.batch, w.T, w.heads, w.heads_per_group, w.d_k, w.d_v, w.chunk,
                           w.levels, w.dtype)
    assert 0 < sml.loglinear_fwd_workspace_bytes(shape) <= sml.STATIC_WORKSPACE_BYTES
    for seed in (1, 2):  # two calls in a row: the array keeps the first call's contents
        x = make_inputs(w, dev, seed=seed)
        ref = sml.loglinear_fwd(x.q, x.k, x.v, x.a, x.lam, chunk=w.chunk)
        got = sml.loglinear_fwd_static_workspace(x.q, x.k, x.v, x.a, x.lam, chunk=w.chunk)
        torch.cuda.synchronize()
        assert sml.loglinear_check_status() == 0
        assert_parity(got.double().cpu().numpy(), ref.double().cpu().numpy(),
                      f"{name} call {seed}", got.dtype)
