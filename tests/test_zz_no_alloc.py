"""The forward entry point that allocates nothing (loglinear_fwd_static_workspace).

Some callers may not allocate device memory while they run: a plugin whose host
application owns every device allocation, or code that shares the CUDA context with a
caching allocator it must not disturb.  For them the library keeps a fixed 32 MiB device
array as the forward's workspace.  These tests call that entry point through the C ABI
and require the same output as loglinear_fwd with a caller-provided workspace: the two
run the same kernels, which have no atomics in the forward, so the results must be
bitwise equal.  One call is also compared with the oracle.

Because every call shares the array and finds the previous call's data in it, the tests
first fill most of the array with a larger problem and then check smaller ones: a kernel
reading a word the current call did not write would see the larger call's data.  The
state export through this entry point is compared with the caller-workspace export.

This file is collected last on purpose, so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity_util import assert_parity
from structured_mask_linear_gb300.inputs import levels_for, make_inputs, to_numpy64, workload


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


def _shape_of(sml, w):
    return sml.make_shape(w.batch, w.T, w.heads, w.heads_per_group, w.d_k, w.d_v, w.chunk,
                          w.levels, w.dtype)


def _large_filler(sml):
    """The tensor-core shape (T = 8192) with the most heads whose workspace fits."""
    best = None
    for heads in range(2, 64, 2):
        w = workload("small", batch=1, heads=heads, T=8192, levels=levels_for(8192))
        if sml.loglinear_fwd_workspace_bytes(_shape_of(sml, w)) > sml.STATIC_WORKSPACE_BYTES:
            break
        best = w
    return best


def _both(sml, w, seed, export=False):
    x = make_inputs(w, "cuda:0", seed=seed)
    kw = {}
    kw_ref = {}
    if export:
        SL = w.T.bit_length() + 1
        mk = lambda: (torch.full((w.batch, w.heads, SL, w.d_k, w.d_v), float("nan"), device="cuda:0"),
                      torch.full((w.batch, w.heads, SL), float("nan"), device="cuda:0"))
        st, lsc = mk()
        st_ref, lsc_ref = mk()
        kw = dict(states_out=st, state_logscale_out=lsc, state_levels=SL)
        kw_ref = dict(states_out=st_ref, state_logscale_out=lsc_ref, state_levels=SL)
    ref = sml.loglinear_fwd(x.q, x.k, x.v, x.a, x.lam, chunk=w.chunk, **kw_ref)
    got = sml.loglinear_fwd_static_workspace(x.q, x.k, x.v, x.a, x.lam, chunk=w.chunk, **kw)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    return x, got, ref, kw, kw_ref


@pytest.mark.gpu
def test_static_workspace_matches_caller_workspace():
    import structured_mask_linear_gb300 as sml
    from oracle import oracle

    filler = _large_filler(sml)
    need = sml.loglinear_fwd_workspace_bytes(_shape_of(sml, filler))
    assert need > sml.STATIC_WORKSPACE_BYTES * 3 // 4
    _, got, ref, _, _ = _both(sml, filler, seed=7)
    assert torch.equal(got, ref), "filler shape"
    cases = [dict(name="small", batch=1, heads=4, T=1024),   # tensor-core path
             dict(name="tiny")]                               # generic path, fp32
    for cfg in cases:
        cfg = dict(cfg)
        name = cfg.pop("name")
        if "T" in cfg:
            cfg["levels"] = levels_for(cfg["T"])
        w = workload(name, **cfg)
        assert 0 < sml.loglinear_fwd_workspace_bytes(_shape_of(sml, w)) <= sml.STATIC_WORKSPACE_BYTES
        for seed in (1, 2):  # two calls in a row: the array keeps the previous call's contents
            x, got, ref, _, _ = _both(sml, w, seed)
            assert torch.equal(got, ref), f"{name} call {seed}"
        ora = oracle.form_q(*(to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam)))
        assert_parity(got.double().cpu().numpy(), ora, f"{name} vs oracle", got.dtype)


@pytest.mark.gpu
def test_static_workspace_state_export():
    """states_out / state_logscale_out through the static workspace equal the export of
    loglinear_fwd on every live level (T = 1536: levels 10 and 11 live)."""
    import structured_mask_linear_gb300 as sml

    w = workload("small", batch=1, heads=4, T=1536, levels=levels_for(1536), decay="slow")
    _, got, ref, kw, kw_ref = _both(sml, w, seed=3, export=True)
    assert torch.equal(got, ref)
    assert torch.all(kw["state_logscale_out"] == 0)
    live = [l for l in range(1, kw["state_levels"]) if (w.T >> (l - 1)) & 1]
    for l in live:
        assert torch.equal(kw["states_out"][:, :, l], kw_ref["states_out"][:, :, l]), f"level {l}"
    assert np.isfinite(kw["states_out"][:, :, live].cpu().numpy()).all()
