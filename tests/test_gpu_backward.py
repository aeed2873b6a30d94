"""GPU parity of loglinear_bwd (dq, dk, dv, d(log a), dlambda of sum(dO * o)) against the
oracle's backward, which is pinned to finite differences of the forward oracle in the
CPU tests.  Called through the C ABI.

The bar is the forward's: relative L2 <= 1e-2 and max |err| <= 5e-2 RMS per gradient,
the cast of dq, dk, dv to the input dtype charged at half an ulp.  Cases: fp32 and
bf16, one, two and four heads per Q/K group, chunk counts that are not powers of two, every chunk
length, slow decay (all levels live) and a one-chunk sequence.  bf16 with d_k = 128,
d_v = 64, T % 128 == 0 and chunk >= 64 takes the tensor-core kernel for the pairs inside
128-token tiles (T = 1024 and 640 here, the decay cases too); the others the CUDA-core one.
"""
import pytest
import torch

from oracle import oracle
from parity_util import assert_parity
from structured_mask_linear_gb300.inputs import levels_for, make_inputs, to_numpy64, workload

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
NAMES = ("dq", "dk", "dv", "dloga", "dlam")


@pytest.fixture(scope="module")
def sml():
    import structured_mask_linear_gb300 as m

    m.lib()
    return m


def _check(sml, w, x, chunk, what):
    gen = torch.Generator().manual_seed(1234)
    dO = torch.randn(x.v.shape, generator=gen).to(x.v.dtype)
    dev = [t.to(DEV) for t in (x.q, x.k, x.v, x.a, x.lam, dO)]
    got = sml.loglinear_bwd(*dev, chunk=chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    ref = oracle.backward(*(to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam, dO)))
    for name, g, r in zip(NAMES, got, ref):
        dtype = g.dtype if name in ("dq", "dk", "dv") else torch.float32
        assert_parity(g.double().cpu().numpy(), r, f"{what} {name}", dtype)


def test_tiny_fp32(sml):
    w = workload("tiny")
    _check(sml, w, make_inputs(w, "cpu", seed=31), w.chunk, "tiny")


@pytest.mark.parametrize("T,chunk", [(1024, 64), (64 * 37, 64), (64, 64), (512, 16), (768, 32),
                                     (1024, 128), (640, 64)])
def test_bf16_grouped(sml, T, chunk):
    w = workload("small", batch=1, heads=4, T=T, levels=levels_for(T))
    _check(sml, w, make_inputs(w, "cpu", seed=32), chunk, f"T={T} C={chunk}")


@pytest.mark.parametrize("decay", ["slow", "ones", "mamba2"])
def test_bf16_decays(sml, decay):
    w = workload("small", batch=2, heads=2, T=1024, levels=levels_for(1024), decay=decay)
    _check(sml, w, make_inputs(w, "cpu", seed=33), 64, decay)


@pytest.mark.parametrize("hpg", [1, 4])
def test_bf16_group_sizes(sml, hpg):
    """The tensor-core path with one and four heads per Q/K group (the pages workload has
    two): dq and dk are the sums over each group's heads."""
    w = workload("small", batch=1, heads=4, heads_per_group=hpg, T=1024, levels=levels_for(1024),
                 decay="slow")
    _check(sml, w, make_inputs(w, "cpu", seed=35), 64, f"hpg={hpg}")


def test_ungrouped_small_dims(sml):
    w = workload("small", batch=1, heads=3, heads_per_group=1, T=640, levels=levels_for(640) + 1,
                 d_k=32, d_v=16, decay="slow")
    _check(sml, w, make_inputs(w, "cpu", seed=34), 32, "ungrouped")


def test_pages_workload_group_slice(sml):
    """The backward at the benchmark's size and launch configuration (pages workload:
    B=4, H=48 in 24 Q/K groups, T=8192, chunk 64): the oracle computes one Q/K group (its
    two heads) of one batch element over the whole sequence, and every gradient of that
    slice is compared (dq and dk are sums over the group's heads)."""
    import numpy as np

    w = workload("pages")
    x = make_inputs(w, DEV, seed=0)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(99)
    dO = torch.randn(x.v.shape, generator=gen, device=DEV).to(x.v.dtype)
    got = sml.loglinear_bwd(x.q, x.k, x.v, x.a, x.lam, dO, chunk=w.chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    r = np.random.default_rng(7)
    b, g = int(r.integers(w.batch)), int(r.integers(w.heads // w.heads_per_group))
    hs = slice(g * w.heads_per_group, (g + 1) * w.heads_per_group)
    gs = slice(g, g + 1)
    bs = slice(b, b + 1)
    ref = oracle.backward(to_numpy64(x.q[bs, :, gs]), to_numpy64(x.k[bs, :, gs]), to_numpy64(x.v[bs, :, hs]),
                          to_numpy64(x.a[bs, :, hs]), to_numpy64(x.lam[bs, :, hs]), to_numpy64(dO[bs, :, hs]))
    sel = (gs, gs, hs, hs, hs)
    for name, t, rr, s in zip(NAMES, got, ref, sel):
        dtype = t.dtype if name in ("dq", "dk", "dv") else torch.float32
        assert_parity(t[bs, :, s].double().cpu().numpy(), rr, f"pages b={b} g={g} {name}", dtype)
