"""GPU parity of the log-linear Gated DeltaNet forward (loglinear_gdn_fwd) against the
oracle's gdn_forward (the masked form over the gated delta rule's transformed values,
pinned to the dense matrix recurrence in the CPU tests), through the C ABI.

Keys are L2-normalised per token, as the model does, and beta = sigmoid(z).  Cases: the
fp32 generic path, the bf16 tensor-core path, a length that is not a multiple of the
tile, chunk 16, slow and mamba2 decays, more than one batch element on the tensor-core
path (the last element's state pass and forward run on a second stream), and more
chunks than SMs (the chunk kernel's persistent CTAs take several each); beta = 0 must
give exactly zero.
"""
import pytest
import torch

from oracle import oracle
from parity_util import assert_parity
from structured_mask_linear_gb300.inputs import levels_for, make_inputs, to_numpy64, workload

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def sml():
    import structured_mask_linear_gb300 as m

    m.lib()
    return m


def _inputs(w, seed):
    x = make_inputs(w, "cpu", seed=seed)
    k = x.k.float()
    x.k = (k / k.norm(dim=-1, keepdim=True)).to(x.k.dtype)
    gen = torch.Generator().manual_seed(seed + 1000)
    beta = torch.sigmoid(torch.randn(x.a.shape, generator=gen))
    return x, beta


def _run(sml, w, x, beta, chunk):
    dev = [t.to(DEV) for t in (x.q, x.k, x.v, x.a, beta, x.lam)]
    o = sml.loglinear_gdn_fwd(*dev, chunk=chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    return o


@pytest.mark.parametrize("name,kw,chunk", [
    ("tiny", {}, 16),
    ("small", dict(batch=1, heads=4, T=1024), 64),            # tensor-core forward
    ("small", dict(batch=1, heads=4, T=64 * 37), 64),         # CUDA-core values, 64-token last tile
    ("small", dict(batch=1, heads=2, T=512), 16),
    ("small", dict(batch=1, heads=4, T=1024, decay="slow"), 64),
    ("small", dict(batch=1, heads=4, T=1024, decay="mamba2"), 64),
    ("small", dict(batch=3, heads=4, T=1024), 64),            # batch split over two streams
    ("small", dict(batch=2, heads=16, T=1024), 64),           # 256 chunks: persistent CTAs take two
])
def test_gdn_matches_oracle(sml, name, kw, chunk):
    if "T" in kw:
        kw = dict(kw, levels=levels_for(kw["T"]))
    w = workload(name, **kw)
    x, beta = _inputs(w, seed=51)
    o = _run(sml, w, x, beta, chunk)
    ref = oracle.gdn_forward(*(to_numpy64(t) for t in (x.q, x.k, x.v, x.a, beta, x.lam)))
    assert_parity(o.double().cpu().numpy(), ref, f"gdn {name} {kw}", o.dtype)


def test_gdn_zero_beta_is_zero(sml):
    w = workload("small", batch=1, heads=2, T=512, levels=levels_for(512))
    x, beta = _inputs(w, seed=52)
    o = _run(sml, w, x, torch.zeros_like(beta), 64)
    assert float(o.abs().max()) == 0.0


def test_pages_workload_sampled(sml):
    """The Gated DeltaNet forward at the benchmark's size (pages workload: B=4, H=48,
    T=8192, chunk 64): the oracle's delta-rule values of two heads over the whole
    sequence, then sampled outputs (edges of tiles, chunks and the sequence, plus random
    positions) through the oracle's point form of the masked sum."""
    import numpy as np

    w = workload("pages")
    x = make_inputs(w, DEV, seed=0)
    k = x.k.float()
    kn = (k / k.norm(dim=-1, keepdim=True)).to(x.k.dtype)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(6)
    beta = torch.sigmoid(torch.randn(x.a.shape, generator=gen, device=DEV))
    o = sml.loglinear_gdn_fwd(x.q, kn, x.v, x.a, beta, x.lam, chunk=w.chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    assert torch.isfinite(o).all()
    r = np.random.default_rng(8)
    T = w.T
    for _ in range(2):
        b, h = int(r.integers(w.batch)), int(r.integers(w.heads))
        g = h // w.heads_per_group
        u = oracle.gdn_values(to_numpy64(kn[b:b + 1, :, g:g + 1]), to_numpy64(x.v[b:b + 1, :, h:h + 1]),
                              to_numpy64(x.a[b:b + 1, :, h:h + 1]), to_numpy64(beta[b:b + 1, :, h:h + 1]))
        ts = {0, 1, 31, 32, 63, 64, 127, 128, T // 2 - 1, T // 2, T - 65, T - 64, T - 1}
        ts = np.array(sorted(ts | set(int(t) for t in r.integers(0, T, size=60))))
        tm = int(ts.max()) + 1
        ref = oracle.form_q_points(to_numpy64(x.q[b, :tm, g]), to_numpy64(kn[b, :tm, g]), u[0, :tm, 0],
                                   to_numpy64(x.a[b, :tm, h]), to_numpy64(x.lam[b, torch.as_tensor(ts, device=DEV), h]),
                                   ts)
        got = o[b, torch.as_tensor(ts, device=DEV), h].double().cpu().numpy()
        assert_parity(got, ref, f"gdn pages b={b} h={h}", o.dtype)
