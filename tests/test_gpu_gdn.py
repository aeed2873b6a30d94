"""GPU parity of the log-linear Gated DeltaNet forward (loglinear_gdn_fwd) against the
oracle's gdn_forward (the masked form over the gated delta rule's transformed values,
pinned to the dense matrix recurrence in the CPU tests), through the C ABI.

Keys are L2-normalised per token, as the model does, and beta = sigmoid(z).  Cases: the
fp32 generic path, the bf16 tensor-core path, a length that is not a multiple of the
tile, chunk 16, slow and mamba2 decays; beta = 0 must give exactly zero.
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
    ("small", dict(batch=1, heads=4, T=64 * 37), 64),         # generic forward
    ("small", dict(batch=1, heads=2, T=512), 16),
    ("small", dict(batch=1, heads=4, T=1024, decay="slow"), 64),
    ("small", dict(batch=1, heads=4, T=1024, decay="mamba2"), 64),
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
