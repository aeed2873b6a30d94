"""GPU parity of the two comparators against the fp64 CPU oracle, through the C ABI.

* loglinear_fwd_naive: the same output as loglinear_fwd with one output pass per level
  (no level fusion), so it must match the oracle under the same bar.
* ssd_fwd: the lambda-constant special case (Mamba-2 SSD), so it must match the oracle
  run with lambda = 1 at every level; the oracle's lambda = 1 case is pinned to the
  textbook SSD recurrence in the CPU tests.
Tile counts include odd ones (ragged Fenwick trees and a one-tile sequence), and slow
decay keeps every level numerically live.
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


def _dev(x):
    return [t.to(DEV) for t in (x.q, x.k, x.v, x.a, x.lam)]


def _np(x, lam=None):
    return tuple(to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam if lam is None else lam))


def _inputs(T, decay, seed, heads=4):
    w = workload("small", batch=1, heads=heads, T=T, levels=levels_for(T), decay=decay)
    return w, make_inputs(w, "cpu", seed=seed)


@pytest.mark.parametrize("T,decay", [(1024, "iid"), (128, "iid"), (384, "slow"), (640, "slow"),
                                     (2048, "ones")])
def test_naive_per_level_matches_oracle(sml, T, decay):
    w, x = _inputs(T, decay, seed=21)
    o = sml.loglinear_fwd_naive(*_dev(x), chunk=w.chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    assert_parity(o.double().cpu().numpy(), oracle.form_q(*_np(x)), f"naive T={T}/{decay}", o.dtype)


def test_naive_per_level_agrees_with_fused(sml):
    """Same inputs, both paths: the fused and the per-level sums differ only by rounding."""
    w, x = _inputs(2048, "slow", seed=22, heads=8)
    d = _dev(x)
    o1 = sml.loglinear_fwd(*d, chunk=w.chunk)
    o2 = sml.loglinear_fwd_naive(*d, chunk=w.chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    assert_parity(o2.double().cpu().numpy(), o1.double().cpu().numpy(), "naive vs fused", o2.dtype)


@pytest.mark.parametrize("T,decay", [(1024, "iid"), (128, "iid"), (384, "slow"), (640, "slow"),
                                     (2048, "mamba2"), (2048, "ones")])
def test_ssd_matches_oracle_with_lambda_one(sml, T, decay):
    w, x = _inputs(T, decay, seed=23)
    q, k, v, a, _ = _dev(x)
    o = sml.ssd_fwd(q, k, v, a, chunk=w.chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    ref = oracle.form_q(*_np(x, lam=torch.ones_like(x.lam)))
    assert_parity(o.double().cpu().numpy(), ref, f"ssd T={T}/{decay}", o.dtype)
