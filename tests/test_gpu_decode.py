"""GPU parity of the decode step (from the forward's state export) against the oracle's
recurrent form, step by step."""
import numpy as np
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


def _prefix_and_steps(sml, x, T0, steps, chunk, L):
    B, _, H, dv = x.v.shape
    dk = x.q.shape[3]
    dev = [t.to(DEV) for t in (x.q, x.k, x.v, x.a, x.lam)]
    q, k, v, a, lam = dev
    st = torch.full((B, H, L, dk, dv), float("nan"), device=DEV)
    lsc = torch.full((B, H, L), float("nan"), device=DEV)
    pre = [t[:, :T0].contiguous() for t in dev]
    sml.loglinear_fwd(*pre, chunk=chunk, states_out=st, state_logscale_out=lsc, state_levels=L)
    outs = []
    for t in range(T0, T0 + steps):
        outs.append(sml.loglinear_decode_step(t, q[:, t].contiguous(), k[:, t].contiguous(),
                                              v[:, t].contiguous(), a[:, t].contiguous(),
                                              lam[:, t].contiguous(), st, lsc))
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    return torch.stack(outs, 1), st, lsc


@pytest.mark.parametrize("cfg", [
    dict(dtype=torch.float32, d_k=32, d_v=16, chunk=16, T0=64, steps=200),
    dict(dtype=torch.bfloat16, d_k=128, d_v=64, chunk=64, T0=256, steps=300),
    dict(dtype=torch.bfloat16, d_k=64, d_v=32, chunk=64, T0=64 * 5, steps=130),
    dict(dtype=torch.bfloat16, d_k=128, d_v=64, chunk=64, T0=64 * 5, steps=100),  # export with a 64-token last tile
])
def test_decode_matches_recurrent_form(sml, cfg):
    T0, steps = cfg["T0"], cfg["steps"]
    T = T0 + steps
    L = T.bit_length() + 1
    w = workload("small", batch=2, heads=4, T=T, levels=L, d_k=cfg["d_k"], d_v=cfg["d_v"],
                 dtype=cfg["dtype"])
    x = make_inputs(w, "cpu", seed=21)
    o, st, lsc = _prefix_and_steps(sml, x, T0, steps, cfg["chunk"], L)
    ref_o, ref_st = oracle.form_r(*(to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam)),
                                  export_levels=L)
    for i in range(steps):
        assert_parity(o[:, i].double().cpu().numpy(), ref_o[:, T0 + i], f"step {T0 + i}", o.dtype)
    # final states: exp(logscale) * states on the live levels of position T
    got = (torch.exp(lsc)[..., None, None] * st).double().cpu().numpy()
    for lvl in range(1, L):
        if (T >> (lvl - 1)) & 1:
            assert_parity(got[:, :, lvl], ref_st[:, :, lvl], f"state level {lvl}", "f32")


def test_decode_workload_sampled(sml):
    """The decode workload: B=64, H=48, prefix 32768 from the forward, 1024 steps; a few
    (b, h) streams checked at every step against the oracle's recurrent form."""
    w = workload("decode")
    x = make_inputs(w, DEV, seed=0)
    T0, steps, L = w.T, w.decode_steps, w.levels
    o, st, lsc = _prefix_and_steps(sml, x, T0, steps, w.chunk, L)
    assert torch.isfinite(o).all()
    r = np.random.default_rng(0)
    for _ in range(2):
        b, h = int(r.integers(w.batch)), int(r.integers(w.heads))
        g = h // w.heads_per_group
        T = T0 + steps
        ref_o, ref_st = oracle.form_r_head(
            to_numpy64(x.q[b, :, g]), to_numpy64(x.k[b, :, g]), to_numpy64(x.v[b, :, h]),
            to_numpy64(x.a[b, :, h]), to_numpy64(x.lam[b, :, h]), [T], levels=L)
        assert_parity(o[b, :, h].double().cpu().numpy(), ref_o[T0:], f"b={b} h={h}", o.dtype)
        got = (torch.exp(lsc[b, h])[:, None, None] * st[b, h]).double().cpu().numpy()
        for lvl in range(1, L):
            if (T >> (lvl - 1)) & 1:
                assert_parity(got[lvl], ref_st[0, lvl], f"b={b} h={h} level {lvl}", "f32")
