"""GPU parity of the far Fenwick levels at the sequence lengths the product runs.

The decays of the benchmark workloads drive every bucket more than a few hundred tokens
back below fp32's range, so the full-size tests there check the far levels against zero
only.  Here the far levels carry real values at T = 32768 and T = 131072 (tile levels
5..10, token levels 13..17), on the tensor-core path (bf16, d_k = 128, d_v = 64):

* a power-of-two probe whose every output element is one exact power of two, compared
  with ``==`` (the level map and the node selection of every inter-tile level);
* lambda one-hot on each token level j >= 8 in turn, with a = 1 (every node's whole
  content counts) and with the slow decay (the decay of the nearer buckets counts),
  compared element by element at sampled queries whose bit j-1 is set;
* every level at once (iid lambda, slow decay) at T = 131072;
* the state export at T = 32768 (one live level-16 bucket holding the whole prefix) and
  256 decode steps from it, every output and the final states against the oracle's
  recurrent form;
* the backward and the Gated DeltaNet forward at T = 8192 with the slow decay.

Sources: the bucket levels of the log-linear attention write-up
(https://www.yoousoft.com/industry/3746.html, section 特殊结构：树划分, Fig. 2) and its
chunkwise algorithm's inter-chunk levels (section 高效训练算法, Algorithm 1).
"""
import types

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


def _fwd(sml, q, k, v, a, lam, **kw):
    o = sml.loglinear_fwd(q.to(DEV), k.to(DEV), v.to(DEV), a.to(DEV), lam.to(DEV), chunk=64, **kw)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    return o


def _points(x, ts, b=0, h=0, hpg=2, v=None):
    """Oracle outputs of head h at the query positions ts (fp64)."""
    g = h // hpg
    tm = int(max(ts)) + 1
    vv = x.v if v is None else v
    return oracle.form_q_points(to_numpy64(x.q[b, :tm, g]), to_numpy64(x.k[b, :tm, g]),
                                to_numpy64(vv[b, :tm, h]), to_numpy64(x.a[b, :tm, h]),
                                to_numpy64(x.lam[b, torch.as_tensor(ts), h]), ts)


def _level_positions(T, j, rng, n_rand=24, n_near=12):
    """Queries t < T whose bucket of token level j exists (bit j-1 of t set): random ones,
    ones just past the bucket's end (small low bits: the bucket is near), tile edges."""
    bit = 1 << (j - 1)
    hi = rng.integers(0, T, size=n_rand + n_near) & ~(2 * bit - 1)
    low_rand = rng.integers(0, bit, size=n_rand)
    low_near = rng.integers(0, min(bit, 300), size=n_near)
    ts = set(int(t) for t in (hi[:n_rand] | bit | low_rand))
    ts |= set(int(t) for t in (hi[n_rand:] | bit | low_near))
    ts |= {bit, bit + 127, bit + 128, (T - 1) | bit}
    return np.array(sorted(t for t in ts if t < T))


# --- power-of-two probe ------------------------------------------------------------------

@pytest.mark.parametrize("T", [32768, 131072])
@pytest.mark.parametrize("where", ["first", "second_tile", "last_tile", "last"])
def test_far_levels_bitexact(sml, T, where):
    """a = 1, q = k = e0, lambda^l = 2^l, and v_s = e_j only at s = j*(T/64) + offset:
    o_t[j] = 2^l(t, s_j) exactly for every earlier s_j, and 0 elsewhere.  The offsets move
    the marked keys to other tiles of each block and to other rows inside a tile."""
    H, dk, dv = 2, 128, 64
    L = levels_for(T)
    blk = T // dv
    offset = {"first": 0, "second_tile": 128 + 77, "last_tile": blk - 128, "last": blk - 1}[where]
    q = torch.zeros(1, T, 1, dk)
    q[..., 0] = 1.0
    v = torch.zeros(1, T, H, dv)
    for j in range(dv):
        v[0, j * blk + offset, :, j] = 1.0
    lam = (2.0 ** torch.arange(L, dtype=torch.float32)).expand(1, T, H, L).contiguous()
    a = torch.ones(1, T, H)
    q, v = q.bfloat16(), v.bfloat16()
    o = _fwd(sml, q, q, v, a, lam)
    rng = np.random.default_rng(T + offset)
    ts = {0, offset, offset + 1, blk + offset - 1, blk + offset, T - 1}
    for m in range(T.bit_length() - 8):  # every tile level: tiles with bit m set
        ts |= set(int(t) for t in ((rng.integers(0, T, size=6) | (128 << m))))
    ts = np.array(sorted(t for t in ts if t < T))
    x = types.SimpleNamespace(q=q, k=q, v=v, a=a, lam=lam)
    for h in range(H):
        ref = _points(x, ts, h=h)
        got = o[0, torch.as_tensor(ts, device=DEV), h].double().cpu().numpy()
        assert np.array_equal(got, ref), f"T={T} offset={offset} h={h}"


# --- one level at a time -----------------------------------------------------------------

@pytest.mark.parametrize("decay", ["ones", "slow"])
@pytest.mark.parametrize("T", [32768, 131072])
def test_far_levels_isolated(sml, T, decay):
    """lambda^l = [l == j] for every inter-tile token level j in turn (j = 8 .. L-1):
    the output is the level-j bucket's term alone, compared with the oracle at queries
    that have that bucket."""
    L = levels_for(T)
    w = workload("small", batch=1, heads=2, heads_per_group=2, T=T, levels=L, decay=decay)
    x = make_inputs(w, "cpu", seed=40 + L)
    rng = np.random.default_rng(T)
    for j in range(8, L):
        lam = torch.zeros_like(x.lam)
        lam[..., j] = 1.0
        x.lam = lam
        o = _fwd(sml, x.q, x.k, x.v, x.a, lam)
        ts = _level_positions(T, j, rng)
        for h in range(2):
            ref = _points(x, ts, h=h)
            assert np.linalg.norm(ref) > 0, f"level {j}: no live contribution at the sampled queries"
            got = o[0, torch.as_tensor(ts, device=DEV), h].double().cpu().numpy()
            assert_parity(got, ref, f"T={T} {decay} level {j} h={h}", o.dtype)


def test_long_all_levels_slow_decay(sml):
    """Every level at once (iid lambda, slow decay) at T = 131072: sampled queries with
    each tile level's bit set, tile edges and random ones."""
    T = 131072
    L = levels_for(T)
    w = workload("small", batch=1, heads=2, heads_per_group=2, T=T, levels=L, decay="slow")
    x = make_inputs(w, "cpu", seed=77)
    o = _fwd(sml, x.q, x.k, x.v, x.a, x.lam)
    rng = np.random.default_rng(5)
    ts = set()
    for j in range(8, L):
        ts |= set(int(t) for t in _level_positions(T, j, rng, n_rand=6, n_near=6))
    ts |= {0, 1, 127, 128, T // 2 - 1, T // 2, T - 129, T - 128, T - 1}
    ts = np.array(sorted(ts))
    for h in range(2):
        ref = _points(x, ts, h=h)
        got = o[0, torch.as_tensor(ts, device=DEV), h].double().cpu().numpy()
        assert_parity(got, ref, f"long slow h={h}", o.dtype)


# --- export at T = 32768 and decode from it ------------------------------------------------

@pytest.mark.parametrize("decay", ["slow", "ones"])
def test_export_32k_and_decode(sml, decay):
    """The forward's export at T0 = 32768 is one live bucket (level 16) holding the whole
    prefix; 256 decode steps from it (B = 1, two heads) are compared at every step with the
    oracle's recurrent form, and the exported and final states level by level."""
    T0, steps = 32768, 256
    T = T0 + steps
    L = T.bit_length() + 1  # 17
    w = workload("small", batch=1, heads=2, heads_per_group=2, T=T, levels=L, decay=decay)
    x = make_inputs(w, "cpu", seed=91)
    q, k, v, a, lam = (t.to(DEV) for t in (x.q, x.k, x.v, x.a, x.lam))
    st = torch.full((1, 2, L, 128, 64), float("nan"), device=DEV)
    lsc = torch.full((1, 2, L), float("nan"), device=DEV)
    pre = [t[:, :T0].contiguous() for t in (q, k, v, a, lam)]
    sml.loglinear_fwd(*pre, chunk=64, states_out=st, state_logscale_out=lsc, state_levels=L)
    torch.cuda.synchronize()
    exported = (torch.exp(lsc)[..., None, None] * st).double().cpu().numpy()
    outs = []
    for t in range(T0, T):
        outs.append(sml.loglinear_decode_step(t, q[:, t].contiguous(), k[:, t].contiguous(),
                                              v[:, t].contiguous(), a[:, t].contiguous(),
                                              lam[:, t].contiguous(), st, lsc))
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    o = torch.stack(outs, 1)
    final = (torch.exp(lsc)[..., None, None] * st).double().cpu().numpy()
    for h in range(2):
        ref_o, ref_st = oracle.form_r_head(
            to_numpy64(x.q[0, :, 0]), to_numpy64(x.k[0, :, 0]), to_numpy64(x.v[0, :, h]),
            to_numpy64(x.a[0, :, h]), to_numpy64(x.lam[0, :, h]), [T0, T], levels=L)
        assert_parity(exported[0, h, 16], ref_st[0, 16], f"{decay} h={h} export level 16", "f32")
        for i in range(steps):
            assert_parity(o[0, i, h].double().cpu().numpy(), ref_o[T0 + i],
                          f"{decay} h={h} step {T0 + i}", o.dtype)
        for lvl in range(1, L):
            if (T >> (lvl - 1)) & 1:  # levels 16 and 9 at T = 33024
                assert_parity(final[0, h, lvl], ref_st[1, lvl], f"{decay} h={h} final level {lvl}", "f32")


# --- next rows at T = 8192 with the slow decay --------------------------------------------------

def test_backward_slow_decay_8k(sml):
    """The backward at T = 8192 (tile levels 0..5, token levels up to 13) with the slow
    decay, so that the far levels' duals and gradients carry real values."""
    T = 8192
    w = workload("small", batch=1, heads=2, heads_per_group=2, T=T, levels=levels_for(T), decay="slow")
    x = make_inputs(w, "cpu", seed=61)
    gen = torch.Generator().manual_seed(62)
    dO = torch.randn(x.v.shape, generator=gen).to(x.v.dtype)
    got = sml.loglinear_bwd(*(t.to(DEV) for t in (x.q, x.k, x.v, x.a, x.lam, dO)), chunk=64)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    ref = oracle.backward(*(to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam, dO)))
    for name, g, r in zip(("dq", "dk", "dv", "dloga", "dlam"), got, ref):
        dtype = g.dtype if name in ("dq", "dk", "dv") else torch.float32
        assert_parity(g.double().cpu().numpy(), r, f"bwd slow 8k {name}", dtype)


def test_gdn_slow_decay_8k(sml):
    """Log-linear Gated DeltaNet at T = 8192 with the slow decay (keys L2-normalised,
    beta = sigmoid(z)), sampled queries at every tile level."""
    T = 8192
    w = workload("small", batch=1, heads=2, heads_per_group=2, T=T, levels=levels_for(T), decay="slow")
    x = make_inputs(w, "cpu", seed=63)
    kf = x.k.float()
    x.k = (kf / kf.norm(dim=-1, keepdim=True)).to(x.k.dtype)
    beta = torch.sigmoid(torch.randn(x.a.shape, generator=torch.Generator().manual_seed(64)))
    o = sml.loglinear_gdn_fwd(*(t.to(DEV) for t in (x.q, x.k, x.v, x.a, beta, x.lam)), chunk=64)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    u = torch.from_numpy(oracle.gdn_values(*(to_numpy64(t) for t in (x.k, x.v, x.a, beta))))
    rng = np.random.default_rng(9)
    ts = set()
    for j in range(8, levels_for(T)):
        ts |= set(int(t) for t in _level_positions(T, j, rng, n_rand=8, n_near=6))
    ts |= {0, 1, 127, 128, T - 1}
    ts = np.array(sorted(ts))
    for h in range(2):
        ref = _points(x, ts, h=h, v=u)
        got = o[0, torch.as_tensor(ts, device=DEV), h].double().cpu().numpy()
        assert_parity(got, ref, f"gdn slow 8k h={h}", o.dtype)
