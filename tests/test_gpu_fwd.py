"""GPU parity of loglinear_fwd against the fp64 CPU oracle (called through the C ABI)."""
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


def _run(sml, x, chunk, **kw):
    dev = [t.to(DEV) for t in (x.q, x.k, x.v, x.a, x.lam)]
    o = sml.loglinear_fwd(*dev, chunk=chunk, **kw)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    return o


def _np(x):
    return tuple(to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam))


@pytest.mark.parametrize("name,T,path", [("small", 2048, 2), ("pages", 8192, 2), ("long", 131072, 2),
                                         ("small", 64 * 37, 2), ("small", 64, 2), ("tiny", 256, 1)])
def test_path_selection(sml, name, T, path):
    """bf16 with d_k = 128, d_v = 64 and T % 64 == 0 runs the tensor-core kernels (a last
    tile of 64 tokens when T % 128 == 64); fp32 runs the CUDA-core ones."""
    w = workload(name, T=T, levels=levels_for(T))
    shape = sml.make_shape(w.batch, T, w.heads, w.heads_per_group, w.d_k, w.d_v, w.chunk,
                           w.levels, w.dtype)
    assert sml.loglinear_fwd_path(shape) == path


def test_tiny_workload_full(sml):
    w = workload("tiny")
    x = make_inputs(w, "cpu", seed=0)
    o = _run(sml, x, w.chunk)
    assert_parity(o.double().cpu().numpy(), oracle.form_q(*_np(x)), "tiny", o.dtype)


def test_small_workload_full(sml):
    w = workload("small")
    x = make_inputs(w, "cpu", seed=0)
    o = _run(sml, x, w.chunk)
    assert_parity(o.double().cpu().numpy(), oracle.form_q(*_np(x)), "small", o.dtype)


@pytest.mark.parametrize("T", [64, 128, 192, 64 * 37])
def test_ragged_chunk_counts(sml, T):
    """Chunk counts that are not powers of two (ragged Fenwick tree), T = C and T = 2C."""
    w = workload("small", batch=1, heads=4, T=T, levels=levels_for(T))
    x = make_inputs(w, "cpu", seed=3)
    o = _run(sml, x, 64)
    assert_parity(o.double().cpu().numpy(), oracle.form_q(*_np(x)), f"T={T}", o.dtype)


@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
def test_chunk_invariance(sml, chunk):
    """The output does not depend on the chunk length (exact re-association)."""
    w = workload("small", batch=1, heads=2, d_k=64, d_v=32, T=1024, levels=levels_for(1024))
    x = make_inputs(w, "cpu", seed=5)
    o = _run(sml, x, chunk)
    assert_parity(o.double().cpu().numpy(), oracle.form_q(*_np(x)), f"chunk={chunk}", o.dtype)


@pytest.mark.parametrize("decay", ["ones", "slow"])
@pytest.mark.parametrize("name", ["tiny", "small"])
def test_slow_decay_keeps_far_levels_live(sml, name, decay):
    w = workload(name, decay=decay)
    if name == "small":
        w = workload(name, decay=decay, batch=1, heads=4)
    x = make_inputs(w, "cpu", seed=11)
    o = _run(sml, x, w.chunk)
    assert_parity(o.double().cpu().numpy(), oracle.form_q(*_np(x)), f"{name}/{decay}", o.dtype)


@pytest.mark.parametrize("dtype,dk,dv", [(torch.float32, 64, 32), (torch.bfloat16, 64, 32),
                                         (torch.bfloat16, 128, 64)])
def test_level_isolation(sml, dtype, dk, dv):
    """lambda^l = [l == j] for each level j, slow decay: each level checked alone (the
    bf16 128/64 case runs the tensor-core path)."""
    T = 1024
    L = levels_for(T)
    w = workload("small", batch=1, heads=2, heads_per_group=2, T=T, levels=L, decay="slow",
                 dtype=dtype, d_k=dk, d_v=dv)
    x = make_inputs(w, "cpu", seed=2)
    for j in range(L):
        lam = torch.zeros_like(x.lam)
        lam[..., j] = 1.0
        x.lam = lam
        o = _run(sml, x, 64)
        ref = oracle.form_q(*_np(x))
        if np.linalg.norm(ref) == 0:
            assert float(o.abs().max()) == 0.0
        else:
            assert_parity(o.double().cpu().numpy(), ref, f"level {j}", o.dtype)


def _probe_inputs(T, H, hpg, dk, dv, L, dtype, v):
    G = H // hpg
    q = torch.zeros(1, T, G, dk)
    q[..., 0] = 1.0
    lam = (2.0 ** torch.arange(L, dtype=torch.float32)).expand(1, T, H, L).contiguous()
    a = torch.ones(1, T, H)
    return q.to(dtype), q.clone().to(dtype), v.to(dtype), a, lam


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("chunk", [16, 64, 128])
def test_bitexact_level_map_intra(sml, dtype, chunk):
    """a = 1, q = k = e0, lambda^l = 2^l, v_s = e_(s mod d_v), T = C: o_t[s] = 2^l(t,s)."""
    T, dv, L = chunk, 64, levels_for(chunk)
    v = torch.zeros(1, T, 2, dv)
    for s in range(T):
        v[0, s, :, s % dv] = 1.0
    q, k, v, a, lam = _probe_inputs(T, 2, 2, 128, dv, L, dtype, v)
    o = sml.loglinear_fwd(q.to(DEV), k.to(DEV), v.to(DEV), a.to(DEV), lam.to(DEV), chunk=chunk)
    ref = oracle.form_q(*(to_numpy64(t) for t in (q, k, v, a, lam)))
    assert np.array_equal(o.double().cpu().numpy(), ref)


@pytest.mark.parametrize("T", [4096, 4032])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_bitexact_level_map_inter(sml, dtype, T):
    """C = 64: v is e_j only at the first token of chunk j, so o_t[j] = 2^l(t, jC) exactly
    for every earlier chunk, which checks every chunk-level bucket (T = 4032: the last
    128-token tile of the bf16 tensor-core path holds 64 tokens)."""
    C, dv = 64, 64
    L = levels_for(T)
    v = torch.zeros(1, T, 2, dv)
    for j in range(T // C):
        v[0, j * C, :, j] = 1.0
    q, k, v, a, lam = _probe_inputs(T, 2, 2, 128, dv, L, dtype, v)
    o = sml.loglinear_fwd(q.to(DEV), k.to(DEV), v.to(DEV), a.to(DEV), lam.to(DEV), chunk=C)
    ref = oracle.form_q(*(to_numpy64(t) for t in (q, k, v, a, lam)))
    assert np.array_equal(o.double().cpu().numpy(), ref)


def test_bitexact_sum_fp32(sml):
    """fp32, T = 4096, v_s = e_(s mod 64): each output is an integer sum of powers of two
    below 2^24, exact in fp32 whatever the summation order."""
    T, C, dv = 4096, 64, 64
    L = levels_for(T)
    v = torch.zeros(1, T, 1, dv)
    for s in range(T):
        v[0, s, 0, s % dv] = 1.0
    q, k, v, a, lam = _probe_inputs(T, 1, 1, 64, dv, L, torch.float32, v)
    o = sml.loglinear_fwd(q.to(DEV), k.to(DEV), v.to(DEV), a.to(DEV), lam.to(DEV), chunk=C)
    ref = oracle.form_q(*(to_numpy64(t) for t in (q, k, v, a, lam)))
    assert np.array_equal(o.double().cpu().numpy(), ref)


@pytest.mark.parametrize("decay", ["iid", "slow"])
@pytest.mark.parametrize("T", [2048, 64 * 37])
def test_state_export(sml, T, decay):
    """Exported bucket states at position T.  With the iid decay the far levels decay
    below the fp32 range, so the live levels are compared jointly (relative to the
    whole export); with slow decay every live level is compared on its own.  Slots of
    levels that are not live hold unspecified values and are not compared."""
    w = workload("small", batch=1, heads=4, T=T, levels=levels_for(T), decay=decay)
    x = make_inputs(w, "cpu", seed=9)
    SL = T.bit_length() + 1
    st = torch.full((1, 4, SL, 128, 64), float("nan"), device=DEV)
    lsc = torch.full((1, 4, SL), float("nan"), device=DEV)
    o = _run(sml, x, 64, states_out=st, state_logscale_out=lsc, state_levels=SL)
    ref_o, ref_st = oracle.form_r(*_np(x), export_levels=SL)
    assert_parity(o.double().cpu().numpy(), ref_o, "o", o.dtype)
    assert torch.all(lsc == 0)
    got = st.double().cpu().numpy()
    live = [lvl for lvl in range(SL) if lvl >= 1 and (T >> (lvl - 1)) & 1]
    for lvl in live:
        if decay == "slow":
            assert_parity(got[:, :, lvl], ref_st[:, :, lvl], f"state level {lvl}", "f32")
    assert_parity(got[:, :, live], ref_st[:, :, live], "live levels", "f32")


def test_many_heads_ungrouped(sml):
    w = workload("small", batch=3, heads=6, heads_per_group=1, T=256, d_k=32, d_v=16,
                 levels=levels_for(256), dtype=torch.float32)
    x = make_inputs(w, "cpu", seed=4)
    o = _run(sml, x, 32)
    assert_parity(o.double().cpu().numpy(), oracle.form_q(*_np(x)), "ungrouped", o.dtype)


def test_timeout_selftest_reports_and_recovers(sml):
    sml.loglinear_selftest_wait_timeout(1000)
    assert sml.loglinear_check_status() == 7  # LL_ERR_TIMEOUT
    assert sml.loglinear_check_status() == 0  # cleared
    w = workload("tiny")
    x = make_inputs(w, "cpu", seed=0)
    o = _run(sml, x, w.chunk)  # the context is still usable
    assert_parity(o.double().cpu().numpy(), oracle.form_q(*_np(x)), "after timeout", o.dtype)


# --- full-size workloads, sampled outputs ------------------------------------

def _sampled_check(sml, name, n_pairs, n_t, seed=0):
    w = workload(name)
    x = make_inputs(w, DEV, seed=seed)
    o = sml.loglinear_fwd(x.q, x.k, x.v, x.a, x.lam, chunk=w.chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    assert torch.isfinite(o).all()
    r = np.random.default_rng(seed)
    T = w.T
    for p in range(n_pairs):
        b = int(r.integers(w.batch))
        h = int(r.integers(w.heads))
        g = h // w.heads_per_group
        ts = {0, 1, 63, 64, 127, 128, T // 2 - 1, T // 2, T - 65, T - 64, T - 1}
        ts |= set(int(t) for t in r.integers(0, T, size=n_t))
        ts = np.array(sorted(ts))
        tm = int(ts.max()) + 1
        ref = oracle.form_q_points(to_numpy64(x.q[b, :tm, g]), to_numpy64(x.k[b, :tm, g]),
                                   to_numpy64(x.v[b, :tm, h]), to_numpy64(x.a[b, :tm, h]),
                                   to_numpy64(x.lam[b, torch.as_tensor(ts, device=DEV), h]), ts)
        got = o[b, torch.as_tensor(ts, device=DEV), h].double().cpu().numpy()
        assert_parity(got, ref, f"{name} b={b} h={h}", o.dtype)


def test_pages_workload_sampled(sml):
    _sampled_check(sml, "pages", n_pairs=4, n_t=100)


def test_long_workload_sampled(sml):
    _sampled_check(sml, "long", n_pairs=2, n_t=40)
