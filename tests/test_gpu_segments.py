"""GPU parity of the sequence-segment entry points against the oracle, through the C ABI:
loglinear_segment_total, loglinear_prefix_states, loglinear_fwd_continue (on the
tensor-core and the CUDA-core paths, with and without the export at the segment's end,
in place), and the sharded forward, both as one process that runs every segment and as
two gloo ranks sharing the GPU.

The prefix memories fed to loglinear_fwd_continue come from the oracle's recurrent form
captured at T0 on the whole sequence, and the reference outputs and end memories from the
same run, so each call is checked on its own.  Slow and a = 1 decays keep the far buckets
live.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch

from oracle import oracle
from parity_util import assert_parity
from structured_mask_linear_gb300.inputs import levels_for, make_inputs, to_numpy64, workload

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sml():
    import structured_mask_linear_gb300 as m

    m.lib()
    return m


def _head_ref(x, b, h, hpg, T_end, caps, levels):
    g = h // hpg
    return oracle.form_r_head(to_numpy64(x.q[b, :T_end, g]), to_numpy64(x.k[b, :T_end, g]),
                              to_numpy64(x.v[b, :T_end, h]), to_numpy64(x.a[b, :T_end, h]),
                              to_numpy64(x.lam[b, :T_end, h]), caps, levels=levels)


CASES = [  # name, overrides, chunk, segment length T, start T0
    ("tc", dict(d_k=128, d_v=64, dtype=torch.bfloat16), 64, 1024, 3072),
    ("tc_far", dict(d_k=128, d_v=64, dtype=torch.bfloat16), 64, 512, 7680),
    ("tc_carry", dict(d_k=128, d_v=64, dtype=torch.bfloat16), 64, 1024, 1024),
    ("tc_partial", dict(d_k=128, d_v=64, dtype=torch.bfloat16), 64, 192, 768),
    ("generic", dict(d_k=32, d_v=16, dtype=torch.float32), 32, 256, 768),
    ("generic_bf16", dict(d_k=64, d_v=32, dtype=torch.bfloat16), 64, 192 * 2, 512 * 3),
]


@pytest.mark.parametrize("decay", ["slow", "ones"])
@pytest.mark.parametrize("name,kw,chunk,T,T0", CASES)
def test_fwd_continue_matches_the_whole_sequence(sml, name, kw, chunk, T, T0, decay):
    """Output over [T0, T0 + T) from the memories at T0, and the memories at T0 + T."""
    B, H, hpg = 1, 4, 2
    N = T0 + T
    L = levels_for(N)
    Ls = N.bit_length() + 1
    w = workload("small", batch=B, heads=H, heads_per_group=hpg, T=N, levels=L, decay=decay, **kw)
    x = make_inputs(w, "cpu", seed=5 + T0)
    dk, dv = w.d_k, w.d_v
    pst = torch.full((B, H, Ls, dk, dv), float("nan"))
    ref_o = np.zeros((B, T, H, dv))
    ref_end = np.zeros((B, H, Ls, dk, dv))
    for h in range(H):
        o, st = _head_ref(x, 0, h, hpg, N, [T0, N], Ls)
        ref_o[0, :, h] = o[T0:]
        ref_end[0, h] = st[1]
        for lvl in range(1, Ls):
            if (T0 >> (lvl - 1)) & 1:
                pst[0, h, lvl] = torch.from_numpy(st[0][lvl]).float()
    # half of the memory's scale goes into the log-scale, as a decode loop leaves it
    lsc = torch.full((B, H, Ls), -0.75)
    pst = pst * float(np.exp(0.75))
    seg = [t[:, T0:].contiguous().to(DEV) for t in (x.q, x.k, x.v, x.a, x.lam)]
    pst_d, lsc_d = pst.to(DEV), lsc.to(DEV)
    end = torch.full((B, H, Ls, dk, dv), float("nan"), device=DEV)
    end_lsc = torch.full((B, H, Ls), float("nan"), device=DEV)
    o = sml.loglinear_fwd_continue(*seg, T0, pst_d, lsc_d, chunk=chunk, states_out=end,
                                   state_logscale_out=end_lsc, state_levels=Ls)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    assert_parity(o.double().cpu().numpy(), ref_o, f"{name} {decay} o", o.dtype)
    live = [l for l in range(1, Ls) if (N >> (l - 1)) & 1]
    assert torch.all(end_lsc[:, :, live] == 0)
    got_end = end.double().cpu().numpy()
    for l in live:
        assert_parity(got_end[:, :, l], ref_end[:, :, l], f"{name} {decay} end level {l}", "f32")
    # in place: the memories at T0 are replaced by those at T0 + T
    o2 = sml.loglinear_fwd_continue(*seg, T0, pst_d, lsc_d, chunk=chunk, states_out=pst_d,
                                    state_logscale_out=lsc_d, state_levels=Ls)
    torch.cuda.synchronize()
    assert torch.equal(o2, o)
    for l in live:
        assert torch.equal(pst_d[:, :, l], end[:, :, l]), f"in place, level {l}"
        assert float(lsc_d[0, 0, l]) == 0.0


def test_fwd_continue_rejects_unaligned_starts(sml):
    w = workload("small", batch=1, heads=2, T=1024, levels=levels_for(4096))
    x = make_inputs(w, DEV, seed=1)
    st = torch.zeros(1, 2, 13, 128, 64, device=DEV)
    lsc = torch.zeros(1, 2, 13, device=DEV)
    for T0 in (512, 1536, 128):  # not multiples of 1024
        with pytest.raises(sml.LogLinearError):
            sml.loglinear_fwd_continue(x.q, x.k, x.v, x.a, x.lam, T0, st, lsc)


@pytest.mark.parametrize("name,kw,chunk,T", [
    ("tc", dict(d_k=128, d_v=64, dtype=torch.bfloat16), 64, 2048),
    ("tc_ragged", dict(d_k=128, d_v=64, dtype=torch.bfloat16), 64, 1408),
    ("tc_partial", dict(d_k=128, d_v=64, dtype=torch.bfloat16), 64, 1472),
    ("generic", dict(d_k=32, d_v=16, dtype=torch.float32), 16, 320),
])
def test_segment_total(sml, name, kw, chunk, T):
    w = workload("small", batch=2, heads=4, heads_per_group=2, T=T, levels=levels_for(T), decay="slow", **kw)
    x = make_inputs(w, "cpu", seed=8)
    tot, g = sml.loglinear_segment_total(*(t.to(DEV) for t in (x.k, x.v, x.a)), chunk=chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    for b in range(2):
        for h in range(4):
            rt, rg = oracle.segment_total(to_numpy64(x.k[b, :, h // 2]), to_numpy64(x.v[b, :, h]),
                                          to_numpy64(x.a[b, :, h]))
            assert_parity(tot[b, h].double().cpu().numpy(), rt, f"{name} total b={b} h={h}", "f32")
            assert abs(float(g[b, h]) - rg) <= 1e-5 * max(1.0, abs(rg))


@pytest.mark.parametrize("n", [1, 2, 3, 5, 7])
def test_prefix_states(sml, n):
    B, H, dk, dv, seg_len = 2, 3, 128, 64, 2048
    gen = torch.Generator().manual_seed(n)
    seg = torch.randn((n, B, H, dk, dv), generator=gen)
    seg_g = -torch.rand((n, B, H), generator=gen) * 3
    T0 = n * seg_len
    Ls = T0.bit_length() + 1
    st, lsc = sml.loglinear_prefix_states(seg.to(DEV), seg_g.to(DEV), seg_len, Ls)
    torch.cuda.synchronize()
    got = st.double().cpu().numpy()
    for b in range(B):
        for h in range(H):
            ref = oracle.prefix_from_segments(seg[:, b, h].double().numpy(), seg_g[:, b, h].double().numpy(),
                                              seg_len, Ls)
            for lvl in range(1, Ls):
                if (T0 >> (lvl - 1)) & 1:
                    assert_parity(got[b, h, lvl], ref[lvl], f"n={n} level {lvl}", "f32")
                    assert float(lsc[b, h, lvl]) == 0.0


def test_sharded_forward_in_one_process(sml):
    """Four segments of 2048 tokens (tensor-core path): segment memories, one gather,
    prefix memories, continuation; the concatenation against the whole sequence."""
    from structured_mask_linear_gb300.sharded import LibraryBackend

    P, T = 4, 2048
    N = P * T
    w = workload("small", batch=1, heads=2, heads_per_group=2, T=N, levels=levels_for(N), decay="slow")
    x = make_inputs(w, "cpu", seed=12)
    dx = [t.to(DEV) for t in (x.q, x.k, x.v, x.a, x.lam)]
    be = LibraryBackend()
    segs = [[t[:, r * T:(r + 1) * T].contiguous() for t in dx] for r in range(P)]
    tots = [be.segment_total(s[1], s[2], s[3], 64) for s in segs]
    outs = []
    for r in range(P):
        if r == 0:
            outs.append(be.fwd_continue(*segs[r], 0, None, None, 64))
            continue
        pst, plsc = be.prefix_states(torch.stack([t[0] for t in tots[:r]]), torch.stack([t[1] for t in tots[:r]]),
                                     T, (r * T).bit_length() + 1)
        outs.append(be.fwd_continue(*segs[r], r * T, pst, plsc, 64))
    o = torch.cat(outs, dim=1)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    rng = np.random.default_rng(3)
    ts = np.array(sorted(set(int(t) for t in rng.integers(0, N, 150)) | {0, T - 1, T, 2 * T, 3 * T + 5, N - 1}))
    for h in range(2):
        ref = oracle.form_q_points(to_numpy64(x.q[0, :, 0]), to_numpy64(x.k[0, :, 0]), to_numpy64(x.v[0, :, h]),
                                   to_numpy64(x.a[0, :, h]), to_numpy64(x.lam[0, torch.as_tensor(ts), h]), ts)
        got = o[0, torch.as_tensor(ts, device=DEV), h].double().cpu().numpy()
        assert_parity(got, ref, f"sharded h={h}", o.dtype)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from structured_mask_linear_gb300.sharded import sharded_forward

    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    T = 2048
    N = world * T
    w = workload("small", batch=1, heads=4, heads_per_group=2, T=N, levels=levels_for(N), decay="slow")
    x = make_inputs(w, "cpu", seed=21)
    seg = [t[:, rank * T:(rank + 1) * T].contiguous().to("cuda:0") for t in (x.q, x.k, x.v, x.a, x.lam)]
    o = sharded_forward(*seg, chunk=64)
    torch.cuda.synchronize()
    dist.destroy_process_group()
    np.save(os.path.join(out, f"o{rank}.npy"), o.float().cpu().numpy())


def test_sharded_forward_two_gloo_ranks(sml, tmp_path):
    """Two processes, each holding one 2048-token segment on the GPU, one gloo exchange."""
    import torch.multiprocessing as mp

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    got = np.concatenate([np.load(tmp_path / f"o{r}.npy") for r in range(2)], axis=1)
    N = 4096
    w = workload("small", batch=1, heads=4, heads_per_group=2, T=N, levels=levels_for(N), decay="slow")
    x = make_inputs(w, "cpu", seed=21)
    ref = oracle.form_q(*(to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam)))
    assert_parity(got, ref, "two gloo ranks", torch.bfloat16)
