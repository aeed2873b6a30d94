"""The sequence-sharded forward's host logic (structured_mask_linear_gb300.sharded) on the
CPU: gloo ranks that each hold one aligned segment exchange their segments' memories
once, build the bucket memories at their starts and continue the forward from them.

Here the three steps run through an oracle-backed backend (the oracle's segment
functions, pinned in test_oracle_segment_pins.py), so that the ranks, the exchange and
the level bookkeeping are checked without a GPU: the concatenated outputs must equal the
oracle's quadratic form over the whole sequence.  The same module over the library's
kernels is checked on the GPU in test_gpu_segments.py.
"""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class OracleBackend:
    """The three steps of the sharded forward computed by the oracle, head by head."""

    def segment_total(self, k, v, a, chunk):
        import torch

        from oracle import oracle

        B, T, G, dk = k.shape
        H, dv = v.shape[2], v.shape[3]
        tot = np.zeros((B, H, dk, dv))
        g = np.zeros((B, H))
        for b in range(B):
            for h in range(H):
                tot[b, h], g[b, h] = oracle.segment_total(k[b, :, h // (H // G)].double().numpy(),
                                                          v[b, :, h].double().numpy(), a[b, :, h].double().numpy())
        return torch.from_numpy(tot), torch.from_numpy(g)

    def prefix_states(self, seg_states, seg_logdecay, seg_len, levels):
        import torch

        from oracle import oracle

        n, B, H, dk, dv = seg_states.shape
        st = np.zeros((B, H, levels, dk, dv))
        for b in range(B):
            for h in range(H):
                st[b, h] = oracle.prefix_from_segments(seg_states[:, b, h].numpy(), seg_logdecay[:, b, h].numpy(),
                                                       seg_len, levels)
        return torch.from_numpy(st), torch.zeros((B, H, levels), dtype=torch.float64)

    def fwd_continue(self, q, k, v, a, lam, T0, prefix_states, prefix_logscale, chunk):
        import torch

        from oracle import oracle

        B, T, G, dk = q.shape
        H, dv = v.shape[2], v.shape[3]
        levels = (T0 + T).bit_length() + 1
        o = np.zeros((B, T, H, dv))
        for b in range(B):
            for h in range(H):
                g = h // (H // G)
                init = None
                if prefix_states is not None:
                    init = (torch.exp(prefix_logscale[b, h])[:, None, None] * prefix_states[b, h]).numpy()
                o[b, :, h], _ = oracle.form_r_from(q[b, :, g].double().numpy(), k[b, :, g].double().numpy(),
                                                   v[b, :, h].double().numpy(), a[b, :, h].double().numpy(),
                                                   lam[b, :, h].double().numpy(), T0, init, levels)
        return torch.from_numpy(o)


def _inputs(world, T, seed):
    from structured_mask_linear_gb300.inputs import levels_for, make_inputs, workload

    N = world * T
    w = workload("tiny", batch=2, heads=4, heads_per_group=2, T=N, d_k=8, d_v=4, levels=levels_for(N),
                 decay="slow")
    return make_inputs(w, "cpu", seed=seed)


def _rank_main(rank, world, port, T, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist

    from structured_mask_linear_gb300.sharded import sharded_forward
    from test_sharded_gloo import OracleBackend

    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = _inputs(world, T, seed=17)
    seg = slice(rank * T, (rank + 1) * T)
    parts = [t[:, seg].contiguous() for t in (x.q, x.k, x.v, x.a, x.lam)]
    o = sharded_forward(*parts, chunk=16, backend=OracleBackend())
    dist.destroy_process_group()
    np.save(os.path.join(out, f"o{rank}.npy"), o.numpy())


@pytest.mark.parametrize("world,T", [(2, 32), (4, 16), (3, 8)])
def test_sharded_forward_matches_the_whole_sequence(tmp_path, world, T):
    import torch.multiprocessing as mp

    from oracle import oracle
    from structured_mask_linear_gb300.inputs import to_numpy64

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_rank_main, args=(world, port, T, str(tmp_path)), nprocs=world, start_method="spawn")
    got = np.concatenate([np.load(tmp_path / f"o{r}.npy") for r in range(world)], axis=1)
    x = _inputs(world, T, seed=17)
    ref = oracle.form_q(*(to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam)))
    np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-10)


def test_segment_length_must_be_a_power_of_two():
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    from structured_mask_linear_gb300.sharded import sharded_forward

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        z = torch.zeros(1, 24, 1, 8)
        with pytest.raises(ValueError):
            sharded_forward(z, z, torch.zeros(1, 24, 1, 4), torch.ones(1, 24, 1), torch.ones(1, 24, 1, 6),
                            backend=OracleBackend())
    finally:
        dist.destroy_process_group()
