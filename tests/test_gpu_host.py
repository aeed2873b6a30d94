"""The end-to-end forward from host buffers (loglinear_fwd_host), through the C ABI.

It cuts the batch into pieces whose copies and forwards overlap on three streams; each
(b, h, tile) is computed the same way as by loglinear_fwd on device buffers, so the host
result must equal the device result exactly.  Cases: batch sizes that give one piece,
uneven pieces and more elements than pieces, on the tensor-core and the generic paths,
and a second call on the same arena.
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


def _host_run(sml, x, chunk, arena=None):
    hq, hk, hv, ha, hl = (t.contiguous().pin_memory() for t in (x.q, x.k, x.v, x.a, x.lam))
    ho = torch.empty(x.v.shape, dtype=x.v.dtype).pin_memory()
    shape = sml.fwd_shape(hq, hv, hl, chunk)
    if arena is None:
        arena = torch.empty(sml.loglinear_fwd_host_arena_bytes(shape), dtype=torch.uint8, device=DEV)
    sml.loglinear_fwd_host(hq, hk, hv, ha, hl, ho, arena, chunk=chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0
    return ho, arena


@pytest.mark.parametrize("name,batch,T", [("small", 1, 1024), ("small", 3, 1024), ("small", 11, 256),
                                          ("tiny", 5, 256)])
def test_host_forward_equals_device_forward(sml, name, batch, T):
    w = workload(name, batch=batch, heads=4 if name == "small" else 2, T=T, levels=levels_for(T))
    x = make_inputs(w, "cpu", seed=61)
    ho, arena = _host_run(sml, x, w.chunk)
    od = sml.loglinear_fwd(*(t.to(DEV) for t in (x.q, x.k, x.v, x.a, x.lam)), chunk=w.chunk)
    torch.cuda.synchronize()
    assert torch.equal(ho, od.cpu())
    if batch == 3:
        assert_parity(ho.double().numpy(), oracle.form_q(*(to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam))),
                      "host forward", ho.dtype)
    # a second call on the same arena with other inputs
    x2 = make_inputs(w, "cpu", seed=62)
    ho2, _ = _host_run(sml, x2, w.chunk, arena)
    od2 = sml.loglinear_fwd(*(t.to(DEV) for t in (x2.q, x2.k, x2.v, x2.a, x2.lam)), chunk=w.chunk)
    torch.cuda.synchronize()
    assert torch.equal(ho2, od2.cpu())


def test_host_forward_from_two_threads(sml):
    """Two host threads call loglinear_fwd_host at once, each on its own stream, arena and
    host buffers, several times over: every result must equal the device forward of its
    own inputs (the library holds a per-device lock while a call enqueues its copies)."""
    import threading

    w = workload("small", batch=3, heads=4, T=1024, levels=levels_for(1024))
    xs = [make_inputs(w, "cpu", seed=71 + i) for i in range(2)]
    refs = []
    for x in xs:
        refs.append(sml.loglinear_fwd(*(t.to(DEV) for t in (x.q, x.k, x.v, x.a, x.lam)), chunk=w.chunk).cpu())
    torch.cuda.synchronize()
    outs = [[], []]
    errors = []

    def run(i):
        try:
            x = xs[i]
            hq, hk, hv, ha, hl = (t.contiguous().pin_memory() for t in (x.q, x.k, x.v, x.a, x.lam))
            shape = sml.fwd_shape(hq, hv, hl, w.chunk)
            arena = torch.empty(sml.loglinear_fwd_host_arena_bytes(shape), dtype=torch.uint8, device=DEV)
            stream = torch.cuda.Stream(device=DEV)
            for _ in range(6):
                ho = torch.empty(x.v.shape, dtype=x.v.dtype).pin_memory()
                sml.loglinear_fwd_host(hq, hk, hv, ha, hl, ho, arena, chunk=w.chunk, stream=stream)
                outs[i].append(ho)
            stream.synchronize()
        except Exception as e:  # reported below, in the test's own thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert sml.loglinear_check_status() == 0
    for i in range(2):
        assert len(outs[i]) == 6
        for ho in outs[i]:
            assert torch.equal(ho, refs[i])
