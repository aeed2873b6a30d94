"""Pins of the oracle's sequence-segment functions (form_r_from, segment_total,
prefix_from_segments) against the forms pinned elsewhere: the recurrent form run over
the whole sequence (form_r_head, pinned to the quadratic form and the brute force) and
the quadratic form itself.

Sources: the per-bucket memories of the log-linear attention write-up
(https://www.yoousoft.com/industry/3746.html, section 特殊结构：树划分, Fig. 2) and the
combination of chunk memories level by level (section 高效训练算法, Algorithm 1).
"""
import numpy as np
import pytest

from oracle import oracle


def _seq(T, dk=5, dv=3, L=None, seed=0, decay=0.3):
    rng = np.random.default_rng(seed)
    L = L or (max(T - 1, 0).bit_length() + 2)
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    a = np.exp(-rng.random(T) * decay)
    lam = rng.random((T, L)) + 0.5
    return q, k, v, a, lam


@pytest.mark.parametrize("T0", [0, 1, 5, 16, 24, 37])
def test_form_r_from_continues_the_whole_sequence(T0):
    """Starting at any position T0 from the memories captured there gives the same outputs
    and the same final memories as the recurrent form run from position 0."""
    T = 48
    q, k, v, a, lam = _seq(T, seed=T0)
    Ls = T.bit_length() + 1
    o, st = oracle.form_r_head(q, k, v, a, lam, [T0, T], levels=Ls)
    o2, fin = oracle.form_r_from(q[T0:], k[T0:], v[T0:], a[T0:], lam[T0:], T0, st[0], Ls)
    np.testing.assert_allclose(o2, o[T0:], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fin, st[1], rtol=1e-12, atol=1e-12)


def test_form_r_from_ignores_dead_levels():
    """Slots of levels that are not live at T0 do not enter (garbage there changes nothing)."""
    T, T0 = 40, 24  # live at 24: levels 4 and 5
    q, k, v, a, lam = _seq(T, seed=3)
    Ls = T.bit_length() + 1
    _, st = oracle.form_r_head(q, k, v, a, lam, [T0], levels=Ls)
    init = st[0].copy()
    for lvl in range(Ls):
        if not (lvl >= 1 and (T0 >> (lvl - 1)) & 1):
            init[lvl] = 1e6
    o1, _ = oracle.form_r_from(q[T0:], k[T0:], v[T0:], a[T0:], lam[T0:], T0, st[0], Ls)
    o2, _ = oracle.form_r_from(q[T0:], k[T0:], v[T0:], a[T0:], lam[T0:], T0, init, Ls)
    np.testing.assert_array_equal(o1, o2)


@pytest.mark.parametrize("T", [1, 2, 7, 16, 33, 64])
def test_segment_total_is_the_sum_of_the_live_memories(T):
    """The memory of a segment of T tokens is the sum of the live bucket memories the
    recurrent form holds at position T (one level-(p+1) bucket when T = 2^p)."""
    q, k, v, a, lam = _seq(T, seed=T)
    Ls = T.bit_length() + 1
    _, st = oracle.form_r_head(q, k, v, a, lam, [T], levels=Ls)
    tot, g = oracle.segment_total(k, v, a)
    np.testing.assert_allclose(tot, st[0].sum(axis=0), rtol=1e-12, atol=1e-12)
    if T & (T - 1) == 0:
        np.testing.assert_allclose(tot, st[0][T.bit_length()], rtol=1e-12, atol=1e-12)
    # the summed log-decay: the factor every earlier memory takes across the segment
    assert np.isclose(np.exp(g), np.prod(a), rtol=1e-12)


@pytest.mark.parametrize("seg_len,P", [(8, 6), (4, 8), (16, 3), (1, 7)])
def test_prefix_from_segments_equals_the_captured_memories(seg_len, P):
    """The bucket memories at T0 = r * seg_len built from the segments' memories equal the
    recurrent form's memories at T0, for every r."""
    T = seg_len * P
    q, k, v, a, lam = _seq(T, seed=seg_len + P, decay=0.2)
    Ls = T.bit_length() + 1
    caps = [r * seg_len for r in range(P + 1)]
    _, st = oracle.form_r_head(q, k, v, a, lam, caps, levels=Ls)
    tots, gs = [], []
    for r in range(P):
        s = slice(r * seg_len, (r + 1) * seg_len)
        t, g = oracle.segment_total(k[s], v[s], a[s])
        tots.append(t)
        gs.append(g)
    for r in range(P + 1):
        pre = oracle.prefix_from_segments(np.array(tots[:r]).reshape(r, 5, 3), np.array(gs[:r]),
                                          seg_len, Ls)
        np.testing.assert_allclose(pre, st[r], rtol=1e-11, atol=1e-12, err_msg=f"r={r}")


@pytest.mark.parametrize("seg_len,P", [(16, 4), (8, 5)])
def test_sharded_composition_equals_the_quadratic_form(seg_len, P):
    """Segment memories -> prefix memories at each segment start -> the recurrent form
    over each segment gives the quadratic form's output on the whole sequence."""
    T = seg_len * P
    q, k, v, a, lam = _seq(T, seed=7, decay=0.1)
    ref = oracle.form_q(q[None, :, None], k[None, :, None], v[None, :, None], a[None, :, None],
                        lam[None, :, None])[0, :, 0]
    tots, gs = [], []
    for r in range(P):
        s = slice(r * seg_len, (r + 1) * seg_len)
        t, g = oracle.segment_total(k[s], v[s], a[s])
        tots.append(t)
        gs.append(g)
    Ls = T.bit_length() + 1
    out = []
    for r in range(P):
        s = slice(r * seg_len, (r + 1) * seg_len)
        pre = oracle.prefix_from_segments(np.array(tots[:r]).reshape(r, 5, 3), np.array(gs[:r]),
                                          seg_len, Ls)
        o, _ = oracle.form_r_from(q[s], k[s], v[s], a[s], lam[s], r * seg_len, pre, Ls)
        out.append(o)
    np.testing.assert_allclose(np.concatenate(out), ref, rtol=1e-10, atol=1e-11)
