"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: hand-derived
closed forms (tests/golden), textbook special cases (cumulative-sum linear
attention, the scalar-decay SSD recurrence), structural properties of the
Fenwick partition, and agreement between independently built forms.
"""
import os

import numpy as np
import pytest

from oracle import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _rand_inputs(B, T, H, hpg, dk, dv, L, decay=(0.6, 1.0), lam=(0.2, 2.0)):
    G = H // hpg
    q = rng.standard_normal((B, T, G, dk))
    k = rng.standard_normal((B, T, G, dk))
    v = rng.standard_normal((B, T, H, dv))
    a = rng.uniform(*decay, size=(B, T, H))
    lm = rng.uniform(*lam, size=(B, T, H, L))
    return q, k, v, a, lm


def _rel(x, y):
    return np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300)


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# --- Fenwick partition ------------------------------------------------------

def test_levels_match_hand_table():
    """l(t, s) equals the hand-written binary-indexed-tree table for T = 8."""
    rows = _read_rows("fenwick_levels_T8.txt")
    assert len(rows) == 8
    for t, row in enumerate(rows):
        assert [int(x) for x in row] == [oracle.level(t, s) for s in range(t + 1)]


def test_scalar_closed_form():
    """Hand-computed T = 8 scalar example: Form Q, Form R and brute force."""
    rows = _read_rows("scalar_T8.txt")
    expect = np.array([float(r[1]) for r in rows])
    T, L = 8, 4
    ones = np.ones((1, T, 1, 1))
    a = np.full((1, T, 1), 0.5)
    lam = np.tile(10.0 ** np.arange(L), (1, T, 1, 1))
    for f in (oracle.form_q, oracle.form_r, oracle.brute):
        o = f(ones, ones, ones, a, lam)[0, :, 0, 0]
        np.testing.assert_allclose(o, expect, rtol=1e-14, atol=0)


@pytest.mark.parametrize("T", [2 ** 16])
def test_bucket_invariants_exhaustive(T):
    """For every query t < 2^16: the buckets of the prefix are disjoint with
    union [0, t), have power-of-two sizes growing with distance from t, number
    popcount(t) <= ceil(log2 T), and every key in a bucket of size n has level
    log2(n) + 1 (the bucket levels are what the mask indexes lambda with)."""
    maxb = (T - 1).bit_length()
    for t in range(T):
        bk = oracle.prefix_buckets(t)
        assert len(bk) == bin(t).count("1") <= maxb
        end = t
        prev = 0
        for lo, n in bk:
            assert n & (n - 1) == 0 and n > prev  # power of two, coarser going back
            assert lo + n == end  # contiguous, nearest first, segment ends where the next begins
            end = lo
            prev = n
            if t < 4096 or t % 97 == 0:
                lvl = n.bit_length()  # log2(n) + 1
                assert oracle.level(t, lo) == lvl and oracle.level(t, lo + n - 1) == lvl
        assert end == 0
        assert oracle.level(t, t) == 0


def test_bucket_levels_sampled_to_2_17():
    r = np.random.default_rng(7)
    for t in r.integers(1, 2 ** 17, size=2000):
        t = int(t)
        for lo, n in oracle.prefix_buckets(t):
            s = int(r.integers(lo, lo + n))
            assert oracle.level(t, s) == n.bit_length()


# --- agreement of independent forms ----------------------------------------

@pytest.mark.parametrize("T", [1, 2, 3, 16, 17, 64])
@pytest.mark.parametrize("hpg", [1, 2])
def test_forms_agree_small(T, hpg):
    L = max(T - 1, 0).bit_length() + 1
    q, k, v, a, lam = _rand_inputs(2, T, 4, hpg, 5, 3, L)
    oq = oracle.form_q(q, k, v, a, lam)
    orr = oracle.form_r(q, k, v, a, lam)
    ob = oracle.brute(q, k, v, a, lam)
    assert _rel(oq, ob) < 1e-12
    assert _rel(orr, ob) < 1e-12


def test_forms_agree_tiny_workload_shape():
    """Form Q = Form R at the tiny workload's shape (T = 256, d = 16, 9 levels)."""
    q, k, v, a, lam = _rand_inputs(1, 256, 2, 1, 16, 16, 9)
    assert _rel(oracle.form_r(q, k, v, a, lam), oracle.form_q(q, k, v, a, lam)) < 1e-12


def test_grouping_reads_group_h_div_hpg():
    """Head h reads Q/K group h // hpg (contiguous grouping, MVA)."""
    T, L = 40, 7
    q, k, v, a, lam = _rand_inputs(1, T, 4, 2, 6, 3, L)
    o = oracle.form_q(q, k, v, a, lam)
    for h in range(4):
        g = h // 2
        oh = oracle.brute(q[:, :, g:g + 1], k[:, :, g:g + 1], v[:, :, h:h + 1],
                          a[:, :, h:h + 1], lam[:, :, h:h + 1])
        assert _rel(o[:, :, h:h + 1], oh) < 1e-12


# --- special cases the pages name ------------------------------------------

def test_cumsum_reduction():
    """lambda = 1, a = 1: causal linear attention, o = tril(Q Kᵀ) V (the 0-1 causal
    mask gives the cumulative-sum recurrence, state-space-duality article,
    section 線性化注意力)."""
    T, L = 100, 8
    q, k, v, _, _ = _rand_inputs(1, T, 1, 1, 7, 5, L)
    a = np.ones((1, T, 1))
    lam = np.ones((1, T, 1, L))
    expect = np.tril(q[0, :, 0] @ k[0, :, 0].T) @ v[0, :, 0]
    for f in (oracle.form_q, oracle.form_r):
        assert _rel(f(q, k, v, a, lam)[0, :, 0], expect) < 1e-12


def test_ssd_reduction():
    """lambda_t^l = c_t for every level: o_t = c_t * SSD, the textbook scalar-decay
    recurrence h_t = a_t h_{t-1} + k_t v_tᵀ, o_t = q_tᵀ h_t (log-linear write-up,
    section 特殊结构：树划分: equal weights reduce to linear attention; SSD article,
    section 狀態空間對偶性)."""
    T, L, dk, dv = 300, 10, 6, 4
    q, k, v, a, _ = _rand_inputs(1, T, 1, 1, dk, dv, L, decay=(0.5, 1.0))
    c = rng.uniform(0.5, 2.0, size=T)
    lam = np.repeat(c[None, :, None, None], L, axis=3)
    h = np.zeros((dk, dv))
    expect = np.zeros((T, dv))
    for t in range(T):
        h = a[0, t, 0] * h + np.outer(k[0, t, 0], v[0, t, 0])
        expect[t] = c[t] * (q[0, t, 0] @ h)
    for f in (oracle.form_q, oracle.form_r):
        assert _rel(f(q, k, v, a, lam)[0, :, 0], expect) < 1e-11


@pytest.mark.parametrize("j", list(range(0, 8)))
def test_level_isolation(j):
    """lambda^l = [l == j]: only keys in the level-j bucket contribute.  The bucket
    is walked from the low bits of t up: each set bit b of t is a segment of 2^b
    keys at level b+1, placed just before the finer ones."""
    T, L = 130, 9
    q, k, v, a, _ = _rand_inputs(1, T, 1, 1, 4, 3, L, decay=(0.9, 1.0))
    lam = np.zeros((1, T, 1, L))
    lam[..., j] = 1.0
    expect = np.zeros((T, 3))
    for t in range(T):
        if j == 0:
            keys = [t]
        else:
            end, keys = t, []
            for b in range(16):
                if (t >> b) & 1:
                    if b + 1 == j:
                        keys = list(range(end - (1 << b), end))
                    end -= 1 << b
        for s in keys:
            dec = np.prod(a[0, s + 1:t + 1, 0])
            expect[t] += dec * (q[0, t, 0] @ k[0, s, 0]) * v[0, s, 0]
    for f in (oracle.form_q, oracle.form_r):
        np.testing.assert_allclose(f(q, k, v, a, lam)[0, :, 0], expect, rtol=1e-11, atol=1e-12)


def test_points_match_full_form():
    T, L = 200, 9
    q, k, v, a, lam = _rand_inputs(1, T, 2, 2, 8, 4, L)
    o = oracle.form_q(q, k, v, a, lam)
    ts = np.array([0, 1, 63, 64, 127, 199])
    op = oracle.form_q_points(q[0, :, 0], k[0, :, 0], v[0, :, 1], a[0, :, 1], lam[0, ts, 1], ts)
    assert _rel(op, o[0, ts, 1]) < 1e-13


# --- the recurrent states (decode hand-off) --------------------------------

def test_state_export_is_bucket_sum():
    """The exported state of level l at position T is the decayed sum of k vᵀ over
    the level-l bucket of T; for T = 2^p the only live level is p+1 and it holds
    the whole prefix (state-space form of the last bucket)."""
    for T in (64, 96, 100):
        L = (T - 1).bit_length() + 1
        Ls = T.bit_length() + 1
        q, k, v, a, lam = _rand_inputs(1, T, 1, 1, 3, 2, L)
        _, st = oracle.form_r(q, k, v, a, lam, export_levels=Ls)
        end = T
        for b in range(Ls - 1):
            lvl = b + 1
            if (T >> b) & 1:
                lo = end - (1 << b)
                S = np.zeros((3, 2))
                for s in range(lo, end):
                    S += np.prod(a[0, s + 1:T, 0]) * np.outer(k[0, s, 0], v[0, s, 0])
                np.testing.assert_allclose(st[0, 0, lvl], S, rtol=1e-12, atol=1e-14)
                end = lo
            else:
                assert np.all(st[0, 0, lvl] == 0)
        assert end == 0


def test_form_r_head_capture_continues_prefix():
    """Running Form R over prefix + steps gives the same outputs for the steps as
    a quadratic evaluation at those points, and captures the prefix state."""
    T0, n = 64, 20
    T = T0 + n
    L = (T - 1).bit_length() + 1
    q, k, v, a, lam = _rand_inputs(1, T, 1, 1, 4, 3, L)
    o, st = oracle.form_r_head(q[0, :, 0], k[0, :, 0], v[0, :, 0], a[0, :, 0], lam[0, :, 0],
                               [T0, T], levels=T.bit_length() + 1)
    ts = np.arange(T0, T)
    op = oracle.form_q_points(q[0, :, 0], k[0, :, 0], v[0, :, 0], a[0, :, 0], lam[0, ts, 0], ts)
    assert _rel(o[T0:], op) < 1e-12
    _, st2 = oracle.form_r(q[:, :T0], k[:, :T0], v[:, :T0], a[:, :T0], lam[:, :T0],
                           export_levels=T.bit_length() + 1)
    assert _rel(st[0], st2[0, 0]) < 1e-13
