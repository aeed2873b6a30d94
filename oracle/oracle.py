"""ctypes wrapper around the fp64 CPU oracle in loglinear_oracle.c.

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the product path.  It
shares no code with the CUDA path: it takes numpy arrays (already rounded to
the dtype the GPU consumes) and returns fp64 numpy arrays.

What each function computes, and the passage it follows, is stated in the C
file's header and above each C function.  Summary:

* ``level(t, s)``           Fenwick level of key s for query t (page 1 of the
                            sources, 特殊结构：树划分).
* ``prefix_buckets(n)``     binary-indexed-tree segments of the prefix [0, n).
* ``form_q``                quadratic masked form (QKᵀ ⊙ M^S ⊙ M^H) V.
* ``form_q_points``         the same at chosen query positions of one head.
* ``form_r``                recurrent per-bucket-state form, optional export
                            of the bucket states at position T.
* ``form_r_head``           one head, capturing states at chosen positions.
* ``brute``                 dense masks built by explicit loops (small T).
* ``backward``              gradients of sum(dO * o) with respect to q, k, v,
                            log a and lambda: the chain rule on the quadratic form.
* ``gdn_values``            Gated DeltaNet's transformed values u (gated delta rule
                            run token by token); ``gdn_forward`` = form_q with v = u.
* ``form_r_from``           the recurrent form over the tokens T0 .. T0+T-1 of one
                            head, starting from the bucket memories at T0.
* ``segment_total``         the memory of a whole segment and its summed log-decay.
* ``prefix_from_segments``  the bucket memories at T0 = r * seg_len built from the
                            memories of the r segments before it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "loglinear_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libloglinear_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_L = ctypes.POINTER(ctypes.c_long)
_l = ctypes.c_long


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP) into oracle/_build/."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_level.restype = ctypes.c_int
            lib.oracle_level.argtypes = [_l, _l]
            lib.oracle_prefix_buckets.restype = ctypes.c_int
            lib.oracle_prefix_buckets.argtypes = [_l, _L, _L, ctypes.c_int]
            lib.oracle_num_threads.restype = ctypes.c_int
            six = [_l] * 7
            lib.oracle_form_q.argtypes = six + [_D] * 6
            lib.oracle_brute.argtypes = six + [_D] * 6
            lib.oracle_form_r.argtypes = six + [_D] * 7 + [_l]
            lib.oracle_form_q_points.argtypes = [_l] * 4 + [_D] * 5 + [_L, _l, _D]
            lib.oracle_form_r_head.argtypes = [_l] * 4 + [_D] * 6 + [_l, _l, _L, _D]
            lib.oracle_backward.argtypes = six + [_D] * 11
            lib.oracle_gdn_values.argtypes = [_l] * 6 + [_D] * 5
            lib.oracle_form_r_from.argtypes = [_l] * 5 + [_D] * 5 + [_l] + [_D] * 3
            lib.oracle_segment_total.argtypes = [_l] * 3 + [_D] * 5
            lib.oracle_prefix_from_segments.argtypes = [_l] * 4 + [_D] * 2 + [_l, _D]
            for f in ("oracle_form_q", "oracle_brute", "oracle_form_r", "oracle_form_q_points",
                      "oracle_form_r_head", "oracle_backward", "oracle_gdn_values",
                      "oracle_form_r_from", "oracle_segment_total", "oracle_prefix_from_segments"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _d(x: np.ndarray):
    return x.ctypes.data_as(_D)


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _bitlen(x: int) -> int:
    return int(x).bit_length()


def level(t: int, s: int) -> int:
    return int(_load().oracle_level(int(t), int(s)))


def prefix_buckets(n: int):
    """Segments (start, length) of the prefix [0, n), nearest first."""
    lo = (ctypes.c_long * 64)()
    ln = (ctypes.c_long * 64)()
    c = _load().oracle_prefix_buckets(int(n), lo, ln, 64)
    return [(int(lo[i]), int(ln[i])) for i in range(c)]


def _check(q, k, v, a, lam):
    q, k, v, a, lam = (_f64(x) for x in (q, k, v, a, lam))
    B, T, G, dk = q.shape
    H, dv = v.shape[2], v.shape[3]
    L = lam.shape[3]
    assert k.shape == q.shape and v.shape[:2] == (B, T) and a.shape == (B, T, H)
    assert lam.shape[:3] == (B, T, H) and H % G == 0
    if T > 0:
        assert L >= _bitlen(T - 1) + 1, "lambda needs bit_length(T-1)+1 levels"
    return q, k, v, a, lam, (B, T, H, H // G, dk, dv, L)


def form_q(q, k, v, a, lam) -> np.ndarray:
    q, k, v, a, lam, shp = _check(q, k, v, a, lam)
    B, T, H, _, _, dv, _ = shp
    o = np.zeros((B, T, H, dv), dtype=np.float64)
    _load().oracle_form_q(*shp, _d(q), _d(k), _d(v), _d(a), _d(lam), _d(o))
    return o


def brute(q, k, v, a, lam) -> np.ndarray:
    q, k, v, a, lam, shp = _check(q, k, v, a, lam)
    B, T, H, _, _, dv, _ = shp
    assert T <= 256, "brute force is for small T"
    o = np.zeros((B, T, H, dv), dtype=np.float64)
    _load().oracle_brute(*shp, _d(q), _d(k), _d(v), _d(a), _d(lam), _d(o))
    return o


def form_r(q, k, v, a, lam, export_levels: int | None = None):
    """Returns o, and the bucket states at position T when export_levels is given
    (shape (B, H, export_levels, dk, dv))."""
    q, k, v, a, lam, shp = _check(q, k, v, a, lam)
    B, T, H, _, dk, dv, L = shp
    Ls = max(L, _bitlen(T) + 1)
    if export_levels is not None:
        assert export_levels >= _bitlen(T) + 1
        Ls = max(Ls, export_levels)
    o = np.zeros((B, T, H, dv), dtype=np.float64)
    st = np.zeros((B, H, Ls, dk, dv), dtype=np.float64) if export_levels is not None else None
    _load().oracle_form_r(*shp, _d(q), _d(k), _d(v), _d(a), _d(lam), _d(o),
                          _d(st) if st is not None else None, Ls)
    if st is None:
        return o
    return o, st[:, :, :export_levels]


def form_q_points(q, k, v, a, lam_pts, ts) -> np.ndarray:
    """One head: q, k (T', dk), v (T', dv), a (T'), lam_pts (n, L) for the
    queries ts (n); positions are 0-based and ts < T'.  Returns (n, dv)."""
    q, k, v, a, lam_pts = (_f64(x) for x in (q, k, v, a, lam_pts))
    ts = np.ascontiguousarray(np.asarray(ts, dtype=np.int64))
    T, dk = q.shape
    dv = v.shape[1]
    n, L = lam_pts.shape
    assert ts.shape == (n,) and (n == 0 or (ts.min() >= 0 and ts.max() < T))
    assert n == 0 or L >= _bitlen(int(ts.max())) + 1
    o = np.zeros((n, dv), dtype=np.float64)
    _load().oracle_form_q_points(T, dk, dv, L, _d(q), _d(k), _d(v), _d(a), _d(lam_pts),
                                 ts.ctypes.data_as(_L), n, _d(o))
    return o


def form_r_head(q, k, v, a, lam, cap_pos, levels: int):
    """One head over T tokens: returns o (T, dv) and states (len(cap_pos),
    levels, dk, dv) captured at each position in cap_pos (ascending, <= T)."""
    q, k, v, a, lam = (_f64(x) for x in (q, k, v, a, lam))
    T, dk = q.shape
    dv = v.shape[1]
    L = lam.shape[1]
    cap = np.ascontiguousarray(np.asarray(cap_pos, dtype=np.int64))
    assert np.all(np.diff(cap) >= 0) and (cap.size == 0 or cap.max() <= T)
    assert levels >= _bitlen(T) + 1 and L >= _bitlen(max(T - 1, 0)) + 1
    o = np.zeros((T, dv), dtype=np.float64)
    st = np.zeros((cap.size, levels, dk, dv), dtype=np.float64)
    _load().oracle_form_r_head(T, dk, dv, L, _d(q), _d(k), _d(v), _d(a), _d(lam), _d(o),
                               levels, cap.size, cap.ctypes.data_as(_L), _d(st))
    return o, st


def backward(q, k, v, a, lam, dO):
    """Gradients of sum(dO * form_q(q, k, v, a, lam)): returns dq, dk (B, T, G, dk),
    dv (B, T, H, dv), dloga (B, T, H: with respect to log a; divide by a for the
    gradient with respect to a) and dlam (B, T, H, L), all fp64."""
    q, k, v, a, lam, shp = _check(q, k, v, a, lam)
    dO = _f64(dO)
    B, T, H, hpg, dk, dv, L = shp
    G = H // hpg
    assert dO.shape == (B, T, H, dv)
    dq = np.zeros((B, T, G, dk))
    dkk = np.zeros((B, T, G, dk))
    dvv = np.zeros((B, T, H, dv))
    dla = np.zeros((B, T, H))
    dl = np.zeros((B, T, H, L))
    _load().oracle_backward(*shp, _d(q), _d(k), _d(v), _d(a), _d(lam), _d(dO), _d(dq), _d(dkk),
                            _d(dvv), _d(dla), _d(dl))
    return dq, dkk, dvv, dla, dl


def gdn_values(k, v, a, beta) -> np.ndarray:
    """u_t = beta_t (v_t - a_t S_{t-1} k_t) of the gated delta rule S_t = a_t S_{t-1} +
    u_t k_tᵀ.  k: (B, T, G, dk); v: (B, T, H, dv); a, beta: (B, T, H).  Returns (B, T, H, dv)."""
    k, v, a, beta = (_f64(x) for x in (k, v, a, beta))
    B, T, G, dk = k.shape
    H, dv = v.shape[2], v.shape[3]
    assert a.shape == (B, T, H) and beta.shape == (B, T, H) and H % G == 0
    u = np.zeros((B, T, H, dv))
    _load().oracle_gdn_values(B, T, H, H // G, dk, dv, _d(k), _d(v), _d(a), _d(beta), _d(u))
    return u


def gdn_forward(q, k, v, a, beta, lam) -> np.ndarray:
    """Log-linear Gated DeltaNet: the masked form with the transformed values u."""
    return form_q(q, k, gdn_values(k, v, a, beta), a, lam)


def form_r_from(q, k, v, a, lam, T0: int, init_states, levels: int):
    """One head, the tokens at positions T0 .. T0+T-1: q, k (T, dk), v (T, dv), a (T),
    lam (T, L), and the bucket memories at T0 init_states (>= bit_length(T0)+1 levels,
    dk, dv; levels not live at T0 are ignored).  Returns o (T, dv) and the live memories
    at T0+T (levels, dk, dv)."""
    q, k, v, a, lam = (_f64(x) for x in (q, k, v, a, lam))
    T, dk = q.shape
    dv = v.shape[1]
    L = lam.shape[1]
    assert levels >= _bitlen(T0 + T) + 1 and L >= _bitlen(max(T0 + T - 1, 0)) + 1
    init = np.zeros((levels, dk, dv))
    if init_states is not None:
        src = _f64(init_states)
        n = min(levels, src.shape[0])
        init[:n] = src[:n]
    o = np.zeros((T, dv))
    fin = np.zeros((levels, dk, dv))
    _load().oracle_form_r_from(int(T0), T, dk, dv, L, _d(q), _d(k), _d(v), _d(a), _d(lam), levels,
                               _d(init), _d(o), _d(fin))
    return o, fin


def segment_total(k, v, a):
    """One head's segment: k (T, dk), v (T, dv), a (T).  Returns the segment's memory
    sum_s (a_{s+1} ... a_{T-1}) k_s v_sᵀ (dk, dv) and its summed log-decay."""
    k, v, a = (_f64(x) for x in (k, v, a))
    T, dk = k.shape
    dv = v.shape[1]
    tot = np.zeros((dk, dv))
    g = np.zeros(1)
    _load().oracle_segment_total(T, dk, dv, _d(k), _d(v), _d(a), _d(tot), _d(g))
    return tot, float(g[0])


def prefix_from_segments(seg_states, seg_logdecay, seg_len: int, levels: int):
    """Bucket memories at T0 = r * seg_len (r = len(seg_states), seg_len a power of two)
    from the r segments' memories (r, dk, dv) and summed log-decays (r)."""
    st = _f64(seg_states)
    g = _f64(seg_logdecay)
    r, dk, dv = st.shape
    assert seg_len > 0 and seg_len & (seg_len - 1) == 0
    assert levels >= _bitlen(r * seg_len) + 1
    out = np.zeros((levels, dk, dv))
    _load().oracle_prefix_from_segments(r, seg_len, dk, dv, _d(st), _d(g), levels, _d(out))
    return out
