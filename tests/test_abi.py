"""CPU tests of the C-ABI boundary: the library builds and loads, exports every
function include/loglinear.h declares, and validates arguments on the host before
any CUDA call (no GPU needed: every call here returns before touching the device)."""
import ctypes
import os
import re

import pytest

import structured_mask_linear_gb300 as sml
from structured_mask_linear_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "loglinear.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return sml.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:loglinear|ssd)_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for need in ("loglinear_fwd", "loglinear_decode_step", "loglinear_fwd_workspace_bytes",
                 "loglinear_check_status", "loglinear_status_string"):
        assert need in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def shape(**kw):
    d = dict(batch=2, T=2048, heads=8, heads_per_group=2, d_k=128, d_v=64, chunk=64, levels=12,
             dtype=sml.LL_BF16)
    d.update(kw)
    return sml.LLShape(**d)


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first or is all we run


@pytest.mark.parametrize("kw,code", [
    (dict(T=2000), 2),                 # T % chunk
    (dict(chunk=48), 2),               # chunk not a power of two
    (dict(chunk=256), 2),
    (dict(d_k=48), 2),
    (dict(d_k=256), 2),
    (dict(d_v=128), 2),
    (dict(heads=6, heads_per_group=4), 2),
    (dict(levels=11), 2),              # needs bit_length(2047) + 1 = 12
    (dict(dtype=7), 3),
    (dict(batch=0), 2),
    (dict(T=0), 2),
])
def test_fwd_rejects_bad_shapes(L, kw, code):
    s = shape(**kw)
    st = L.loglinear_fwd(ctypes.byref(s), *([FAKE] * 7), 1 << 40, None, None, 0, None)
    assert st == code
    if code == 2 or code == 3:
        assert L.loglinear_fwd_workspace_bytes(ctypes.byref(s)) == 0
        assert L.loglinear_fwd_path(ctypes.byref(s)) == 0


def test_fwd_rejects_null_and_misaligned(L):
    s = shape()
    assert L.loglinear_fwd(None, *([FAKE] * 7), 1 << 40, None, None, 0, None) == 1
    args = [FAKE] * 7
    for i in range(6):
        a = list(args)
        a[i] = None
        assert L.loglinear_fwd(ctypes.byref(s), *a, 1 << 40, None, None, 0, None) == 1
        a[i] = FAKE + 8
        assert L.loglinear_fwd(ctypes.byref(s), *a, 1 << 40, None, None, 0, None) == 4


def test_fwd_rejects_small_workspace_and_bad_export(L):
    s = shape()
    need = L.loglinear_fwd_workspace_bytes(ctypes.byref(s))
    assert need > 0
    assert L.loglinear_fwd(ctypes.byref(s), *([FAKE] * 6), None, need, None, None, 0, None) == 5
    assert L.loglinear_fwd(ctypes.byref(s), *([FAKE] * 7), need - 1, None, None, 0, None) == 5
    # export needs bit_length(2048) + 1 = 13 slots
    assert L.loglinear_fwd(ctypes.byref(s), *([FAKE] * 7), need, FAKE, None, 12, None) == 2
    assert L.loglinear_fwd(ctypes.byref(s), *([FAKE] * 7), need, FAKE + 4, None, 13, None) == 4


def test_decode_validation(L):
    s = shape(levels=17)
    args = [FAKE] * 8
    assert L.loglinear_decode_step(ctypes.byref(s), -1, *args, None) == 2
    # pos + 1 = 65536 needs 18 levels
    assert L.loglinear_decode_step(ctypes.byref(s), 65535, *args, None) == 2
    a = list(args)
    a[6] = None
    assert L.loglinear_decode_step(ctypes.byref(s), 100, *a, None) == 1
    a = list(args)
    a[6] = FAKE + 4
    assert L.loglinear_decode_step(ctypes.byref(s), 100, *a, None) == 4
    assert L.loglinear_decode_step(None, 100, *args, None) == 1


def test_workspace_and_arena_sizes(L):
    s = shape()
    ws = L.loglinear_fwd_workspace_bytes(ctypes.byref(s))
    arena = L.loglinear_fwd_host_arena_bytes(ctypes.byref(s))
    inputs = 2 * (2 * 2048 * 4 * 128 * 2) + 2 * (2 * 2048 * 8 * 64 * 2) + 2 * 2048 * 8 * 4 * 13
    assert arena >= ws + inputs
    assert L.loglinear_fwd_path(ctypes.byref(s)) in (1, 2)
    assert L.loglinear_fwd_path(ctypes.byref(shape(dtype=sml.LL_F32, d_k=16, d_v=16, chunk=16))) == 1


def test_status_strings(L):
    for code in range(9):
        assert len(sml.loglinear_status_string(code)) > 0
    assert sml.loglinear_status_string(99) == "unknown status"


def test_comparators_validate_on_the_host(L):
    """The naive per-level forward and the SSD special case exist for the tensor-core
    shape only: other shapes are rejected before any launch."""
    bad = shape(T=2000)
    assert L.loglinear_fwd_naive_workspace_bytes(ctypes.byref(bad)) == 0
    assert L.ssd_fwd_workspace_bytes(ctypes.byref(bad)) == 0
    assert L.loglinear_fwd_naive(ctypes.byref(bad), *([FAKE] * 6), FAKE, 1 << 30, None) == 2
    assert L.ssd_fwd(ctypes.byref(bad), *([FAKE] * 5), FAKE, 1 << 30, None) == 2
    other = shape(dtype=sml.LL_F32, d_k=64, d_v=32)
    assert L.loglinear_fwd_naive_workspace_bytes(ctypes.byref(other)) == 0
    assert L.loglinear_fwd_naive(ctypes.byref(other), *([FAKE] * 6), FAKE, 1 << 30, None) == 8
    assert L.ssd_fwd(ctypes.byref(other), *([FAKE] * 5), FAKE, 1 << 30, None) == 8
    assert L.ssd_fwd(ctypes.byref(shape()), None, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None) in (1, 8)


def test_binding_signatures_match_the_header(L):
    """Every function the binding declares to ctypes takes as many arguments as the
    header's prototype (a miscount shifts every argument after it)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = dict(re.findall(r"\b((?:loglinear|ssd)_\w+)\s*\(([^)]*)\)\s*;", text))
    checked = 0
    for name, params in protos.items():
        fn = getattr(L, name)
        if getattr(fn, "argtypes", None) is None:
            continue
        n = 0 if params.strip() in ("", "void") else params.count(",") + 1
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)
        checked += 1
    assert checked >= 10
