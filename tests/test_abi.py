"""C-ABI checks that need no GPU: the library loads, exports every function
include/m2rnn.h declares, and rejects bad arguments on the host before any
device work."""
import ctypes
import os
import re

import pytest

from non_linear_matrix_gb300 import build as nb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    nb.build()
    from non_linear_matrix_gb300 import m2rnn
    return m2rnn.lib()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(m2rnn_\w+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert "m2rnn_fwd" in names and "m2rnn_bwd" in names
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    from non_linear_matrix_gb300 import m2rnn
    assert lib.m2rnn_version() >= 201
    for code in range(-8, 1):
        assert m2rnn.status_string(code) != "unknown status", code
        assert code in m2rnn.STATUS, code
    assert m2rnn.status_string(12345) == "unknown status"


def test_checked_build_is_a_separate_library(lib):
    """The normal build reports m2rnn_checked() == 0; the checked build (same
    sources, -DM2RNN_CHECK=1) reports 1, exports the same functions and
    describes M2RNN_ERR_BOUNDS."""
    from non_linear_matrix_gb300 import m2rnn
    assert lib.m2rnn_checked() == 0
    path = nb.build(checked=True)
    assert path == m2rnn.LIB_CHECKED_PATH and path != m2rnn.LIB_PATH
    chk = ctypes.CDLL(path)
    chk.m2rnn_checked.restype = ctypes.c_int
    chk.m2rnn_status_string.restype = ctypes.c_char_p
    chk.m2rnn_status_string.argtypes = [ctypes.c_int]
    assert chk.m2rnn_checked() == 1
    for name in _declared_functions():
        assert hasattr(chk, name), name
    assert b"checked build" in chk.m2rnn_status_string(-8)


def test_fault_injection_modes(lib):
    assert lib.m2rnn_set_fault_injection(2) == -1
    assert lib.m2rnn_set_fault_injection(0) == 0


def test_num_checkpoints(lib):
    from non_linear_matrix_gb300.m2rnn import Shape, num_checkpoints
    assert num_checkpoints(Shape(8, 4096, 32, 64, 16, 1, 64)) == 64
    assert num_checkpoints(Shape(1, 100, 4, 64, 16, 1, 64)) == 2
    assert num_checkpoints(Shape(1, 64, 4, 64, 16, 1, 64)) == 1
    assert num_checkpoints(Shape(1, 0, 4, 64, 16, 1, 64)) == 0
    assert num_checkpoints(Shape(1, 64, 4, 64, 16, 1, 0)) == 0


@pytest.mark.parametrize("shape,code", [
    (None, -1),
    ((1, 8, 2, 48, 16, 1, 0), -2),   # K not supported
    ((1, 8, 2, 64, 24, 1, 0), -2),   # V not supported
    ((1, 8, 2, 64, 16, 7, 0), -1),   # bad dtype
    ((0, 8, 2, 64, 16, 1, 0), -1),   # B < 1
    ((1, -1, 2, 64, 16, 1, 0), -1),  # T < 0
    ((1, 8, 2, 64, 16, 1, -4), -1),  # negative checkpoint interval
])
def test_fwd_rejects_bad_shapes_before_launch(lib, shape, code):
    from non_linear_matrix_gb300.m2rnn import Shape
    s = None if shape is None else ctypes.byref(Shape(*shape))
    p = ctypes.c_void_p(16)
    rc = lib.m2rnn_fwd(s, p, p, p, p, p, p, None, p, None, None, None)
    assert rc == code


def test_bwd_rejects_bad_shapes_before_launch(lib):
    from non_linear_matrix_gb300.m2rnn import Shape
    p = ctypes.c_void_p(16)
    s = ctypes.byref(Shape(1, 8, 2, 48, 16, 1, 4))
    rc = lib.m2rnn_bwd(s, *([p] * 6), None, None, p, None, *([p] * 6), None, None, p,
                       ctypes.c_size_t(1 << 20), None)
    assert rc in (-1, -2)


def test_decode_rejects_bad_arguments_before_launch(lib):
    """T must be 1 and K, V supported; both are checked before any device
    call."""
    from non_linear_matrix_gb300.m2rnn import Shape
    p = ctypes.c_void_p(16)
    assert lib.m2rnn_decode(ctypes.byref(Shape(4, 2, 2, 64, 16, 1, 0)), *([p] * 10)) == -1
    assert lib.m2rnn_decode(ctypes.byref(Shape(4, 1, 2, 48, 16, 1, 0)), *([p] * 10)) == -2
    assert lib.m2rnn_decode(None, *([p] * 10)) == -1


def test_gated_entry_points_reject_bad_shapes_before_launch(lib):
    from non_linear_matrix_gb300.m2rnn import Shape
    p = ctypes.c_void_p(16)
    bad = ctypes.byref(Shape(1, 8, 2, 48, 16, 1, 4))
    assert lib.m2rnn_fwd_gated(bad, *([p] * 8), None, p, None, None, None) == -2
    assert lib.m2rnn_fwd_gated(None, *([p] * 8), None, p, None, None, None) == -1
    assert lib.m2rnn_bwd_gated(bad, *([p] * 8), None, None, p, None, *([p] * 8), None, None, p,
                               ctypes.c_size_t(1 << 20), None) == -2
    nock = ctypes.byref(Shape(1, 8, 2, 64, 16, 1, 0))  # ckpt_every must be > 0
    assert lib.m2rnn_bwd_gated(nock, *([p] * 8), None, None, p, None, *([p] * 8), None, None, p,
                               ctypes.c_size_t(1 << 20), None) == -1


@pytest.mark.parametrize("Nq", [-1, 3, 5])
def test_groups_must_divide_heads(lib, Nq):
    """Nq query/key groups must be >= 0 (0 reads as 1) and divide N; checked
    before any device call."""
    from non_linear_matrix_gb300.m2rnn import Shape
    p = ctypes.c_void_p(16)
    s = ctypes.byref(Shape(1, 8, 4, 64, 16, 1, 0, Nq))
    assert lib.m2rnn_fwd(s, p, p, p, p, p, p, None, p, None, None, None) == -1
    assert lib.m2rnn_decode(ctypes.byref(Shape(1, 1, 4, 64, 16, 1, 0, Nq)), *([p] * 10)) == -1


def test_norm_entry_points_take_f_or_gate(lib):
    """m2rnn_fwd_norm / m2rnn_bwd_norm take f or (a, alpha, beta), exactly
    one form; the choice is checked before anything else."""
    from non_linear_matrix_gb300.m2rnn import Shape
    p = ctypes.c_void_p(16)
    s = ctypes.byref(Shape(1, 8, 2, 64, 16, 1, 4))
    eps = ctypes.c_float(0.0)
    both = [p, p, p, p]      # f and the gate
    neither = [None] * 4
    for fa in (both, neither, [p, p, None, p]):
        assert lib.m2rnn_fwd_norm(s, p, p, p, *fa, p, p, None, p, p, eps, p, p, p, None, None,
                                  None) == -1
        assert lib.m2rnn_bwd_norm(s, p, p, p, *fa, p, p, None, None, *([p] * 5), None,
                                  *([p] * 10), None, None, p, ctypes.c_size_t(1 << 20),
                                  None) == -1
