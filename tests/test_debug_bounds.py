"""The bounds-checking debug build of the C-ABI library (compiled with
-DSAGE_DEBUG_BOUNDS): it builds for sm_103a, exports the same functions as
the normal library, and reports itself as the debug build.  No compute call
is made here (these tests run without a GPU); the GPU side is in
test_gpu_debug_bounds.py."""

import ctypes as C
import os

import pytest

import quantized_attention_sage_gb300 as qas
from quantized_attention_sage_gb300.build import DEBUG_LIB, build

from test_abi import declared_functions


@pytest.fixture(scope="module")
def debug_lib():
    path = build(debug_bounds=True)
    assert path == DEBUG_LIB and os.path.exists(path)
    return C.CDLL(path)


def test_debug_library_exports_every_declared_function(debug_lib):
    for n in declared_functions():
        assert hasattr(debug_lib, n), n


def test_debug_flag_is_set_only_in_the_debug_build(debug_lib):
    qas.build()
    assert qas.lib().sage_debug_bounds_enabled() == 0
    debug_lib.sage_debug_bounds_enabled.restype = C.c_int
    assert debug_lib.sage_debug_bounds_enabled() == 1


def test_debug_bounds_rejects_a_null_record_pointer(debug_lib):
    # host-side argument check, before any CUDA call
    debug_lib.sage_debug_bounds.restype = C.c_int
    debug_lib.sage_debug_bounds.argtypes = [C.c_void_p]
    assert debug_lib.sage_debug_bounds(None) == 1  # SAGE_ERR_INVALID_ARG
    qas.build()
    assert qas.lib().sage_debug_bounds(None) == 1


def test_normal_build_records_nothing_without_touching_the_device():
    qas.build()
    site = C.c_int32(-5)
    assert qas.lib().sage_debug_bounds(C.byref(site)) == 0
    assert site.value == 0
