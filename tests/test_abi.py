"""C ABI of libsnack on the host: the library loads, exports every entry point
declared in include/snack.h, and rejects bad arguments before touching a GPU."""

import ctypes
import os
import re

import pytest

from spmm_row_sorted_gb300 import build as snack_build
from spmm_row_sorted_gb300 import snack

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "snack.h")


@pytest.fixture(scope="module")
def lib():
    snack_build.build()
    return snack.load()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(snack_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(snack.EXPORTED), names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_status_strings(lib):
    assert snack.snack_version() == 1
    for code in range(9):
        assert snack.snack_status_string(code)
    assert "unknown" in snack.snack_status_string(99)


def test_query_sizes_monotone_in_batch(lib):
    prev = 0
    for b in (1, 2, 3, 8, 17, 32, 33, 64, 100, 1024):
        _, ws = snack.snack_query_sizes(4096, 2048, 50000, b, 0, 0)
        assert ws >= prev
        prev = ws
    plan, ws = snack.snack_query_sizes(16384, 16384, 2684355, 32, 0, 0)
    assert plan % 256 == 0 and ws % 256 == 0
    assert plan >= 4 * (16384 + 1) + 8 * 2684355


@pytest.mark.parametrize("args", [
    (0, 10, 5, 8, 0, 0),        # out_f < 1
    (10, 0, 5, 8, 0, 0),        # in_f < 1
    (10, 10, 101, 8, 0, 0),     # nnz > out*in
    (10, 10, -1, 8, 0, 0),      # nnz < 0
    (10, 10, 5, 0, 0, 0),       # max_batch < 1
    (10, 10, 5, 70000, 0, 0),   # max_batch too large
    (10, 10, 5, 8, 0, 5),       # bad dtype
])
def test_query_rejects_bad_shapes(lib, args):
    with pytest.raises(snack.SnackError) as e:
        snack.snack_query_sizes(*args)
    assert e.value.status == 1


def test_mixed_dtypes_unsupported(lib):
    with pytest.raises(snack.SnackError) as e:
        snack.snack_query_sizes(10, 10, 5, 8, 0, 1)
    assert e.value.status == 7


def test_null_handle_rejected_without_gpu(lib):
    vp = ctypes.c_void_p
    assert lib.snack_spmm_fwd(None, None, None, None, None, 1, None, None, None, 0, None) == 1
    assert lib.snack_spmm_dx(None, None, None, None, None, 1, None, None, 0, None) == 1
    assert lib.snack_sddmm_dw(None, None, None, None, None, 1, None, None, None, 0, None) == 1
    assert lib.snack_restructure(None, None, None, None, 1, 0, 0, None, None, None, None, None, 0, None) == 1
    b = ctypes.c_size_t(0)
    assert lib.snack_restructure_workspace_size(None, 0, ctypes.byref(b)) == 1
    lib.snack_destroy(None)  # allowed
    h = vp(0)
    # shape errors come before any CUDA call
    assert lib.snack_create(ctypes.byref(h), 0, 4, 0, 1, 0, 0, None, None, None, 0, None, 0, 0, None) == 1
    assert lib.snack_create(None, 4, 4, 0, 1, 0, 0, None, None, None, 0, None, 0, 0, None) == 1
    # missing buffers, misaligned plan, too-small plan: all host-side
    fake = vp(1 << 20)
    assert lib.snack_create(ctypes.byref(h), 4, 4, 2, 1, 0, 0, None, None, fake, 1 << 20, fake, 1 << 20, 0,
                            None) == 1
    odd = vp((1 << 20) + 8)
    assert lib.snack_create(ctypes.byref(h), 4, 4, 2, 1, 0, 0, fake, fake, odd, 1 << 20, fake, 1 << 20, 0,
                            None) == 1
    assert lib.snack_create(ctypes.byref(h), 4, 4, 2, 1, 0, 0, fake, fake, fake, 16, fake, 1 << 20, 0, None) == 4
    assert lib.snack_create(ctypes.byref(h), 4, 4, 2, 1, 0, 0, fake, fake, fake, 1 << 20, fake, 16, 0, None) == 4
    assert h.value is None


def test_trace_rejects_bad_arguments_on_the_host(lib):
    # capacity < 1, and a read without an open trace, fail before any CUDA call
    assert lib.snack_trace_start(0) == 1
    assert lib.snack_trace_start(-5) == 1
    assert lib.snack_trace_stop() == 0
    n = ctypes.c_int32(7)
    assert lib.snack_trace_read(None, None, 0, ctypes.byref(n)) == 1 and n.value == 0
    assert lib.snack_trace_read(None, None, 0, None) == 1
    assert lib.snack_trace_stop() == 0  # closing twice is fine
