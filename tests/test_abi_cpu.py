"""The C-ABI library without a GPU: it builds, loads, exports every entry point
declared in include/tri_attn.h, and rejects bad arguments before touching CUDA.
Also checks that the product package never reaches the CPU oracle."""
import ctypes
import os
import re

import pytest

from pair_representation_triangular_gb300 import binding as tb
from pair_representation_triangular_gb300 import build as tbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    tbuild.build()
    return tb.load_library()


def test_exports_every_declared_entry_point(lib):
    names = tb.exported_names()
    assert "tri_attn_create" in names and "tri_attn_forward" in names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/tri_attn.h but not exported"


def test_status_strings(lib):
    assert tb.tri_attn_status_string(tb.TRI_ATTN_OK) == "ok"
    assert "timed out" in tb.tri_attn_status_string(tb.TRI_ATTN_ERR_DEVICE_TIMEOUT)
    assert tb.tri_attn_status_string(99) == "unknown status"


def _create(lib, B, N, D, h, dtype, mode=0, ptr=16, out=True):
    handle = ctypes.c_void_p()
    args = [ctypes.byref(handle) if out else None, B, N, D, h, dtype, mode] + [ptr] * 10 + [None]
    return lib.tri_attn_create(*args)


def test_create_rejects_bad_arguments_before_cuda(lib):
    assert _create(lib, 1, 8, 64, 4, 0, out=False) == tb.TRI_ATTN_ERR_INVALID_ARG
    assert _create(lib, 1, 8, 65, 4, 0) == tb.TRI_ATTN_ERR_INVALID_ARG      # D % h
    assert _create(lib, 0, 8, 64, 4, 0) == tb.TRI_ATTN_ERR_INVALID_ARG      # B < 1
    assert _create(lib, 1, 0, 64, 4, 0) == tb.TRI_ATTN_ERR_INVALID_ARG      # N < 1
    assert _create(lib, 1, 8, 64, 4, 7) == tb.TRI_ATTN_ERR_INVALID_ARG      # dtype
    assert _create(lib, 1, 8, 64, 4, 0, mode=4) == tb.TRI_ATTN_ERR_INVALID_ARG   # unknown bit
    assert _create(lib, 1, 8, 64, 4, 0, mode=-1) == tb.TRI_ATTN_ERR_INVALID_ARG
    assert _create(lib, 1, 8, 64, 4, 0, ptr=0) == tb.TRI_ATTN_ERR_INVALID_ARG  # NULL weights
    assert _create(lib, 1, 8, 64, 4, 0, ptr=24) == tb.TRI_ATTN_ERR_INVALID_ARG  # misaligned
    assert _create(lib, 1, 8, 512, 4, 0) == tb.TRI_ATTN_ERR_UNSUPPORTED     # f32 D > 256
    assert _create(lib, 1, 8, 33, 3, 0) == tb.TRI_ATTN_ERR_UNSUPPORTED      # f32 odd D
    assert _create(lib, 1, 8, 512, 4, 1) == tb.TRI_ATTN_ERR_UNSUPPORTED     # bf16 D > 256
    assert _create(lib, 1, 8, 33, 3, 1) == tb.TRI_ATTN_ERR_UNSUPPORTED      # bf16 odd D


# bf16 runs on the tensor-core kernels alone: D in {32, 64, 128} and
# d = D / h in {16, 32, 64}. Every other bf16 shape is refused before any CUDA
# call (there is no other bf16 backend); fp32 handles of those shapes are taken.
BF16_SHAPES = [(32, 2), (32, 1), (64, 4), (64, 2), (64, 1), (128, 8), (128, 4), (128, 2)]
BF16_REFUSED = [(96, 3), (96, 2), (128, 1), (256, 4), (64, 8), (32, 4), (48, 3), (128, 16), (16, 1)]


@pytest.mark.parametrize("D,h", BF16_REFUSED)
def test_bf16_shapes_outside_the_tensor_core_set_are_refused(lib, D, h):
    assert _create(lib, 1, 8, D, h, tb.TRI_ATTN_BF16) == tb.TRI_ATTN_ERR_UNSUPPORTED
    with pytest.raises(tb.TriAttnError) as e:
        tb.tri_attn_workspace_bytes(1, 8, D, h, tb.TRI_ATTN_BF16)
    assert e.value.status == tb.TRI_ATTN_ERR_UNSUPPORTED
    if D <= 256 and D // h <= 128 and D % 2 == 0:
        assert tb.tri_attn_workspace_bytes(1, 8, D, h, tb.TRI_ATTN_F32) > 0


@pytest.mark.parametrize("D,h", BF16_SHAPES)
def test_bf16_tensor_core_shapes_are_accepted(lib, D, h):
    n = tb.tri_attn_workspace_bytes(2, 40, D, h, tb.TRI_ATTN_BF16)
    cells = 2 * 40 * 40
    assert n >= 5 * cells * D * 2 + 2 * h * 40 * 40 * (4 + 2)


def test_null_handle_calls(lib):
    assert lib.tri_attn_forward(None, None, 16, 16, 16) == tb.TRI_ATTN_ERR_INVALID_ARG
    assert lib.tri_attn_forward_host(None, None, 16, 16, 16) == tb.TRI_ATTN_ERR_INVALID_ARG
    assert lib.tri_attn_sync_check(None, None) == tb.TRI_ATTN_ERR_INVALID_ARG
    assert lib.tri_attn_set_wait_limit(None, 5) == tb.TRI_ATTN_ERR_INVALID_ARG
    assert lib.tri_attn_destroy(None) == tb.TRI_ATTN_OK


def test_workspace_bytes(lib):
    n = tb.tri_attn_workspace_bytes(2, 32, 64, 4, tb.TRI_ATTN_F32)
    cells = 2 * 32 * 32
    assert n >= 5 * cells * 64 * 4 + 2 * 4 * 32 * 32 * 4
    with pytest.raises(tb.TriAttnError):
        tb.tri_attn_workspace_bytes(2, 32, 65, 4, tb.TRI_ATTN_F32)


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "pair_representation_triangular_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, f)) as fh:
                    src = fh.read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "tri_attn_oracle" not in src, f
