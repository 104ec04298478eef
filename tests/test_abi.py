"""The C-ABI library loads and exports every entry point the header declares;
host-side argument checks work without a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import bit_grouped_gemm_gb300 as bg
from bit_grouped_gemm_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_grouped_gemm_gb300 import build
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moe_w4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_plan_create", "moe_route", "moe_grouped_w4_ffn", "moe_forward_layer",
              "moe_plan_destroy", "moe_get_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert getattr(lib, name) is not None


def test_struct_layouts_match_header():
    # sizes of the POD structs as declared (ints and pointers only)
    assert ctypes.sizeof(bg.MoePlanDesc) == 11 * 4
    assert ctypes.sizeof(bg.MoeW4) == 3 * 8
    assert ctypes.sizeof(bg.MoeExperts) == 9 * 8
    assert ctypes.sizeof(bg.MoeRouting) == 10 * 8
    assert ctypes.sizeof(bg.MoeLayer) == 2 * 8 + 2 * 9 * 8


def test_version_and_strings(lib):
    assert bg.moe_version() >= 100
    assert bg.moe_status_string(0) == "ok"
    assert "timed out" in bg.moe_status_string(5)


def test_scratch_bytes_host_only(lib):
    d = bg.plan_desc(max_tokens=4096)
    n = bg.moe_plan_scratch_bytes(d)
    rows = 4096 * 9
    assert n >= rows * (2048 + 512 + 2048) * 2      # xs, act, d
    assert n < rows * (2048 + 512 + 2048) * 2 + 64 * 2 ** 20


@pytest.mark.parametrize("field,value,status", [
    ("hidden", 0, 1), ("group_size", 32, 2), ("block_m", 64, 2), ("hidden", 2112, 2),
    ("num_experts", 12, 2), ("top_k", 300, 1), ("max_tokens", -1, 1), ("gemm_path", 5, 1),
    ("top_k", 40, 2),
])
def test_invalid_descriptions_rejected_on_host(lib, field, value, status):
    d = bg.plan_desc()
    setattr(d, field, value)
    with pytest.raises(bg.MoeError) as ei:
        bg.moe_plan_scratch_bytes(d)
    assert ei.value.status == status
    with pytest.raises(bg.MoeError) as ei:
        bg.moe_plan_create(d, 0)
    assert ei.value.status == status


def test_null_arguments_rejected(lib):
    assert lib.moe_plan_create(None, 0, None) == 1
    assert lib.moe_route(None, None, 1, None, None, None, None) == 1
    assert lib.moe_forward_layer(None, None, 1, None, None, None, None, None, None) == 1
    assert lib.moe_forward_layer_residual(None, None, 1, None, None, None, None, 0.0, None, None,
                                          None) == 1
    assert lib.moe_forward_stack(None, None, None, 1, None, 1, 0.0, None) == 1
    assert lib.moe_get_error(None) == 1
    assert lib.moe_set_tail_split(None, 1) == 1


def test_noalloc_host_checks(lib):
    """moe_route_noalloc's size limits are checked on the host before any
    CUDA call: top_k above 32 is unsupported (as for a plan), T above 4096 or
    more than 512 experts exceed its fixed scratch."""
    fake = 1 << 20                                   # aligned, never dereferenced
    r = bg.MoeRouting(*([fake] * 10))
    call = lambda T, E, k: lib.moe_route_noalloc(fake, T, 2048, fake, None, E, k,
                                                 ctypes.byref(r), None)
    assert call(16, 64, 33) == 2                     # MOE_ERR_UNSUPPORTED
    assert call(4097, 256, 8) == 4                   # MOE_ERR_CAPACITY
    assert call(16, 520, 8) == 4
    assert call(0, 256, 8) == 1                      # MOE_ERR_INVALID_ARG
    assert call(16, 256, 0) == 1
