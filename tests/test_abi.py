"""The C-ABI library: it loads, exports every declared entry point, and its
host-side validation works without a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import software_pipelined_gb300 as g
from software_pipelined_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return g.load()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        names += re.findall(r"GEMM_F32_API\s+[\w\s\*]+?\b(gemm_f32_\w+)\s*\(", text)
    return names


def test_header_declares_the_binding_names():
    assert set(declared_functions()) == set(g.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_version(lib):
    assert g.gemm_f32_status_string(0) == "GEMM_F32_OK"
    assert g.gemm_f32_status_string(4) == "GEMM_F32_ERR_TIMEOUT"
    assert g.gemm_f32_status_string(99) == "GEMM_F32_ERR_UNKNOWN"
    assert g.gemm_f32_version() >= 101


def test_opts_layout_matches_header(lib):
    # int32 x6, int64, int32 x10 -> 6*4 + 8 + 10*4 = 72 bytes
    assert ctypes.sizeof(g.Opts) == 72
    o = g.gemm_f32_opts_init()
    assert o.variant == 0 and o.split_k == 0 and o.wait_timeout_cycles == 0


@pytest.mark.parametrize("dims", [
    (-1, 4, 4, 4, 4, 4),      # negative M
    (4, -1, 4, 4, 4, 4),
    (4, 4, -1, 4, 4, 4),
    (4, 4, 8, 7, 4, 4),       # lda < K
    (4, 8, 4, 4, 7, 8),       # ldb < N
    (4, 8, 4, 4, 8, 7),       # ldc < N
    (4, 4, 4, 0, 4, 4),       # ld < 1
    (1 << 31, 4, 4, 4, 4, 4),  # beyond the size limit
])
def test_plan_rejects_bad_dims(lib, dims):
    s, h = g.gemm_f32_plan(*dims)
    assert s == g.ERR_INVALID_ARG and h is None


def test_plan_rejects_bad_options(lib):
    for field, value in [("variant", 7), ("variant", 5), ("split_k", 65), ("tf32_terms", 2), ("stages", -1),
                         ("wait_timeout_cycles", -5), ("operand_split", 6), ("tile_group", 65),
                         ("host_panels", 65), ("host_panels", -1), ("split_reduce", 5), ("split_reduce", -1), ("k_slices", 3), ("k_slices", 8),
                         ("host_col_blocks", -1), ("host_col_blocks", 17), ("simt_fragments", 2)]:
        o = g.gemm_f32_opts_init()
        setattr(o, field, value)
        s, h = g.gemm_f32_plan_ex(64, 64, 64, 64, 64, 64, o)
        assert s == g.ERR_INVALID_ARG and h is None, field


def test_null_out_pointer_rejected(lib):
    assert lib.gemm_f32_plan(4, 4, 4, 4, 4, 4, None) == g.ERR_INVALID_ARG


def test_empty_problem_plans_without_a_gpu(lib):
    s, h = g.gemm_f32_plan(0, 16, 16, 16, 16, 16)
    assert s == g.OK and h
    s, desc = g.gemm_f32_plan_describe(h)
    assert s == g.OK and desc.startswith("noop")
    assert g.gemm_f32_run(h, 0, 0, 0, 0) == g.OK
    assert g.gemm_f32_check(h, 0) == g.OK
    assert g.gemm_f32_plan_workspace_bytes(h) == 0
    g.gemm_f32_plan_destroy(h)


def test_null_plan_calls(lib):
    assert g.gemm_f32_run(None, 0, 0, 0, 0) == g.ERR_INVALID_ARG
    assert g.gemm_f32_run_host(None, 0, 0, 0, 0) == g.ERR_INVALID_ARG
    assert g.gemm_f32_check(None, 0) == g.ERR_INVALID_ARG
    assert lib.gemm_f32_plan_describe(None, None, 0) == g.ERR_INVALID_ARG
    g.gemm_f32_plan_destroy(None)


def test_real_problem_needs_a_gb300(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    s, h = g.gemm_f32_plan(64, 64, 64, 64, 64, 64)
    assert s == g.ERR_UNSUPPORTED and h is None


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    import software_pipelined_gb300 as mod
    fresh = importlib.util.spec_from_file_location("sp_fresh", mod.__file__)
    m = importlib.util.module_from_spec(fresh)
    fresh.loader.exec_module(m)
    with pytest.raises(RuntimeError, match="not built"):
        m.load(str(tmp_path / "missing.so"))


@pytest.mark.parametrize("args", [
    (8, 8, 8, 8, 8, 8, -1, 64, 64, 64),       # negative batch
    (8, 8, 8, 8, 8, 8, 65536, 64, 64, 64),    # beyond the grid limit
    (8, 8, 8, 8, 8, 8, 4, -64, 64, 64),       # negative stride
    (8, 8, 8, 8, 8, 8, 4, 64, 64, 63),        # outputs would overlap
])
def test_batched_plan_rejects_bad_args(lib, args):
    s, h = g.gemm_f32_plan_batched(*args, None)
    assert s == g.ERR_INVALID_ARG and h is None


def test_batched_plan_rejects_tensor_core_variant(lib):
    o = g.gemm_f32_opts_init()
    o.variant = g.VARIANT_TCGEN05
    s, h = g.gemm_f32_plan_batched(8, 8, 8, 8, 8, 8, 4, 64, 64, 64, o)
    assert s == g.ERR_UNSUPPORTED and h is None
