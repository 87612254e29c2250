"""CPU checks of the C ABI: the library builds, loads, and exports every
entry point declared in include/moe.h; host-side argument checks work
without a GPU (no compute call is made)."""
import ctypes
import os
import re

import pytest

from helpers import ROOT, build_lib


@pytest.fixture(scope="module")
def lib_path():
    return build_lib()


def _declared():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        src = f.read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


def test_header_declares_the_entry_points():
    """The calls of the boundary: init, workspace sizing, routing, permute,
    group-aware quantization, the grouped GEMM (fwd, dgrad, wgrad), combine
    and the two backward helpers."""
    names = set(_declared())
    for n in ("moe_init", "moe_workspace_size", "moe_route_topk", "moe_permute", "mxfp8_group_quantize",
              "grouped_gemm_mxfp8", "moe_unpermute_combine", "moe_combine_bwd", "moe_route_bwd",
              "mxfp8_scale_layout", "mxfp8_group_quantize_ex"):
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_matches_header(lib_path):
    from grouped_gemm_top_gb300 import ops
    assert set(ops.EXPORTS) == set(_declared())
    assert ops.moe_abi_version() == 200


def test_host_only_calls_and_argument_checks(lib_path):
    from grouped_gemm_top_gb300 import ops
    lib = ops.lib
    assert ops.moe_row_capacity(256, 8, 2) == 1536            # ceil128(512 + 127*8)
    assert ops.moe_row_capacity(24576, 256, 8) == 229120
    assert ops.moe_row_capacity(1, 8, 2) == 256               # 2 pairs: at most 2 groups of 128 rows
    assert ops.moe_route_workspace_size(24576, 256) == 192 * 256 * 4
    # moe_workspace_size dispatches over the calls: only routing and permute take one
    assert ops.moe_workspace_size(ops.MOE_OP_ROUTE_TOPK, 24576, 7168, 256, 8, 2048) == 192 * 256 * 4
    assert ops.moe_workspace_size(ops.MOE_OP_PERMUTE, 24576, 7168, 256, 8, 2048) == \
        ops.moe_permute_workspace_size(24576, 256)
    for op in (ops.MOE_OP_GROUP_QUANTIZE, ops.MOE_OP_GATHER_QUANTIZE, ops.MOE_OP_GROUPED_GEMM,
               ops.MOE_OP_UNPERMUTE_COMBINE, ops.MOE_OP_COMBINE_BWD, ops.MOE_OP_ROUTE_BWD):
        assert ops.moe_workspace_size(op, 24576, 7168, 256, 8, 2048) == 0
    assert ops.moe_workspace_size(99, 256, 512, 8, 2, 256) == -1
    assert ops.moe_workspace_size(ops.MOE_OP_ROUTE_TOPK, 256, 512, 0, 2, 256) == -1
    assert ops.status_string(ops.MOE_ERR_BAD_OFFSETS).startswith("group offsets")
    # NULL pointers / bad sizes are rejected before any device work
    st = lib.moe_route_topk(None, 16, 8, 2, 0, 1, None, None, None, None, None, 0, None, None)
    assert st == ops.MOE_ERR_INVALID_ARG
    st = lib.moe_route_topk(None, 16, 8, 9, 0, 1, None, None, None, None, None, 0, None, None)
    assert st == ops.MOE_ERR_INVALID_ARG
    st = lib.mxfp8_group_quantize(ctypes.c_void_p(16), 100, 128, 0, None, 0, ctypes.c_void_p(16),
                                  ctypes.c_void_p(16), None, None)
    assert st == ops.MOE_ERR_UNSUPPORTED                       # rows % 128 != 0
    st = lib.grouped_gemm_mxfp8(0, ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                ctypes.c_void_p(16), 0, ctypes.c_void_p(16), 4, 256, 200, 256, 0, None,
                                ctypes.c_void_p(16), None, None, None)
    assert st == ops.MOE_ERR_UNSUPPORTED                       # N % 256 != 0
    st = lib.grouped_gemm_mxfp8(0, ctypes.c_void_p(8), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                ctypes.c_void_p(16), 0, ctypes.c_void_p(16), 4, 256, 256, 256, 0, None,
                                ctypes.c_void_p(16), None, None, None)
    assert st == ops.MOE_ERR_ALIGNMENT
    # the gathered quantization writes rowwise codes as 32-byte sectors:
    # a 16-byte aligned codes_row is refused
    st = lib.mxfp8_gather_quantize(ctypes.c_void_p(64), 256, 128, 1, None, None, ctypes.c_void_p(64), 1, 256,
                                   ctypes.c_void_p(48), ctypes.c_void_p(64), None, None, None, None)
    assert st == ops.MOE_ERR_ALIGNMENT
    # kernel options out of range are refused before anything else runs
    bad = ops.gemm_opts("pair")
    bad.kernel = 9
    st = lib.grouped_gemm_mxfp8_ex(0, ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                   ctypes.c_void_p(16), 0, ctypes.c_void_p(16), 4, 256, 256, 256, 0, None,
                                   ctypes.c_void_p(16), None, ctypes.byref(bad), None, None)
    assert st == ops.MOE_ERR_INVALID_ARG
    # the weight-gradient group filter: lo, hi >= 0; only WGRAD
    for lo, hi in ((-1, 0), (0, -512)):
        bad = ops.gemm_opts("auto", wgrad_rows=(lo, hi))
        st = lib.grouped_gemm_mxfp8_ex(2, ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                       ctypes.c_void_p(16), 0, ctypes.c_void_p(16), 4, 256, 256, 256, 0, None,
                                       ctypes.c_void_p(16), None, ctypes.byref(bad), None, None)
        assert st == ops.MOE_ERR_INVALID_ARG, (lo, hi)
    fwd_filter = ops.gemm_opts("auto", wgrad_rows=(0, 512))
    st = lib.grouped_gemm_mxfp8_ex(0, ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                   ctypes.c_void_p(16), 0, ctypes.c_void_p(16), 4, 256, 256, 256, 0, None,
                                   ctypes.c_void_p(16), None, ctypes.byref(fwd_filter), None, None)
    assert st == ops.MOE_ERR_UNSUPPORTED
    # both columnwise scale layouts: accepted by the fused quantizers (the
    # call then stops at the next check, rows % 128 != 0), refused by the
    # plain one.  Every call here must fail before any device work, also in
    # a process that has initialised the library: the pointers are fake.
    p64 = ctypes.c_void_p(64)
    for layout, want in ((ops.MOE_SF_TILE224_AND_ATOMS, ops.MOE_ERR_UNSUPPORTED),
                         (ops.MOE_SF_CANONICAL, ops.MOE_ERR_INVALID_ARG)):
        st = lib.mxfp8_gather_quantize_ex(p64, 100, 128, 1, None, None, p64, 1, 100, p64, p64, p64, p64, layout,
                                          None, None)
        assert st == want, layout
    st = lib.mxfp8_group_quantize_ex(ctypes.c_void_p(16), 128, 128, ops.MOE_QUANT_ROWWISE, None, 0,
                                     ctypes.c_void_p(16), ctypes.c_void_p(16), None,
                                     ops.MOE_SF_TILE224_AND_ATOMS, None, None)
    assert st == ops.MOE_ERR_INVALID_ARG
    assert ops.col_sf_bytes(ops.MOE_SF_TILE224_AND_ATOMS, 256, 448) == 2 * 2 * 1024 + 256 * 14
    st = lib.mxfp8_scale_layout(ctypes.c_void_p(16), 100, 128, 1, ctypes.c_void_p(16), None)
    assert st == ops.MOE_ERR_UNSUPPORTED                       # rows % 128 != 0
    st = lib.moe_hbm_fill(ctypes.c_void_p(16), 24, 0, 0, None)
    assert st == ops.MOE_ERR_UNSUPPORTED                       # bytes % 16 != 0
    p16 = ctypes.c_void_p(16)
    st = lib.mxfp8_group_quantize_ex(p16, 128, 128, ops.MOE_QUANT_ROWWISE, None, 0, p16, p16, None, 7, None, None)
    assert st == ops.MOE_ERR_INVALID_ARG                       # unknown scale layout
    st = lib.mxfp8_group_quantize_ex(p16, 128, 128, ops.MOE_QUANT_COLWISE_GROUPED, None, 1, p16, p16, p16,
                                     ops.MOE_SF_CANONICAL, None, None)
    assert st == ops.MOE_ERR_INVALID_ARG                       # padded offsets of a grouped axis need gofs


def test_no_environment_variables_in_the_library():
    """Kernel variants are chosen per call (moe_gemm_opts_t), never by the
    environment: no getenv in the CUDA sources."""
    csrc = os.path.join(ROOT, "grouped_gemm_top_gb300", "csrc")
    for fn in os.listdir(csrc):
        with open(os.path.join(csrc, fn)) as f:
            assert "getenv" not in f.read(), fn


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "grouped_gemm_top_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, fn)) as f:
                    src = f.read()
                assert "oracle" not in re.sub(r"#.*|//.*", "", src).lower() or fn == "__init__.py", fn
