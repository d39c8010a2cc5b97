"""The C-ABI library builds, loads, exports every declared symbol, and checks
its arguments on the host (CPU only: no compute call is made)."""

import os
import re

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import build
    build.build()
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b((?:mxfp4|a16wfp4)_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_path(capi):
    names = declared_functions()
    for must in ("mxfp4_pack_weights", "mxfp4_quant_act", "mxfp4_gemm", "a16wfp4_bmm"):
        assert must in names


def test_every_declared_symbol_is_exported(capi):
    for name in declared_functions():
        assert hasattr(capi.lib, name), name


def test_every_declared_symbol_has_a_binding(capi):
    # the thin binding carries the header's names (size queries and calls alike)
    for name in declared_functions():
        assert callable(getattr(capi, name, None)), name


def test_abi_version_and_status_strings(capi):
    assert capi.mxfp4_abi_version() == 3
    for s in range(8):
        assert capi.mxfp4_status_string(s).startswith("MXFP4_")
    assert capi.mxfp4_status_string(99) == "MXFP4_ERR_UNKNOWN"


@pytest.mark.parametrize("B,N,K", [(1, 1024, 5120), (1, 1000, 5152), (64, 512, 192), (3, 5, 40)])
def test_packed_size_matches_layout_statement(capi, B, N, K):
    from oracle import tile_layout as tl
    assert capi.mxfp4_packed_weight_bytes(B, N, K) == B * tl.weight_packed_bytes(N, K)


def test_size_queries(capi):
    from oracle import tile_layout as tl
    assert capi.mxfp4_act_code_bytes(16, 5120, capi.LAYOUT_ROWMAJOR) == 16 * 2560
    assert capi.mxfp4_act_scale_bytes(16, 5120, capi.LAYOUT_ROWMAJOR) == 16 * 160
    assert capi.mxfp4_act_scale_bytes(3, 5152, capi.LAYOUT_ROWMAJOR) == 3 * 161
    assert capi.mxfp4_act_code_bytes(17, 5152, capi.LAYOUT_TILED) == tl.code_bytes(17, 5152)
    assert capi.mxfp4_act_scale_bytes(17, 5152, capi.LAYOUT_TILED) == tl.scale_bytes(17, 5152)
    for bad in [(0, 32), (4, 0), (4, 33), (-1, 32)]:
        assert capi.mxfp4_act_code_bytes(*bad, capi.LAYOUT_ROWMAJOR) == 0
    assert capi.mxfp4_act_code_bytes(4, 32, 7) == 0
    assert capi.mxfp4_packed_weight_bytes(0, 4, 32) == 0
    assert capi.mxfp4_packed_weight_bytes(1, 4, 31) == 0
    assert capi.mxfp4_gemm_workspace_bytes(16, 1024, 5120) >= tl.code_bytes(16, 5120) + tl.scale_bytes(16, 5120)
    assert capi.mxfp4_gemm_workspace_bytes(0, 1, 32) == 0


def test_argument_checks_precede_any_launch(capi):
    lib = capi.lib
    A = 1 << 20   # a 16-byte aligned fake address: never dereferenced, checks fail first
    # null pointers
    assert lib.mxfp4_pack_weights(None, A, 1, 4, 32, A, None) == capi.ERR_INVALID_ARG
    assert lib.mxfp4_quant_act(None, 4, 32, 32, A, A, 0, None) == capi.ERR_INVALID_ARG
    assert lib.a16wfp4_bmm(A, None, A, 1, 1, 1, 64, 0, None) == capi.ERR_INVALID_ARG
    # non-positive sizes, bad enums
    assert lib.mxfp4_quant_act(A, 0, 32, 32, A, A, 0, None) == capi.ERR_INVALID_ARG
    assert lib.mxfp4_quant_act(A, 4, 32, 32, A, A, 5, None) == capi.ERR_INVALID_ARG
    assert lib.a16wfp4_bmm(A, A, A, 1, 1, 1, 64, 3, None) == capi.ERR_INVALID_ARG
    # odd K, ld too small, K not a multiple of 64 for the BMM
    assert lib.mxfp4_pack_weights(A, A, 1, 4, 33, A, None) == capi.ERR_UNSUPPORTED_SHAPE
    assert lib.mxfp4_quant_act(A, 4, 32, 16, A, A, 0, None) == capi.ERR_UNSUPPORTED_SHAPE
    assert lib.a16wfp4_bmm(A, A, A, 1, 1, 1, 96, 0, None) == capi.ERR_UNSUPPORTED_SHAPE
    # misaligned
    assert lib.mxfp4_pack_weights(A, A, 1, 4, 32, A + 8, None) == capi.ERR_MISALIGNED
    assert lib.a16wfp4_bmm(A + 4, A, A, 1, 1, 1, 64, 0, None) == capi.ERR_MISALIGNED
    # gemm: both or neither activation forms, workspace too small
    ws = capi.mxfp4_gemm_workspace_bytes(4, 8, 64)
    assert lib.mxfp4_gemm(A, 64, A, A, 0, A, None, A, 8, 4, 8, 64, A, ws, None) == capi.ERR_INVALID_ARG
    assert lib.mxfp4_gemm(None, 0, None, None, 0, A, None, A, 8, 4, 8, 64, A, ws, None) == capi.ERR_INVALID_ARG
    assert lib.mxfp4_gemm(A, 64, None, None, 0, A, None, A, 8, 4, 8, 64, A, ws - 1, None) == capi.ERR_WORKSPACE
    assert lib.mxfp4_gemm(A, 64, None, None, 0, A, None, A, 8, 4, 8, 64, None, ws, None) == capi.ERR_WORKSPACE
    assert lib.mxfp4_gemm(A, 64, None, None, 0, A, None, A, 4, 4, 8, 64, A, ws, None) == capi.ERR_UNSUPPORTED_SHAPE
    assert lib.mxfp4_gemm(A, 64, None, None, 0, A + 2, None, A, 8, 4, 8, 64, A, ws, None) == capi.ERR_MISALIGNED


def test_mxfp4_out_gemm_argument_checks(capi):
    lib, A = capi.lib, 1 << 20
    ws = capi.mxfp4_gemm_workspace_bytes(4, 8, 64)
    f = lib.mxfp4_gemm_mxfp4_out
    assert f(A, 64, None, None, 0, A, None, None, A, 4, 8, 64, A, ws, None) == capi.ERR_INVALID_ARG
    assert f(A, 64, None, None, 0, A, None, A, None, 4, 8, 64, A, ws, None) == capi.ERR_INVALID_ARG
    assert f(A, 64, None, None, 0, None, None, A, A, 4, 8, 64, A, ws, None) == capi.ERR_INVALID_ARG
    assert f(A, 64, None, None, 0, A, None, A, A, 4, 7, 64, A, ws, None) == capi.ERR_UNSUPPORTED_SHAPE   # odd N
    assert f(A, 64, None, None, 0, A, None, A, A, 4, 8, 63, A, ws, None) == capi.ERR_UNSUPPORTED_SHAPE   # odd K
    assert f(A, 64, None, None, 0, A, None, A, A, 4, 8, 64, A, ws - 1, None) == capi.ERR_WORKSPACE
    assert f(A, 64, None, None, 0, A + 8, None, A, A, 4, 8, 64, A, ws, None) == capi.ERR_MISALIGNED
    if not torch.cuda.is_available():
        # unaligned outputs are accepted: the call gets as far as the device check
        assert f(A, 64, None, None, 0, A, None, A + 1, A + 3, 4, 8, 64, A, ws, None) in (capi.ERR_NO_DEVICE,
                                                                                        capi.ERR_CUDA)


def test_rmsnorm_quant_argument_checks(capi):
    lib, A = capi.lib, 1 << 20
    f = lib.mxfp4_rmsnorm_quant_act
    ok = (A, 64, None, 0, A, 1e-6, 4, 64, A, A, 1, None, 0, None)

    def call(**kw):
        names = ("x", "ldx", "res", "ldr", "gamma", "eps", "M", "K", "codes", "scales", "layout", "y", "ldy", "s")
        args = dict(zip(names, ok))
        args.update(kw)
        return f(*args.values())

    assert call(x=None) == capi.ERR_INVALID_ARG
    assert call(gamma=None) == capi.ERR_INVALID_ARG
    assert call(scales=None) == capi.ERR_INVALID_ARG
    assert call(M=0) == capi.ERR_INVALID_ARG
    assert call(eps=-1.0) == capi.ERR_INVALID_ARG
    assert call(eps=float("nan")) == capi.ERR_INVALID_ARG
    assert call(layout=2) == capi.ERR_INVALID_ARG
    assert call(K=63, ldx=64) == capi.ERR_UNSUPPORTED_SHAPE
    assert call(ldx=32) == capi.ERR_UNSUPPORTED_SHAPE
    assert call(res=A, ldr=8) == capi.ERR_UNSUPPORTED_SHAPE
    assert call(y=A, ldy=8) == capi.ERR_UNSUPPORTED_SHAPE
    assert call(x=A + 1) == capi.ERR_MISALIGNED
    assert call(gamma=A + 1) == capi.ERR_MISALIGNED
    assert call(codes=A + 4) == capi.ERR_MISALIGNED          # TILED wants 16-byte alignment
    if not torch.cuda.is_available():
        assert call(codes=A + 4, layout=0) in (capi.ERR_NO_DEVICE, capi.ERR_CUDA)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device answer")
def test_valid_call_without_device_reports_no_device(capi):
    A = 1 << 20
    st = capi.lib.mxfp4_quant_act(A, 4, 32, 32, A, A, 0, None)
    assert st in (capi.ERR_NO_DEVICE, capi.ERR_CUDA)


def test_noalloc_gemm_argument_checks(capi):
    lib, A = capi.lib, 1 << 20
    f = lib.mxfp4_gemm_noalloc
    cap = capi.mxfp4_gemm_noalloc_max_scratch_bytes()
    assert cap == 48 << 20
    assert f(None, 64, A, None, A, 8, 4, 8, 64, None) == capi.ERR_INVALID_ARG
    assert f(A, 64, None, None, A, 8, 4, 8, 64, None) == capi.ERR_INVALID_ARG
    assert f(A, 64, A, None, None, 8, 4, 8, 64, None) == capi.ERR_INVALID_ARG
    assert f(A, 64, A, None, A, 8, 0, 8, 64, None) == capi.ERR_INVALID_ARG
    # a problem whose scratch exceeds the fixed array is refused before any device use
    M, N, K = 8192, 34816, 5120
    assert capi.mxfp4_gemm_workspace_bytes(M, N, K) > cap
    assert f(A, K, A, None, A, N, M, N, K, None) == capi.ERR_WORKSPACE
    # a valid small call reaches the device query (only without a GPU: the
    # fake addresses must never reach a kernel)
    if not torch.cuda.is_available():
        assert f(A, 64, A, None, A, 8, 4, 8, 64, None) in (capi.ERR_NO_DEVICE, capi.ERR_CUDA)


def test_split_cat_argument_checks(capi):
    # checked on the host before any device work: group sizes and the outputs the groups need
    f = capi.lib.mxfp4_gemm_split_cat
    p = 1 << 20   # a 16-byte aligned stand-in address; the checks below return before using it
    common = (p, 64, None, None, 0, p, None, 4, 256, 64)
    assert f(*common, 0, 0, None, 0, p, p, p, 1 << 20, None) == capi.ERR_INVALID_ARG      # s1 + s2 == 0
    assert f(*common, -8, 16, None, 0, p, p, p, 1 << 20, None) == capi.ERR_INVALID_ARG    # negative
    assert f(*common, 8, 8, None, 8, p, p, p, 1 << 20, None) == capi.ERR_INVALID_ARG      # s3 > 0 without z
    assert f(*common, 8, 8, p, 8, None, p, p, 1 << 20, None) == capi.ERR_INVALID_ARG      # no cat output
    assert f(*common, 8, 8, None, 0, p, None, p, 1 << 20, None) == capi.ERR_INVALID_ARG   # no split output
    assert f(*common, 4, 12, None, 0, p, p, p, 1 << 20, None) == capi.ERR_UNSUPPORTED_SHAPE   # not multiples of 8
    assert f(*common, 48, 48, None, 0, p, p, p, 1 << 20, None) == capi.ERR_UNSUPPORTED_SHAPE  # N % 96 != 0
    assert f(*common, 8, 8, p + 8, 8, p, p, p, 1 << 20, None) == capi.ERR_MISALIGNED     # z misaligned
