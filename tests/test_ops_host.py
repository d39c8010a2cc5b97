"""The torch.library operators on the host: shape-only fake kernels, graph
tracing, argument checks, and that their size arithmetic agrees with the
library's own size queries (no compute call is made)."""

import subprocess
import sys

import pytest
import torch
from torch.fx.experimental.proxy_tensor import make_fx

from mxfp4_quantized_gemm_gb300 import ops

BF, U8 = torch.bfloat16, torch.uint8


def meta(*shape, dtype=BF):
    return torch.empty(*shape, dtype=dtype, device="meta")


def packed_meta(batch, N, K):
    return meta(ops._packed_weight_bytes(batch, N, K), dtype=U8)


def test_importing_ops_does_not_load_the_library():
    code = ("import sys, mxfp4_quantized_gemm_gb300.ops as o, torch; "
            "assert hasattr(torch.ops.mxfp4, 'linear'); "
            "assert 'mxfp4_quantized_gemm_gb300.capi' not in sys.modules")
    subprocess.run([sys.executable, "-c", code], check=True, cwd=ops.__file__.rsplit("/", 2)[0])


@pytest.mark.parametrize("lead", [(7,), (2, 5), (1, 3, 4)])
def test_linear_flattens_leading_dims(lead):
    y = torch.ops.mxfp4.linear(meta(*lead, 1024), packed_meta(1, 300, 1024), meta(300), 300)
    assert y.shape == (*lead, 300) and y.dtype == BF


def test_prequant_and_bmm_shapes():
    M, N, K = 37, 520, 5120
    codes, scales = torch.ops.mxfp4.quant_act(meta(M, K), ops.LAYOUT_ROWMAJOR)
    assert codes.shape == (M, K // 2) and scales.shape == (M, K // 32) and codes.dtype == U8
    y = torch.ops.mxfp4.linear_prequant(codes, scales, ops.LAYOUT_ROWMAJOR, packed_meta(1, N, K), None, M, N, K)
    assert y.shape == (M, N)
    x = meta(16, 40, 512)
    assert torch.ops.mxfp4.a16wfp4_bmm(x, packed_meta(16, 128, 512), 128, False).shape == (16, 40, 128)
    assert torch.ops.mxfp4.a16wfp4_bmm(x, packed_meta(16, 128, 512), 128, True).shape == (40, 16, 128)


def test_rmsnorm_quant_shapes():
    c, s = torch.ops.mxfp4.rmsnorm_quant_act(meta(2, 3, 5120), meta(5120), 1e-6, ops.LAYOUT_TILED, meta(2, 3, 5120))
    assert c.numel() == 128 * 5120 // 2 and s.numel() == 128 * 5120 // 32
    c, s = torch.ops.mxfp4.rmsnorm_quant_act(meta(7, 100), meta(100), 1e-6, ops.LAYOUT_ROWMAJOR, None)
    assert c.shape == (7, 50) and s.shape == (7, 4)


def test_linear_mxfp4_out_shapes():
    c, s = torch.ops.mxfp4.linear_mxfp4_out(meta(2, 5, 1024), packed_meta(1, 1000, 1024), None, 1000)
    assert c.shape == (10, 500) and s.shape == (10, 32) and c.dtype == U8
    with pytest.raises(RuntimeError, match="even"):
        torch.ops.mxfp4.linear_mxfp4_out(meta(2, 1024), packed_meta(1, 999, 1024), None, 999)


def test_linear_split_cat_shapes():
    cat, split = torch.ops.mxfp4.linear_split_cat(meta(3, 512), packed_meta(1, 16 * 256, 512), None,
                                                  meta(3, 16, 64), 128, 128)
    assert cat.shape == (3, 16, 192) and split.shape == (3, 16, 128) and cat.dtype == BF
    cat, split = torch.ops.mxfp4.linear_split_cat(meta(2, 4, 256), packed_meta(1, 5 * 16, 256), None,
                                                  meta(8, 5, 0), 8, 8)
    assert cat.shape == (8, 5, 8) and split.shape == (8, 5, 8)
    with pytest.raises(RuntimeError, match="multiples of 8"):
        torch.ops.mxfp4.linear_split_cat(meta(3, 512), packed_meta(1, 16 * 20, 512), None, meta(3, 16, 8), 4, 16)
    with pytest.raises(RuntimeError, match="rows"):
        torch.ops.mxfp4.linear_split_cat(meta(3, 512), packed_meta(1, 16 * 16, 512), None, meta(4, 16, 8), 8, 8)


def test_pack_weights_shape():
    w = torch.ops.mxfp4.pack_weights(meta(3, 300, 256, dtype=U8), meta(3, 300, 16, dtype=U8), 512)
    assert w.numel() == 3 * 2 * 2 * 34816


def test_make_fx_records_the_operator():
    def layer(x, w, b):
        return torch.nn.functional.silu(torch.ops.mxfp4.linear(x, w, b, 300))

    g = make_fx(layer, tracing_mode="symbolic")(meta(2, 5, 1024), packed_meta(1, 300, 1024), meta(300))
    targets = [n.target for n in g.graph.nodes if n.op == "call_function"]
    assert torch.ops.mxfp4.linear.default in targets


def test_argument_checks():
    with pytest.raises(RuntimeError, match="must be torch.bfloat16"):
        torch.ops.mxfp4.linear(meta(4, 1024, dtype=torch.float32), packed_meta(1, 300, 1024), None, 300)
    with pytest.raises(RuntimeError, match="bytes"):
        torch.ops.mxfp4.linear(meta(4, 1024), packed_meta(1, 256, 1024), None, 300)
    with pytest.raises(RuntimeError, match="even"):
        torch.ops.mxfp4.linear(meta(4, 1023), packed_meta(1, 300, 1024), None, 300)
    # host memory must never reach the kernels
    with pytest.raises(RuntimeError, match="not a CUDA device"):
        torch.ops.mxfp4.a16wfp4_bmm(torch.zeros(2, 3, 64, dtype=BF), torch.zeros(2 * 34816, dtype=U8), 128, False)


def test_size_checks_keep_kernels_in_bounds():
    w = packed_meta(1, 300, 1024)
    with pytest.raises(RuntimeError, match="bias"):
        torch.ops.mxfp4.linear(meta(4, 1024), w, meta(299), 300)
    with pytest.raises(RuntimeError, match="needed"):
        torch.ops.mxfp4.linear_prequant(meta(4, 511, dtype=U8), meta(4, 32, dtype=U8), 0, w, None, 4, 300, 1024)
    with pytest.raises(RuntimeError, match="do not hold"):
        torch.ops.mxfp4.pack_weights(meta(300, 256, dtype=U8), meta(300, 32, dtype=U8), 1024)
    with pytest.raises(RuntimeError, match="leading"):
        torch.ops.mxfp4.pack_weights(meta(300, 512, dtype=U8), meta(301, 32, dtype=U8), 1024)
    with pytest.raises(RuntimeError, match="gamma"):
        torch.ops.mxfp4.rmsnorm_quant_act(meta(4, 1024), meta(1000), 1e-6, 0, None)
    with pytest.raises(RuntimeError, match="bias"):
        torch.ops.mxfp4.linear_mxfp4_out(meta(4, 1024), w, meta(301), 300)


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import build
    build.build()
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


@pytest.mark.parametrize("B,N,K", [(1, 1, 2), (1, 300, 1000), (64, 512, 192), (1, 34816, 5120), (3, 257, 4097 + 1)])
def test_packed_size_matches_library(capi, B, N, K):
    assert ops._packed_weight_bytes(B, N, K) == capi.mxfp4_packed_weight_bytes(B, N, K)


@pytest.mark.parametrize("M,K", [(1, 2), (5, 100), (130, 5120), (8193, 14336)])
@pytest.mark.parametrize("layout", [0, 1])
def test_activation_sizes_match_library(capi, M, K, layout):
    assert ops._act_bytes(M, K, layout) == (capi.mxfp4_act_code_bytes(M, K, layout),
                                            capi.mxfp4_act_scale_bytes(M, K, layout))
