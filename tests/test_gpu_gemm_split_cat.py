"""GPU parity of the split + cat fused epilogue (mxfp4_gemm_split_cat).

The epilogue is the data movement of ``oracle.mxfp4_ref.split_cat`` applied to
the GEMM's own bf16 result: every output bit must equal the oracle's
rearrangement of mxfp4_gemm's bf16 output (and the copied z values), and that
bf16 output is itself compared with the float64 oracle within the GEMM
tolerance.  Covered: every store path (decode whole tiles and cluster-split
tiles, the decode kernel with more tiles than SMs, prefill whole tiles and the
stream-K fix-up), bf16 and pre-quantized activations, with and without bias,
z wider than a group, an empty concatenated part, an empty split part.
"""

import numpy as np
import pytest
import torch

from oracle import mxfp4_ref as ref
from mxfp4_quantized_gemm_gb300 import synth
from helpers import check_close, dev_bf16, dev_u8, gemm_workspace, host_bits, oracle_gemm_rows, pack_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


def run(capi, M, H, s1, s2, s3, K, seed, with_bias=True, prequant=False):
    N = H * (s1 + s2)
    x = synth.activations(M, K, seed=seed, outlier_frac=0.01)
    wc = synth.weight_codes(N, K, seed=seed)
    ws = synth.weight_scales(N, K, -6, 0, seed=seed)
    b = synth.bias(N, seed=seed) if with_bias else None
    z = synth.activations(M, H * s3, seed=seed + 1).reshape(M, H, s3) if s3 else np.zeros((M, H, 0), np.uint16)
    packed = pack_weights(capi, wc, ws, K)
    bias = dev_bf16(b) if b is not None else None
    wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    work = gemm_workspace(capi, wsb)
    if prequant:
        c_ref, s_ref = ref.quantize_mxfp4(ref.bf16_bits_to_f64(x))
        a = (None, 0, dev_u8(c_ref), dev_u8(s_ref), capi.LAYOUT_ROWMAJOR)
    else:
        a = (dev_bf16(x), K, None, None, 0)
    y = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    capi.mxfp4_gemm(*a, packed, bias, y, N, M, N, K, work, wsb)
    cat = torch.full((M, H, s1 + s3), float("nan"), dtype=torch.bfloat16, device="cuda")
    split = torch.full((M, H, s2), float("nan"), dtype=torch.bfloat16, device="cuda")
    zd = dev_bf16(z) if s3 else None
    capi.mxfp4_gemm_split_cat(*a, packed, bias, M, N, K, s1, s2, zd, s3, cat if s1 + s3 else None,
                              split if s2 else None, work, wsb)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    y_bits = host_bits(y)
    want_cat, want_split = ref.split_cat(y_bits, z, s1, s2)
    assert np.array_equal(host_bits(cat), want_cat)
    assert np.array_equal(host_bits(split), want_split)
    rows = np.unique(np.array([0, M // 2, M - 1]))
    acc, mag = oracle_gemm_rows(x, rows, wc, ws, K, b)
    check_close(y_bits[rows], acc, mag, -(-K // 64) + 4, what=f"split-cat GEMM M={M} N={N} K={K}", K=K)


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_decode_mla_shape(capi, M):
    # 16 heads of a 128-column part joined with 64 separately computed values and a 128-column part
    run(capi, M, 16, 128, 128, 64, 512, seed=M)


@pytest.mark.parametrize("M", [300, 2048, 2432])   # 2432: 152 tiles, whole tiles per CTA (no fix-up)
def test_prefill_mla_shape(capi, M):
    run(capi, M, 16, 128, 128, 64, 512, seed=M)


def test_more_tiles_than_sms(capi):
    run(capi, 4, 170, 128, 128, 64, 512, seed=5)


@pytest.mark.parametrize("M,H,s1,s2,s3,K", [(5, 40, 8, 8, 24, 256), (33, 12, 24, 40, 8, 1024),
                                            (70, 6, 0, 64, 16, 288), (3, 10, 32, 0, 0, 5120)])
def test_odd_groups(capi, M, H, s1, s2, s3, K):
    run(capi, M, H, s1, s2, s3, K, seed=M + H, with_bias=(M % 2 == 1))


@pytest.mark.parametrize("M", [2, 200])
def test_prequantized_input(capi, M):
    run(capi, M, 8, 64, 64, 32, 768, seed=90 + M, prequant=True)
