"""GPU parity of the activation quantizer and the weight repack (bit-exact).

Quantized codes and scales must equal the oracle's byte for byte, in both
layouts; the packed weights must equal the oracle's layout statement.
"""

import numpy as np
import pytest
import torch

from oracle import mxfp4_ref as ref
from oracle import tile_layout as tl
from mxfp4_quantized_gemm_gb300 import synth
from helpers import dev_bf16, dev_u8, empty_u8, pack_weights, tiled_from_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


def quant_both(capi, x_bits, K, ldx=None):
    M = x_bits.shape[0]
    if ldx is not None and ldx != K:
        wide = np.zeros((M, ldx), np.uint16)
        wide[:, :K] = x_bits
        x = dev_bf16(wide)
    else:
        ldx = K
        x = dev_bf16(x_bits)
    out = {}
    for layout in (capi.LAYOUT_ROWMAJOR, capi.LAYOUT_TILED):
        c = empty_u8(capi.mxfp4_act_code_bytes(M, K, layout))
        s = empty_u8(capi.mxfp4_act_scale_bytes(M, K, layout))
        capi.mxfp4_quant_act(x, M, K, ldx, c, s, layout)
        torch.cuda.synchronize()
        out[layout] = (c.cpu().numpy(), s.cpu().numpy())
    return out


CASES = [
    # (M, K, outliers, edge rows)  -- shapes of the five workloads
    (16, 5120, 0.0, False),      # synthetic GEMM (16, 1024, 5120)
    (64, 14336, 0.01, False),    # decode sweep, outlier channels
    (4, 5120, 0.01, False),
    (2, 5120, 0.0, True),        # edge / tail cases
    (3, 5120, 0.0, True),
    (17, 5120, 0.0, True),
    (64, 5120, 0.0, True),
    (1, 5120, 0.0, True),
    (16, 5152, 0.0, True),
    (8193, 5152, 0.0, True),
    (5, 40, 0.0, True),          # K not a multiple of 32
    (130, 96, 0.0, True),
]


@pytest.mark.parametrize("M,K,outl,edge", CASES)
def test_quant_bit_exact(capi, M, K, outl, edge):
    x = synth.activations(M, K, seed=M + K, outlier_frac=outl)
    if edge:
        x = synth.with_edge_rows(x, seed=M)
    got = quant_both(capi, x, K)
    c_ref, s_ref = ref.quantize_mxfp4(ref.bf16_bits_to_f64(x))
    c_rm, s_rm = got[capi.LAYOUT_ROWMAJOR]
    assert np.array_equal(c_rm.reshape(M, K // 2), c_ref)
    assert np.array_equal(s_rm.reshape(M, -1), s_ref)
    tc, ts = tiled_from_oracle(c_ref, s_ref, K)
    c_t, s_t = got[capi.LAYOUT_TILED]
    assert np.array_equal(c_t, tc)
    assert np.array_equal(s_t, ts)


def test_quant_leading_dimension(capi):
    M, K = 9, 320
    x = synth.with_edge_rows(synth.activations(M, K, seed=7), seed=7)
    got = quant_both(capi, x, K, ldx=K + 24)
    c_ref, s_ref = ref.quantize_mxfp4(ref.bf16_bits_to_f64(x))
    assert np.array_equal(got[capi.LAYOUT_ROWMAJOR][0].reshape(M, -1), c_ref)
    assert np.array_equal(got[capi.LAYOUT_ROWMAJOR][1].reshape(M, -1), s_ref)


def test_quant_nonfinite_blocks(capi):
    M, K = 2, 64
    x = synth.activations(M, K, seed=3)
    x[0, 5] = 0x7F80      # +Inf in block 0 of row 0
    x[1, 40] = 0x7FC1     # NaN in block 1 of row 1
    got = quant_both(capi, x, K)
    c_ref, s_ref = ref.quantize_mxfp4(ref.bf16_bits_to_f64(x))
    assert s_ref[0, 0] == 0xFF and s_ref[1, 1] == 0xFF
    assert np.array_equal(got[capi.LAYOUT_ROWMAJOR][0].reshape(M, -1), c_ref)
    assert np.array_equal(got[capi.LAYOUT_ROWMAJOR][1].reshape(M, -1), s_ref)


@pytest.mark.parametrize("B,N,K", [(1, 1000, 5152), (1, 128, 5120), (1, 1024, 5120), (3, 512, 192),
                                   (2, 256, 512), (1, 5, 40), (1, 14336, 5120)])
def test_pack_bit_exact(capi, B, N, K):
    codes = synth.weight_codes(N, K, seed=N, batch=B)
    scales = synth.weight_scales(N, K, -8, 2, seed=N, batch=B)
    packed = pack_weights(capi, codes, scales, K)
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), tl.pack_weights_batched(codes, scales, K))
