"""GPU parity of the GEMM with the MXFP4 output epilogue.

The epilogue quantizes the GEMM's own bf16 results (an integer decision taken
in the kernel's precision), so its codes and scales must equal the oracle
quantizer applied to mxfp4_gemm's bf16 output for the same inputs, bit for
bit.  That output is itself checked against the float64 oracle (2 bf16 ulp)
on sampled rows here and exhaustively in test_gpu_gemm.py, and the GEMM is
bit-reproducible run to run.  Shapes cover the decode kernel's whole-tile and
cluster split-K paths and the prefill kernel's whole-tile and stream-K
fix-up paths, with ragged N.
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


def problem(M, N, K, seed, with_bias, edge=False):
    x = synth.activations(M, K, seed=seed, outlier_frac=0.01)
    if edge:
        x = synth.with_edge_rows(x, seed=seed)
    wc = synth.weight_codes(N, K, seed=seed)
    ws = synth.weight_scales(N, K, -8, 0, seed=seed)
    b = synth.bias(N, seed=seed) if with_bias else None
    return x, wc, ws, b


def run_both(capi, x_bits, packed, b_bits, M, N, K, out_offset=0, pre=None):
    """bf16 output of mxfp4_gemm and (codes, scales) of mxfp4_gemm_mxfp4_out."""
    nbytes = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    bias = dev_bf16(b_bits) if b_bits is not None else None
    xd = dev_bf16(x_bits) if pre is None else None
    a_codes, a_scales, layout = pre if pre is not None else (None, None, 0)
    lda = K if pre is None else 0
    out = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    capi.mxfp4_gemm(xd, lda, a_codes, a_scales, layout, packed, bias, out, N, M, N, K,
                    gemm_workspace(capi, nbytes), nbytes)
    nb = -(-N // 32)
    cbuf = torch.full((out_offset + M * (N // 2),), 0xA5, dtype=torch.uint8, device="cuda")
    sbuf = torch.full((out_offset + M * nb,), 0xA5, dtype=torch.uint8, device="cuda")
    capi.mxfp4_gemm_mxfp4_out(xd, lda, a_codes, a_scales, layout, packed, bias, cbuf[out_offset:],
                              sbuf[out_offset:], M, N, K, gemm_workspace(capi, nbytes), nbytes)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    c = cbuf.cpu().numpy()
    s = sbuf.cpu().numpy()
    assert np.all(c[:out_offset] == 0xA5) and np.all(s[:out_offset] == 0xA5)
    return host_bits(out), c[out_offset:].reshape(M, N // 2), s[out_offset:].reshape(M, nb)


def check(capi, M, N, K, seed, with_bias=True, oracle_rows=None, edge=False, **kw):
    x, wc, ws, b = problem(M, N, K, seed, with_bias, edge)
    packed = pack_weights(capi, wc, ws, K)
    y, codes, scales = run_both(capi, x, packed, b, M, N, K, **kw)
    c_ref, s_ref = ref.quantize_mxfp4(ref.bf16_bits_to_f64(y))
    assert np.array_equal(scales, s_ref), f"scales differ in {int((scales != s_ref).sum())} places"
    assert np.array_equal(codes, c_ref), f"codes differ in {int((codes != c_ref).sum())} places"
    rows = np.arange(M) if oracle_rows is None else oracle_rows
    acc, mag = oracle_gemm_rows(x, rows, wc, ws, K, b)
    check_close(y[rows], acc, mag, -(-K // 64) + 4, what=f"M={M} N={N} K={K}")
    return x, wc, ws, b, packed, codes, scales


@pytest.mark.parametrize("M,N,K", [
    (1, 1000, 256), (4, 2048, 256),              # decode, one k-range per tile: whole-tile stores
    (1, 5120, 5120), (5, 1000, 5152),            # decode, cluster split-K sums
    (16, 14336, 5120), (33, 998, 2048), (64, 5120, 14336),
])
def test_decode_paths(capi, M, N, K):
    check(capi, M, N, K, seed=M + N + K)


@pytest.mark.parametrize("M,N,K", [(65, 1000, 2048), (300, 5120, 5120), (2048, 1024, 5120), (1000, 3000, 1536),
                                   (2432, 2040, 512)])     # 152 tiles: whole tiles per CTA, no fix-up
def test_prefill_paths(capi, M, N, K):
    check(capi, M, N, K, seed=M + N, oracle_rows=np.array([0, 1, M // 2, M - 1]))


def test_without_bias(capi):
    check(capi, 7, 1536, 4096, seed=3, with_bias=False)
    check(capi, 400, 1536, 4096, seed=4, with_bias=False, oracle_rows=np.array([0, 399]))


@pytest.mark.parametrize("M,N,K", [(24, 1000, 256), (24, 3000, 5120), (200, 3000, 2048)])
def test_edge_rows_without_bias(capi, M, N, K):
    """Rows of +0, of -0, of ties and of subnormals: a zero row's sums are
    signed zeros, and every store path must quantize the same bf16 values the
    bf16 output holds (no bias: nothing is added to them)."""
    check(capi, M, N, K, seed=M + K, with_bias=False, edge=True, oracle_rows=np.arange(min(M, 24)))


@pytest.mark.parametrize("M", [3, 200])
def test_unaligned_outputs(capi, M):
    check(capi, M, 1000, 1024, seed=M, out_offset=1, oracle_rows=np.array([0, M - 1]))


@pytest.mark.parametrize("M", [8, 130])
def test_prequantized_input(capi, M):
    N, K = 768, 2048
    x, wc, ws, b = problem(M, N, K, M, True)
    packed = pack_weights(capi, wc, ws, K)
    ac, asc = ref.quantize_mxfp4(ref.bf16_bits_to_f64(x))
    y, codes, scales = run_both(capi, x, packed, b, M, N, K, pre=(dev_u8(ac), dev_u8(asc), capi.LAYOUT_ROWMAJOR))
    c_ref, s_ref = ref.quantize_mxfp4(ref.bf16_bits_to_f64(y))
    assert np.array_equal(codes, c_ref) and np.array_equal(scales, s_ref)


@pytest.mark.parametrize("M", [4, 256])
def test_two_layers_chained(capi, M):
    """Layer 1's MXFP4 output fed to layer 2 as its pre-quantized input equals
    layer 2 quantizing layer 1's bf16 output itself."""
    N1, K1, N2 = 2048, 1024, 768
    x, wc, ws, b, packed, codes, scales = check(capi, M, N1, K1, seed=M, oracle_rows=np.array([0, M - 1]))
    wc2 = synth.weight_codes(N2, N1, seed=M + 1)
    ws2 = synth.weight_scales(N2, N1, -8, 0, seed=M + 1)
    packed2 = pack_weights(capi, wc2, ws2, N1)
    y1, _, _ = run_both(capi, x, packed, b, M, N1, K1)
    nbytes = capi.mxfp4_gemm_workspace_bytes(M, N2, N1)
    o_pre = torch.empty(M, N2, dtype=torch.bfloat16, device="cuda")
    o_bf = torch.empty(M, N2, dtype=torch.bfloat16, device="cuda")
    capi.mxfp4_gemm(None, 0, dev_u8(codes), dev_u8(scales), capi.LAYOUT_ROWMAJOR, packed2, None, o_pre, N2, M, N2,
                    N1, gemm_workspace(capi, nbytes), nbytes)
    capi.mxfp4_gemm(dev_bf16(y1), N1, None, None, 0, packed2, None, o_bf, N2, M, N2, N1,
                    gemm_workspace(capi, nbytes), nbytes)
    torch.cuda.synchronize()
    assert torch.equal(o_pre, o_bf)
