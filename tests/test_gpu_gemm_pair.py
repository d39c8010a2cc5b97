"""GPU parity of the CTA-pair GEMM kernel (mxfp4_diag_gemm_pair: 256 x 256 tiles on 2-CTA clusters).

mxfp4_gemm never runs this kernel (measured no faster than the single-CTA
one); the diagnostic entry point runs it where it applies: M > 64, the
128-row activation tiles pair up (an even count, or at least 16) and the
last wave of 256-row pair tiles over the device's co-resident pairs (76 on a
152-SM GB300) is at most 8% idle.  Every shape here meets that rule.  Each
pair's second CTA holds rows 128..255 of a tile and half of its weight rows,
so the checks cover rows on both sides of every 128-row boundary, ragged M,
N and K, both scale paths (activation scales kept in TMEM across tiles for
K <= 5120, copied every k-step above), a change of activation row tile
inside one pair's run of tiles, and a last pair tile whose second half lies
past M.  Where mxfp4_gemm's own kernel also takes whole tiles (no stream-K
parts summed afterwards) the two outputs are equal bit for bit: both kernels
then add the same fp32 products in the same order.
"""

import numpy as np
import pytest
import torch

from oracle import mxfp4_ref as ref
from helpers import (check_close, dev_bf16, dev_u8, gemm_workspace, host_bits, oracle_gemm_rows, pack_weights,
                     sample_rows, tiled_from_oracle)
from test_gpu_gemm import make_problem, n_acc, run_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


def run_pair(capi, x_bits, packed, bias_bits, M, N, K, pre=None):
    out = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    bias = dev_bf16(bias_bits) if bias_bits is not None else None
    a = (dev_bf16(x_bits), K, None, None, 0) if pre is None else (None, 0) + pre
    capi.mxfp4_diag_gemm_pair(*a, packed, bias, out, N, M, N, K, gemm_workspace(capi, wsb), wsb)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    return host_bits(out)


def library_takes_whole_tiles(M, N, K):
    """The single-CTA kernel's rule: whole tiles per CTA when there are at least as many tiles as
    CTAs and under 8% of the last wave is idle."""
    tiles = -(-M // 128) * -(-N // 256)
    grid = min(torch.cuda.get_device_properties(0).multi_processor_count, 256, tiles * -(-K // 256))
    waves = tiles / grid
    return tiles >= grid and (-(-tiles // grid) - waves) / waves < 0.08


def check(capi, M, N, K, seed, rows=None, **kw):
    x, wc, ws, b = make_problem(M, N, K, seed, with_bias=True, **kw)
    packed = pack_weights(capi, wc, ws, K)
    got = run_pair(capi, x, packed, b, M, N, K)
    rows = np.arange(M) if rows is None else rows
    acc, mag = oracle_gemm_rows(x, rows, wc, ws, K, b)
    check_close(got[rows], acc, mag, n_acc(K), what=f"pair M={M} N={N} K={K}", K=K)
    if library_takes_whole_tiles(M, N, K):
        single = run_gemm(capi, x, packed, b, M, N, K)
        assert np.array_equal(got, single), f"{int((got != single).sum())} outputs differ from mxfp4_gemm"


@pytest.mark.parametrize("M,N,K", [
    (256, 512, 512),        # two pairs, one tile each
    (200, 1000, 5152),      # ragged M (second CTA half empty), N and K; scales copied every k-step
    (256, 512, 14336),      # long K, scales copied every k-step
    (512, 19456, 1024),     # 152 pair tiles: two per pair, activation scales reused across them
])
def test_pair_tiles_every_output(capi, M, N, K):
    check(capi, M, N, K, seed=M + N + K, edge=True)


@pytest.mark.parametrize("M,N,K", [
    (768, 19456, 512),      # three tiles per pair; some pairs change activation row tile mid-run
    (4352, 1024, 5120),     # 68 pairs, one tile each
    (8193, 5800, 512),      # 65 row tiles: the last pair tile's second half lies past M
    (8192, 14336, 5120),    # a prefill shape of the benchmark
])
def test_pair_tiles_sampled_rows(capi, M, N, K):
    check(capi, M, N, K, seed=M + 3, rows=sample_rows(M, seed=M, n_random=32, boundary_stride=1))


@pytest.mark.parametrize("M", [200, 512])
def test_pair_prequantized_inputs_match_bf16_input(capi, M):
    """The two pre-quantized input forms (row-major, re-laid out into the workspace, and the TILED
    layout read in place) give the bits of the bf16 input quantized by the library."""
    N, K = 19456, 1024
    x, wc, ws, b = make_problem(M, N, K, seed=13, edge=True, with_bias=True)
    packed = pack_weights(capi, wc, ws, K)
    fused = run_pair(capi, x, packed, b, M, N, K)
    c_ref, s_ref = ref.quantize_mxfp4(ref.bf16_bits_to_f64(x))
    rm = run_pair(capi, x, packed, b, M, N, K, pre=(dev_u8(c_ref), dev_u8(s_ref), capi.LAYOUT_ROWMAJOR))
    tc, ts = tiled_from_oracle(c_ref, s_ref, K)
    tiled = run_pair(capi, x, packed, b, M, N, K, pre=(dev_u8(tc), dev_u8(ts), capi.LAYOUT_TILED))
    assert np.array_equal(fused, rm)
    assert np.array_equal(fused, tiled)


@pytest.mark.parametrize("M,N,K", [(64, 1024, 512), (300, 1024, 512), (2048, 5120, 14336)])
def test_pair_refuses_shapes_it_does_not_cover(capi, M, N, K):
    # M <= 64; three 128-row tiles; 160 pair tiles over 76 pairs (42% of the last wave idle)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    packed = torch.zeros(capi.mxfp4_packed_weight_bytes(1, N, K), dtype=torch.uint8, device="cuda")
    wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    work = gemm_workspace(capi, wsb)
    st = capi.lib.mxfp4_diag_gemm_pair(x.data_ptr(), K, None, None, 0, packed.data_ptr(), None, out.data_ptr(), N,
                                       M, N, K, work.data_ptr(), wsb, torch.cuda.current_stream().cuda_stream)
    assert st == capi.ERR_UNSUPPORTED_SHAPE
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
