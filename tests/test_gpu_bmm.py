"""GPU parity of the A16WFP4 batched matmul (MLA absorbed K-up / V-up)."""

import numpy as np
import pytest
import torch

from oracle import mxfp4_ref as ref
from mxfp4_quantized_gemm_gb300 import synth
from helpers import check_close, dev_bf16, host_bits, pack_weights, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


def run_bmm(capi, x_bits, packed, B, M, N, K, batch_major):
    out = torch.zeros(B * M * N, dtype=torch.bfloat16, device="cuda")
    capi.a16wfp4_bmm(dev_bf16(x_bits), packed, out, B, M, N, K,
                     capi.OUT_MBN if batch_major else capi.OUT_BMN)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    o = host_bits(out)
    return o.reshape(M, B, N) if batch_major else o.reshape(B, M, N)


def oracle_rows(x_bits, rows, wc, ws, K):
    x = ref.bf16_bits_to_f64(x_bits[:, rows, :])
    return ref.a16wfp4_bmm_f64(x, wc, ws, K)


@pytest.mark.parametrize("kind,N,K,batch_major", [("K-up", 512, 192, False), ("V-up", 256, 512, True)])
@pytest.mark.parametrize("M", [16, 4096])
def test_mla_absorbed_bmm(capi, kind, N, K, batch_major, M):
    B = 64
    x = synth.bmm_activations(B, M, K, seed=M + N)
    wc = synth.weight_codes(N, K, seed=N, batch=B)
    ws = synth.weight_scales(N, K, -6, 0, seed=N, batch=B)
    packed = pack_weights(capi, wc, ws, K)
    got = run_bmm(capi, x, packed, B, M, N, K, batch_major)
    rows = np.arange(M) if M <= 64 else sample_rows(M, seed=4, n_random=16, boundary_stride=4)
    acc, mag = oracle_rows(x, rows, wc, ws, K)
    got_bmn = got.transpose(1, 0, 2) if batch_major else got
    check_close(got_bmn[:, rows, :], acc, mag, -(-K // 16) + 2, what=kind)


@pytest.mark.parametrize("B,M,N,K", [(1, 1, 128, 64), (3, 130, 200, 128), (2, 257, 64, 256), (5, 33, 512, 192),
                                     (3, 200, 256, 512), (2, 300, 200, 384), (4, 17, 512, 448), (1, 129, 40, 320),
                                     (2, 150, 256, 768), (1, 260, 300, 1024)])   # K > 512: 64-row weight tiles
@pytest.mark.parametrize("batch_major", [False, True])
def test_bmm_small_shapes(capi, B, M, N, K, batch_major):
    x = synth.bmm_activations(B, M, K, seed=B * M)
    wc = synth.weight_codes(N, K, seed=N, batch=B)
    ws = synth.weight_scales(N, K, -8, 2, seed=N, batch=B)
    packed = pack_weights(capi, wc, ws, K)
    got = run_bmm(capi, x, packed, B, M, N, K, batch_major)
    acc, mag = ref.a16wfp4_bmm_f64(ref.bf16_bits_to_f64(x), wc, ws, K)
    got_bmn = got.transpose(1, 0, 2) if batch_major else got
    check_close(got_bmn, acc, mag, -(-K // 16) + 2)


@pytest.mark.parametrize("B,M,N,K", [(185, 600, 128, 64), (89, 700, 300, 192)])
@pytest.mark.parametrize("batch_major", [False, True])
def test_bmm_more_pairs_than_sms(capi, B, M, N, K, batch_major):
    """More (batch, weight tile) pairs than a GB300 has SMs (178 and 185
    against 152), several M tiles each, ragged M and N: the grid runs in two
    waves of one-CTA-per-SM blocks.  Every output is compared."""
    x = synth.bmm_activations(B, M, K, seed=B + M)
    wc = synth.weight_codes(N, K, seed=N + 1, batch=B)
    ws = synth.weight_scales(N, K, -8, 2, seed=N + 1, batch=B)
    packed = pack_weights(capi, wc, ws, K)
    got = run_bmm(capi, x, packed, B, M, N, K, batch_major)
    acc, mag = ref.a16wfp4_bmm_f64(ref.bf16_bits_to_f64(x), wc, ws, K)
    got_bmn = got.transpose(1, 0, 2) if batch_major else got
    check_close(got_bmn, acc, mag, -(-K // 16) + 2)
