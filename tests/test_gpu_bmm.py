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
    check_close(got_bmn[:, rows, :], acc, mag, -(-K // 16) + 2, what=kind, K=K)


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
    check_close(got_bmn, acc, mag, -(-K // 16) + 2, what=f"bmm B={B} M={M} N={N} K={K}", K=K)


@pytest.mark.parametrize("B,M,N,K", [(185, 600, 128, 64), (89, 700, 300, 192), (80, 300, 200, 320)])
@pytest.mark.parametrize("batch_major", [False, True])
def test_bmm_more_pairs_than_sms(capi, B, M, N, K, batch_major):
    """More (batch, weight tile) pairs than a GB300 has SMs (185, 178 and 160
    against 152; the last with its weight tiles in TMEM), several M tiles
    each, ragged M and N: the grid runs in two waves of one-CTA-per-SM
    blocks.  Every output is compared."""
    x = synth.bmm_activations(B, M, K, seed=B + M)
    wc = synth.weight_codes(N, K, seed=N + 1, batch=B)
    ws = synth.weight_scales(N, K, -8, 2, seed=N + 1, batch=B)
    packed = pack_weights(capi, wc, ws, K)
    got = run_bmm(capi, x, packed, B, M, N, K, batch_major)
    acc, mag = ref.a16wfp4_bmm_f64(ref.bf16_bits_to_f64(x), wc, ws, K)
    got_bmn = got.transpose(1, 0, 2) if batch_major else got
    check_close(got_bmn, acc, mag, -(-K // 16) + 2, what=f"bmm B={B} M={M} N={N} K={K}", K=K)


@pytest.mark.parametrize("band", ["low", "high"])
@pytest.mark.parametrize("batch_major", [False, True])
def test_bmm_weight_scales_at_the_e8m0_extremes(capi, band, batch_major):
    """Live weight blocks at the ends of E8M0: bytes 0x00..0x06 against
    activations near 2^100, and 0xF0..0xFC against activations near 2^-118,
    every product and sum inside the fp32 range.  The kernel forms
    e2m1 * 2^(s-127) in bf16 before the MMA: exact for every code at these
    scales (the 0x00 values are bf16 subnormals); at 0xFD and 0xFE the larger
    codes exceed the bf16 range, outside what this kernel represents."""
    B, M, N, K = 3, 130, 256, 512
    x = synth.bmm_activations(B, M, K, seed=11)
    g = np.random.default_rng(5)
    wc = synth.weight_codes(N, K, seed=12, batch=B)
    nb = K // 32
    if band == "low":
        ws = g.integers(0x00, 0x07, size=(B, N, nb)).astype(np.uint8)
        ws[:, :, 0] = 0x00
        e = 100
    else:
        ws = g.integers(0xF0, 0xFD, size=(B, N, nb)).astype(np.uint8)
        ws[:, :, 0] = 0xFC
        e = -118
    x = ref.f64_to_bf16_bits(ref.bf16_bits_to_f64(x) * 2.0 ** e)
    packed = pack_weights(capi, wc, ws, K)
    got = run_bmm(capi, x, packed, B, M, N, K, batch_major)
    acc, mag = ref.a16wfp4_bmm_f64(ref.bf16_bits_to_f64(x), wc, ws, K)
    assert np.isfinite(acc).all()
    got_bmn = got.transpose(1, 0, 2) if batch_major else got
    check_close(got_bmn, acc, mag, -(-K // 16) + 2, what=f"bmm {band} scales", K=K)


@pytest.mark.parametrize("K", [192, 384])
@pytest.mark.parametrize("batch_major", [False, True])
def test_bmm_nan_weight_scale_poisons_its_output_column(capi, batch_major, K):
    """A live 0xFF (NaN) weight scale makes that batch's weight row's outputs
    NaN for every activation row, and nothing else (weight tile in shared
    memory at K = 192, in TMEM at K = 384)."""
    B, M, N = 2, 70, 200
    x = synth.bmm_activations(B, M, K, seed=13)
    wc = synth.weight_codes(N, K, seed=14, batch=B)
    ws = synth.weight_scales(N, K, -6, 0, seed=14, batch=B).copy()
    ws[1, 77, 3] = 0xFF
    packed = pack_weights(capi, wc, ws, K)
    got = run_bmm(capi, x, packed, B, M, N, K, batch_major)
    acc, mag = ref.a16wfp4_bmm_f64(ref.bf16_bits_to_f64(x), wc, ws, K)
    assert np.isnan(acc[1, :, 77]).all() and np.isfinite(acc[0]).all()
    got_bmn = got.transpose(1, 0, 2) if batch_major else got
    check_close(got_bmn, acc, mag, -(-K // 16) + 2, what="bmm NaN scale", K=K)


def test_bmm_from_new_host_threads(capi):
    """Calls from host threads that have made no CUDA call before (the x
    tensor map is encoded in the calling thread's device context): two
    threads, each its own stream, K-up and V-up shapes, the bits of the same
    calls made on the main thread."""
    import threading

    jobs = []
    for i, (B, M, N, K, bm) in enumerate([(4, 300, 512, 192, False), (4, 300, 256, 512, True)]):
        x = synth.bmm_activations(B, M, K, seed=70 + i)
        wc = synth.weight_codes(N, K, seed=71 + i, batch=B)
        ws = synth.weight_scales(N, K, -8, 2, seed=71 + i, batch=B)
        packed = pack_weights(capi, wc, ws, K)
        want = run_bmm(capi, x, packed, B, M, N, K, bm)
        jobs.append(dict(B=B, M=M, N=N, K=K, layout=capi.OUT_MBN if bm else capi.OUT_BMN, x=dev_bf16(x),
                         packed=packed, want=want, stream=torch.cuda.Stream(),
                         out=torch.zeros(B * M * N, dtype=torch.bfloat16, device="cuda")))
    torch.cuda.synchronize()
    errors = []

    def worker(j):
        try:
            for _ in range(5):
                capi.a16wfp4_bmm(j["x"], j["packed"], j["out"], j["B"], j["M"], j["N"], j["K"], j["layout"],
                                 j["stream"])
        except Exception as e:   # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert capi.mxfp4_get_device_error() == capi.OK
    for j in jobs:
        got = host_bits(j["out"])
        assert np.array_equal(got.reshape(j["want"].shape), j["want"]), (j["M"], j["N"], j["K"])
