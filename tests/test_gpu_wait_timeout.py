"""A device-side wait that runs out: the error path, made on purpose without a fault.

Every device-side wait of the library is bounded; one that gives up records
an error word, the kernel stops waiting, lets the copies it issued land and
exits, and mxfp4_get_device_error reports MXFP4_ERR_TIMEOUT.  This test makes
such a wait run out in the fused RMSNorm -> MXFP4 producer: with the bound of
its waits on the row copies lowered to one clock cycle
(mxfp4_diag_set_wait_cycles), the first wait of every block gives up while
its copy is still in flight.  Nothing is faulted and nothing is left in
flight: the kernel drains its copies under the full bound before it exits.
The host must then read MXFP4_ERR_TIMEOUT exactly once, and the same GPU must
serve the next calls normally (the producer bit for bit as before, a GEMM
against the oracle).
"""

import numpy as np
import pytest
import torch

from mxfp4_quantized_gemm_gb300 import synth
from helpers import check_close, dev_bf16, gemm_workspace, host_bits, oracle_gemm_rows, pack_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


def producer(capi, x, g, M, K):
    codes = torch.full((capi.mxfp4_act_code_bytes(M, K, 1),), 0xA5, dtype=torch.uint8, device="cuda")
    scales = torch.full((capi.mxfp4_act_scale_bytes(M, K, 1),), 0xA5, dtype=torch.uint8, device="cuda")
    capi.mxfp4_rmsnorm_quant_act(x, K, None, K, g, 1e-6, M, K, codes, scales, 1)
    return codes, scales


def test_bounded_wait_runs_out_and_the_gpu_stays_usable(capi):
    M, K = 512, 5120          # the bulk-copy producer kernel (K <= 8192, aligned rows)
    x = dev_bf16(synth.activations(M, K, seed=3))
    g = dev_bf16(synth.norm_gamma(K, seed=3))
    want_c, want_s = producer(capi, x, g, M, K)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK

    capi.mxfp4_diag_set_wait_cycles(1)
    try:
        producer(capi, x, g, M, K)
        torch.cuda.synchronize()
    finally:
        capi.mxfp4_diag_set_wait_cycles(0)
    assert capi.mxfp4_get_device_error() == capi.ERR_TIMEOUT
    assert capi.mxfp4_get_device_error() == capi.OK          # read and cleared

    got_c, got_s = producer(capi, x, g, M, K)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    assert torch.equal(got_c, want_c) and torch.equal(got_s, want_s)

    Mg, N, Kg = 16, 1024, 5120
    xb = synth.activations(Mg, Kg, seed=4)
    wc = synth.weight_codes(N, Kg, seed=4)
    ws = synth.weight_scales(N, Kg, -6, 0, seed=4)
    packed = pack_weights(capi, wc, ws, Kg)
    out = torch.empty(Mg, N, dtype=torch.bfloat16, device="cuda")
    wsb = capi.mxfp4_gemm_workspace_bytes(Mg, N, Kg)
    capi.mxfp4_gemm(dev_bf16(xb), Kg, None, None, 0, packed, None, out, N, Mg, N, Kg, gemm_workspace(capi, wsb), wsb)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    acc, mag = oracle_gemm_rows(xb, np.arange(Mg), wc, ws, Kg)
    check_close(host_bits(out), acc, mag, Kg // 64 + 4, what="GEMM after the timeout", K=Kg)


def test_wait_bound_argument_checked(capi):
    assert capi.lib.mxfp4_diag_set_wait_cycles(-1) == capi.ERR_INVALID_ARG
    assert capi.lib.mxfp4_diag_set_wait_cycles(0) == capi.OK
