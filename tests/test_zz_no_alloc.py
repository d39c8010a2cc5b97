"""The allocation-free GEMM entry point (mxfp4_gemm_noalloc).

Callers that cannot allocate device memory where they run the layer (inside
stream capture, in serving loops that must avoid cudaMalloc's implicit
synchronisation, or under a foreign allocator) use this entry point; its
scratch lives in a fixed device array inside the library.  The test calls it
through the C ABI twice in a row and checks each output bit for bit against
the workspace-taking mxfp4_gemm (the same kernels run on the same inputs, so
any difference would be a scratch-carving error, such as stale partial sums
of the previous call), and against the float64 oracle within the tolerance of
the other GEMM tests; it also checks that problems larger than the fixed
scratch are refused.  It sits in its own file so that pytest collects it
last.
"""

import numpy as np
import pytest
import torch

from mxfp4_quantized_gemm_gb300 import synth
from helpers import (check_close, dev_bf16, empty_u8, gemm_workspace, host_bits, oracle_gemm_rows, pack_weights,
                     sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


def with_workspace(capi, x, packed, bias, M, N, K):
    out = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    capi.mxfp4_gemm(x, K, None, None, 0, packed, bias, out, N, M, N, K, gemm_workspace(capi, wsb), wsb)
    torch.cuda.synchronize()
    return host_bits(out)


def without_workspace(capi, x, packed, bias, M, N, K):
    out = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    capi.mxfp4_gemm_noalloc(x, K, packed, bias, out, N, M, N, K)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    return host_bits(out)


@pytest.mark.parametrize("M,N,K", [(16, 14336, 5120), (64, 5120, 14336), (300, 1000, 5152)])
def test_noalloc_matches_workspace_entry_twice(capi, M, N, K):
    wc = synth.weight_codes(N, K, seed=M)
    ws = synth.weight_scales(N, K, -8, 2, seed=M)
    packed = pack_weights(capi, wc, ws, K)
    bias_bits = synth.bias(N, seed=M)
    bias = dev_bf16(bias_bits)
    for call in range(2):     # two calls in a row share the fixed scratch
        x_bits = synth.activations(M, K, seed=100 * M + call, outlier_frac=0.01)
        x = dev_bf16(x_bits)
        want = with_workspace(capi, x, packed, bias, M, N, K)
        got = without_workspace(capi, x, packed, bias, M, N, K)
        assert np.array_equal(got, want), f"call {call}: {int((got != want).sum())} outputs differ"
        rows = sample_rows(M, seed=call, n_random=8)
        acc, mag = oracle_gemm_rows(x_bits, rows, wc, ws, K, bias_bits)
        check_close(got[rows], acc, mag, -(-K // 64) + 4, what=f"noalloc call {call}")


def test_noalloc_refuses_problems_beyond_its_scratch(capi):
    M, N, K = 8192, 1024, 14336
    assert capi.mxfp4_gemm_workspace_bytes(M, N, K) > capi.mxfp4_gemm_noalloc_max_scratch_bytes()
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    packed = empty_u8(capi.mxfp4_packed_weight_bytes(1, N, K))
    st = capi.lib.mxfp4_gemm_noalloc(x.data_ptr(), K, packed.data_ptr(), None, out.data_ptr(), N, M, N, K,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == capi.ERR_WORKSPACE
