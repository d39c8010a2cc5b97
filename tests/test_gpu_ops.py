"""GPU: the torch.library operators give bit-for-bit the results of the C-ABI
calls they wrap, agree with the oracle, and run under torch.compile and CUDA
graph capture."""

import numpy as np
import pytest
import torch

from oracle import mxfp4_ref as ref
from mxfp4_quantized_gemm_gb300 import ops, synth
from helpers import check_close, dev_bf16, dev_u8, gemm_workspace, host_bits, oracle_gemm_rows, pack_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


def problem(M, N, K, seed, with_bias=True):
    x = synth.activations(M, K, seed=seed)
    wc = synth.weight_codes(N, K, seed=seed)
    ws = synth.weight_scales(N, K, -6, 0, seed=seed)
    b = synth.bias(N, seed=seed) if with_bias else None
    return x, wc, ws, b


def capi_gemm(capi, x_bits, packed, b_bits, M, N, K):
    out = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    nbytes = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    capi.mxfp4_gemm(dev_bf16(x_bits), K, None, None, 0, packed, None if b_bits is None else dev_bf16(b_bits), out,
                    N, M, N, K, gemm_workspace(capi, nbytes), nbytes)
    torch.cuda.synchronize()
    return host_bits(out)


def test_pack_weights_op_matches_capi(capi):
    N, K, B = 300, 1000, 3
    wc = synth.weight_codes(N, K, seed=1, batch=B)
    ws = synth.weight_scales(N, K, -8, 2, seed=1, batch=B)
    got = torch.ops.mxfp4.pack_weights(dev_u8(wc), dev_u8(ws), K)
    want = pack_weights(capi, wc, ws, K)
    assert torch.equal(got, want[:got.numel()])


@pytest.mark.parametrize("layout", [0, 1])
def test_quant_act_op_matches_oracle(capi, layout):
    M, K = 130, 5120
    x = synth.with_edge_rows(synth.activations(M, K, seed=3), seed=3)
    codes, scales = torch.ops.mxfp4.quant_act(dev_bf16(x).view(2, 65, K), layout)
    torch.cuda.synchronize()
    c2 = torch.empty(capi.mxfp4_act_code_bytes(M, K, layout), dtype=torch.uint8, device="cuda")
    s2 = torch.empty(capi.mxfp4_act_scale_bytes(M, K, layout), dtype=torch.uint8, device="cuda")
    capi.mxfp4_quant_act(dev_bf16(x), M, K, K, c2, s2, layout)
    torch.cuda.synchronize()
    if layout == ops.LAYOUT_ROWMAJOR:
        oc, osc = ref.quantize_mxfp4(ref.bf16_bits_to_f64(x))
        assert np.array_equal(codes.cpu().numpy(), oc) and np.array_equal(scales.cpu().numpy(), osc)
    assert torch.equal(codes.flatten(), c2) and torch.equal(scales.flatten(), s2)


@pytest.mark.parametrize("lead,N,K", [((1,), 1024, 5120), ((2, 4), 1000, 5152), ((3, 100), 520, 2048)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_linear_op_matches_capi_and_oracle(capi, lead, N, K, with_bias):
    M = int(np.prod(lead))
    x, wc, ws, b = problem(M, N, K, seed=M + N, with_bias=with_bias)
    packed = pack_weights(capi, wc, ws, K)
    y = torch.ops.mxfp4.linear(dev_bf16(x).view(*lead, K), packed, None if b is None else dev_bf16(b), N)
    torch.cuda.synchronize()
    assert y.shape == (*lead, N)
    got = host_bits(y.reshape(M, N))
    assert np.array_equal(got, capi_gemm(capi, x, packed, b, M, N, K))
    rows = np.arange(M) if M <= 64 else np.array([0, 1, M // 2, M - 2, M - 1])
    acc, mag = oracle_gemm_rows(x, rows, wc, ws, K, b)
    check_close(got[rows], acc, mag, -(-K // 64) + 4, what="linear op")


@pytest.mark.parametrize("M", [16, 300])
@pytest.mark.parametrize("layout", [0, 1])
def test_prequant_op_matches_fused(capi, M, layout):
    N, K = 768, 2048
    x, wc, ws, b = problem(M, N, K, seed=M)
    packed = pack_weights(capi, wc, ws, K)
    xd, bd = dev_bf16(x), dev_bf16(b)
    codes, scales = torch.ops.mxfp4.quant_act(xd, layout)
    y = torch.ops.mxfp4.linear_prequant(codes, scales, layout, packed, bd, M, N, K)
    assert torch.equal(y, torch.ops.mxfp4.linear(xd, packed, bd, N))


def test_linear_mxfp4_out_op_feeds_linear_prequant(capi):
    M, N, K, N2 = 12, 1024, 2048, 512
    x, wc, ws, b = problem(M, N, K, seed=17)
    packed = pack_weights(capi, wc, ws, K)
    packed2 = pack_weights(capi, synth.weight_codes(N2, N, seed=18), synth.weight_scales(N2, N, -6, 0, seed=18), N)
    xd, bd = dev_bf16(x).view(3, 4, K), dev_bf16(b)
    codes, scales = torch.ops.mxfp4.linear_mxfp4_out(xd, packed, bd, N)
    y = torch.ops.mxfp4.linear(xd, packed, bd, N)
    c2, s2 = torch.ops.mxfp4.quant_act(y, 0)
    assert torch.equal(codes, c2) and torch.equal(scales, s2)
    z = torch.ops.mxfp4.linear_prequant(codes, scales, 0, packed2, None, M, N2, N)
    assert torch.equal(z, torch.ops.mxfp4.linear(y.view(M, N), packed2, None, N2))


def test_rmsnorm_quant_op_matches_capi(capi):
    M, K = 6, 5120
    x = dev_bf16(synth.activations(M, K, seed=21)).view(2, 3, K)
    gamma = dev_bf16(synth.norm_gamma(K, seed=21))
    res0 = dev_bf16(synth.residual(M, K, seed=21)).view(2, 3, K)
    res = res0.clone()
    codes, scales = torch.ops.mxfp4.rmsnorm_quant_act(x, gamma, 1e-6, 1, res)
    res2 = res0.clone().view(M, K)
    c2 = torch.empty_like(codes)
    s2 = torch.empty_like(scales)
    capi.mxfp4_rmsnorm_quant_act(x.view(M, K), K, res2, K, gamma, 1e-6, M, K, c2, s2, 1)
    torch.cuda.synchronize()
    assert torch.equal(codes, c2) and torch.equal(scales, s2) and torch.equal(res.view(M, K), res2)
    assert not torch.equal(res, res0)


@pytest.mark.parametrize("batch_major", [False, True])
def test_bmm_op_matches_capi(capi, batch_major):
    B, M, N, K = 16, 40, 512, 192
    x = synth.bmm_activations(B, M, K, seed=5)
    wc = synth.weight_codes(N, K, seed=5, batch=B)
    ws = synth.weight_scales(N, K, -6, 0, seed=5, batch=B)
    packed = pack_weights(capi, wc, ws, K)
    y = torch.ops.mxfp4.a16wfp4_bmm(dev_bf16(x), packed, N, batch_major)
    want = torch.zeros_like(y)
    capi.a16wfp4_bmm(dev_bf16(x), packed, want, B, M, N, K, capi.OUT_MBN if batch_major else capi.OUT_BMN)
    torch.cuda.synchronize()
    assert torch.equal(y, want)


def test_opcheck_schema_and_fake(capi):
    """Every operator: schema checks, and the fake kernel's outputs match the
    real kernel's in shape, dtype and strides."""
    M, N, K = 5, 300, 1024
    x, wc, ws, b = problem(M, N, K, seed=9)
    packed = pack_weights(capi, wc, ws, K)
    xd, bd = dev_bf16(x), dev_bf16(b)
    utils = ("test_schema", "test_faketensor")
    torch.library.opcheck(torch.ops.mxfp4.linear.default, (xd, packed, bd, N), test_utils=utils)
    torch.library.opcheck(torch.ops.mxfp4.linear_mxfp4_out.default, (xd, packed, bd, N), test_utils=utils)
    for layout in (0, 1):
        torch.library.opcheck(torch.ops.mxfp4.quant_act.default, (xd, layout), test_utils=utils)
        codes, scales = torch.ops.mxfp4.quant_act(xd, layout)
        torch.library.opcheck(torch.ops.mxfp4.linear_prequant.default, (codes, scales, layout, packed, bd, M, N, K),
                              test_utils=utils)
        torch.library.opcheck(torch.ops.mxfp4.rmsnorm_quant_act.default,
                              (xd, dev_bf16(synth.norm_gamma(K, seed=9)), 1e-6, layout, None), test_utils=utils)
    # the residual form: the schema check also confirms that only the declared
    # argument is written
    torch.library.opcheck(torch.ops.mxfp4.rmsnorm_quant_act.default,
                          (xd, dev_bf16(synth.norm_gamma(K, seed=9)), 1e-6, 0, dev_bf16(synth.residual(M, K, seed=9))),
                          test_utils=utils)
    torch.library.opcheck(torch.ops.mxfp4.pack_weights.default, (dev_u8(wc), dev_u8(ws), K), test_utils=utils)
    # split + cat: 10 groups of 16 + 16 columns, z of 24 values per group
    Ns = 10 * 32
    ps = pack_weights(capi, synth.weight_codes(Ns, K, seed=10), synth.weight_scales(Ns, K, -6, 0, seed=10), K)
    zd = dev_bf16(synth.activations(M, 10 * 24, seed=10)).reshape(M, 10, 24)
    torch.library.opcheck(torch.ops.mxfp4.linear_split_cat.default, (xd, ps, None, zd, 16, 16), test_utils=utils)
    B = 2
    xb = dev_bf16(synth.bmm_activations(B, 7, 192, seed=9))
    pb = pack_weights(capi, synth.weight_codes(256, 192, seed=9, batch=B),
                      synth.weight_scales(256, 192, -6, 0, seed=9, batch=B), 192)
    for bm in (False, True):
        torch.library.opcheck(torch.ops.mxfp4.a16wfp4_bmm.default, (xb, pb, 256, bm), test_utils=utils)


def test_compiled_layer_matches_eager(capi):
    M, N, K = 24, 1024, 2048
    x, wc, ws, b = problem(M, N, K, seed=11)
    packed = pack_weights(capi, wc, ws, K)
    xd, bd = dev_bf16(x).view(2, 12, K), dev_bf16(b)

    def layer(x):
        return torch.ops.mxfp4.linear(x, packed, bd, N).float().square().sum(-1)

    eager = layer(xd)
    compiled = torch.compile(layer, backend="aot_eager", fullgraph=True)(xd)
    assert torch.equal(eager, compiled)


def test_graph_captured_ops_replay(capi):
    M, N, K = 8, 1536, 4096
    x, wc, ws, b = problem(M, N, K, seed=13)
    packed = pack_weights(capi, wc, ws, K)
    xd, bd = dev_bf16(x), dev_bf16(b)
    want = torch.ops.mxfp4.linear(xd, packed, bd, N)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        torch.ops.mxfp4.linear(xd, packed, bd, N)   # warm the allocator on the side stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        y = torch.ops.mxfp4.linear(xd, packed, bd, N)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, want)
    assert capi.mxfp4_get_device_error() == capi.OK


def test_split_cat_op_matches_capi(capi):
    M, H, s1, s2, s3, K = 6, 12, 16, 48, 8, 512
    N = H * (s1 + s2)
    x, wc, ws, b = problem(M, N, K, seed=13)
    packed = pack_weights(capi, wc, ws, K)
    z = dev_bf16(synth.activations(M, H * s3, seed=14)).reshape(M, H, s3)
    cat, split = torch.ops.mxfp4.linear_split_cat(dev_bf16(x), packed, dev_bf16(b), z, s1, s2)
    y = torch.ops.mxfp4.linear(dev_bf16(x), packed, dev_bf16(b), N)
    torch.cuda.synchronize()
    yg = y.reshape(M, H, s1 + s2)
    assert torch.equal(cat, torch.cat([yg[:, :, :s1], z], dim=2))
    assert torch.equal(split, yg[:, :, s1:])
