"""GPU parity of the fused RMSNorm -> MXFP4 producer against the oracle.

y is floating point: each value must lie within half a bf16 ulp of the exact
float64 RMSNorm plus 2**-18 relative (fp32 squares and sums over K <= 16384
terms, the hardware reciprocal square root and two fp32 products stay far
inside that), and at most 1% of the values may differ from the oracle's
correctly rounded bf16.  The residual update is exact (bit-identical).  The
quantization is an integer decision taken on the kernel's own bf16 y, so its
codes and scales must equal the oracle quantizer applied to that y, bit for
bit; against the oracle's own y they may differ only in blocks where the two
y differ.
"""

import numpy as np
import pytest
import torch

from oracle import mxfp4_ref as ref
from oracle import rmsnorm_ref as rn
from mxfp4_quantized_gemm_gb300 import synth
from oracle import tile_layout as tl
from helpers import dev_bf16, gemm_workspace, host_bits, pack_weights, sample_rows, ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


def run(capi, x_bits, gamma_bits, eps, layout, res_bits=None, want_y=True, ldx=None, offset=0):
    M, K = x_bits.shape
    ldx = ldx or K
    xbuf = np.zeros(offset + M * ldx, np.uint16)
    xbuf[offset:].reshape(M, ldx)[:, :K] = x_bits
    xd = dev_bf16(xbuf)
    x_view = xd[offset:]
    res = dev_bf16(res_bits) if res_bits is not None else None
    codes = torch.full((capi.mxfp4_act_code_bytes(M, K, layout),), 0xA5, dtype=torch.uint8, device="cuda")
    scales = torch.full((capi.mxfp4_act_scale_bytes(M, K, layout),), 0xA5, dtype=torch.uint8, device="cuda")
    y = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda") if want_y else None
    capi.mxfp4_rmsnorm_quant_act(x_view, ldx, res, K, dev_bf16(gamma_bits), eps, M, K, codes, scales, layout,
                                 y, K if want_y else 0)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    out = {"codes": codes.cpu().numpy(), "scales": scales.cpu().numpy()}
    if want_y:
        out["y"] = host_bits(y)
    if res is not None:
        out["h"] = host_bits(res)
    return out


def rows_of(got, M, K, layout):
    """Kernel codes [M, K/2] / scales [M, ceil(K/32)]; for TILED also checks
    that every padding byte holds the padding value (code 0, scale 0x7F)."""
    nb = -(-K // 32)
    if layout == 0:
        return got["codes"].reshape(M, K // 2), got["scales"].reshape(M, nb)
    c, sc = tl.unpack(np.concatenate([got["codes"], got["scales"]]), M, K)
    assert not c[M:].any() and not c[:, K // 2:].any(), "TILED code padding"
    assert np.all(sc[M:] == 0x7F) and np.all(sc[:, nb:] == 0x7F), "TILED scale padding"
    return c[:M, :K // 2], sc[:M, :nb]


def check(capi, M, K, layout, eps, with_res, seed, sample=None, **kw):
    x = synth.activations(M, K, seed=seed)
    gamma = synth.norm_gamma(K, seed=seed)
    res = synth.residual(M, K, seed=seed) if with_res else None
    got = run(capi, x, gamma, eps, layout, res, **kw)
    rows = np.arange(M) if sample is None else sample
    want = rn.rmsnorm_quant(x[rows], gamma, eps, res_bits=None if res is None else res[rows])
    if with_res:
        assert np.array_equal(got["h"][rows], want["h"]), "residual update"
    yk = got["y"][rows]
    y = ref.bf16_bits_to_f64(yk)
    err = np.abs(y - want["y_exact"])
    tol = 0.5 * ulp_bf16(want["y_exact"]) + 2.0 ** -18 * np.abs(want["y_exact"])
    assert np.all(err <= tol), f"y off by up to {np.max(err / np.maximum(tol, 1e-300)):.3f} x tolerance"
    n_diff = int((yk != want["y"]).sum())
    assert n_diff <= max(2, y.size // 100), f"{n_diff} of {y.size} y values differ from the rounded oracle"
    # the integer decision, taken on the kernel's own y
    codes, scales = rows_of(got, M, K, layout)
    c_k, s_k = ref.quantize_mxfp4(y)
    assert np.array_equal(codes[rows], c_k) and np.array_equal(scales[rows], s_k)
    # against the oracle's own y: differences only inside blocks where y differs
    R, nb = len(rows), -(-K // 32)
    ydiff = np.zeros((R, nb * 32), bool)
    ydiff[:, :K] = yk != want["y"]
    blk_diff = ydiff.reshape(R, nb, 32).any(axis=2)
    assert not ((s_k != want["scales"]) & ~blk_diff).any()
    cdiff = np.zeros((R, nb * 16), bool)
    cdiff[:, :K // 2] = c_k != want["codes"]
    assert not (cdiff.reshape(R, nb, 16).any(axis=2) & ~blk_diff).any()
    return n_diff


@pytest.mark.parametrize("M,K", [(1, 5120), (7, 5120), (64, 7168), (130, 5152), (300, 2048), (5, 100), (2, 34),
                                 (3, 8192), (33, 8448), (4, 14336)])
@pytest.mark.parametrize("layout", [0, 1])
def test_parity(capi, M, K, layout):
    check(capi, M, K, layout, 1e-6, False, seed=M + K)


@pytest.mark.parametrize("M,K", [(1, 5120), (130, 5152), (9, 14336), (6, 98)])
@pytest.mark.parametrize("layout", [0, 1])
def test_parity_with_residual(capi, M, K, layout):
    check(capi, M, K, layout, 1e-5, True, seed=3 * M + K)


@pytest.mark.parametrize("layout", [0, 1])
def test_residual_add_on_edge_rows(capi, layout):
    """x and residual both hold the structured edge rows (zeros of both signs,
    exact powers of two, rounding ties, bf16 subnormals): the fused add must
    round each exact sum once, with no flush of subnormals."""
    M, K = 40, 1024
    x = synth.with_edge_rows(synth.activations(M, K, seed=31), seed=31)
    res = synth.with_edge_rows(synth.residual(M, K, seed=32), seed=32)
    gamma = synth.norm_gamma(K, seed=31)
    got = run(capi, x, gamma, 1e-6, layout, res)
    assert np.array_equal(got["h"], rn.add_residual(x, res))


@pytest.mark.parametrize("eps", [0.0, 0.25, 4.0])
def test_eps_values(capi, eps):
    # eps comparable to the mean square (1 for these rows) moves every output
    check(capi, 20, 4096, 1, eps, False, seed=int(eps * 8))


def test_full_size_prefill_rows(capi):
    # the prefill activation shape: 8192 rows of the 5120-wide hidden state
    check(capi, 8192, 5120, 1, 1e-6, True, seed=99, sample=sample_rows(8192, seed=1))


@pytest.mark.parametrize("ldx,offset", [(5125, 0), (5120, 1), (5128, 3)])
def test_unaligned_rows(capi, ldx, offset):
    check(capi, 5, 5120, 0, 1e-6, False, seed=ldx + offset, ldx=ldx, offset=offset)


def test_codes_do_not_depend_on_the_y_output(capi):
    x = synth.activations(40, 5120, seed=4)
    gamma = synth.norm_gamma(5120, seed=4)
    a = run(capi, x, gamma, 1e-6, 1, want_y=True)
    b = run(capi, x, gamma, 1e-6, 1, want_y=False)
    assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["scales"], b["scales"])


def test_zero_and_nonfinite_rows(capi):
    K = 256
    x = synth.activations(4, K, seed=6)
    x[0] = 0                    # zero row, eps > 0: y = 0
    x[1, 17] = 0x7FC0           # NaN: the whole row is NaN -> scales 0xFF, codes 0
    x[2, 200] = 0xFF80          # -Inf: that element NaN, the rest 0
    gamma = synth.norm_gamma(K, seed=6)
    got = run(capi, x, gamma, 1e-6, 0)
    want = rn.rmsnorm_quant(x, gamma, 1e-6)
    # rows 0-2 are decided exactly; row 3 (ordinary values) is left to test_parity
    assert np.array_equal(got["codes"].reshape(4, K // 2)[:3], want["codes"][:3])
    assert np.array_equal(got["scales"].reshape(4, K // 32)[:3], want["scales"][:3])
    yk, yo = ref.bf16_bits_to_f64(got["y"]), ref.bf16_bits_to_f64(want["y"])
    assert np.array_equal(np.isnan(yk), np.isnan(yo))
    assert np.array_equal(yk[:3][~np.isnan(yk[:3])], yo[:3][~np.isnan(yo[:3])])


@pytest.mark.parametrize("M", [4, 300])
def test_fused_producer_feeds_the_gemm(capi, M):
    """Producer (TILED) -> GEMM equals the GEMM quantizing the producer's bf16 y itself."""
    N, K = 1024, 5120
    x = synth.activations(M, K, seed=M)
    gamma = synth.norm_gamma(K, seed=M)
    wc = synth.weight_codes(N, K, seed=M)
    ws = synth.weight_scales(N, K, -6, 0, seed=M)
    packed = pack_weights(capi, wc, ws, K)
    codes = torch.empty(capi.mxfp4_act_code_bytes(M, K, 1), dtype=torch.uint8, device="cuda")
    scales = torch.empty(capi.mxfp4_act_scale_bytes(M, K, 1), dtype=torch.uint8, device="cuda")
    y = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    capi.mxfp4_rmsnorm_quant_act(dev_bf16(x), K, None, 0, dev_bf16(gamma), 1e-6, M, K, codes, scales, 1, y, K)
    nbytes = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    out_pre = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    out_bf = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    capi.mxfp4_gemm(None, 0, codes, scales, 1, packed, None, out_pre, N, M, N, K, gemm_workspace(capi, nbytes), nbytes)
    capi.mxfp4_gemm(y, K, None, None, 0, packed, None, out_bf, N, M, N, K, gemm_workspace(capi, nbytes), nbytes)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    assert torch.equal(out_pre, out_bf)
