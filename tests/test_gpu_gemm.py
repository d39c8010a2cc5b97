"""GPU parity of the W4A4 MXFP4 GEMM against the oracle.

Covers the five workloads: the synthetic (16, 1024, 5120) GEMM; the decode
sweep with outlier channels; prefill with bias (sampled rows); the edge and
tail cases (N = 128 at small M, M in {1, 8193}, N = 1000 with K = 5152, edge
rows); plus the three activation input forms, padding invariance, run-to-run
determinism and a sweep of tiny shapes.
"""

import numpy as np
import pytest
import torch

from oracle import mxfp4_ref as ref
from mxfp4_quantized_gemm_gb300 import synth
from helpers import (check_close, dev_bf16, dev_u8, empty_u8, gemm_workspace, host_bits, oracle_gemm_rows,
                     pack_weights,
                     sample_rows, tiled_from_oracle)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from mxfp4_quantized_gemm_gb300 import capi as c
    return c


def make_problem(M, N, K, seed, w_lo=-6, w_hi=0, outliers=0.0, edge=False, with_bias=False):
    x = synth.activations(M, K, seed=seed, outlier_frac=outliers)
    if edge:
        x = synth.with_edge_rows(x, seed=seed)
    wc = synth.weight_codes(N, K, seed=seed)
    ws = synth.weight_scales(N, K, w_lo, w_hi, seed=seed)
    b = synth.bias(N, seed=seed) if with_bias else None
    return x, wc, ws, b


def run_gemm(capi, x_bits, packed, bias_bits, M, N, K, ldo=None, mode="bf16", pre=None):
    ldo = ldo or N
    out = torch.zeros(M, ldo, dtype=torch.bfloat16, device="cuda")
    ws_bytes = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    ws = gemm_workspace(capi, ws_bytes)
    bias = dev_bf16(bias_bits) if bias_bits is not None else None
    if mode == "bf16":
        capi.mxfp4_gemm(dev_bf16(x_bits), K, None, None, 0, packed, bias, out, ldo, M, N, K, ws, ws_bytes)
    else:
        codes, scales, layout = pre
        capi.mxfp4_gemm(None, 0, codes, scales, layout, packed, bias, out, ldo, M, N, K, ws, ws_bytes)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    return host_bits(out)[:, :N]


def n_acc(K):
    return -(-K // 64) + 4


def full_check(capi, M, N, K, seed, **kw):
    x, wc, ws, b = make_problem(M, N, K, seed, **kw)
    packed = pack_weights(capi, wc, ws, K)
    got = run_gemm(capi, x, packed, b, M, N, K)
    acc, mag = oracle_gemm_rows(x, np.arange(M), wc, ws, K, b)
    return check_close(got, acc, mag, n_acc(K), what=f"M={M} N={N} K={K}")


def test_synthetic_16x1024x5120(capi):
    full_check(capi, 16, 1024, 5120, seed=0)


@pytest.mark.parametrize("M", [2, 3, 17, 64])
def test_small_n_rows_all_correct(capi, M):
    # the pages' gfx950 heuristic returned wrong rows 1..M-1 for N <= 128, 2 <= M <= 64
    full_check(capi, M, 128, 5120, seed=M, edge=True)


@pytest.mark.parametrize("M,N,K", [(1, 1024, 5120), (16, 1000, 5152)])
def test_tail_shapes_small_m(capi, M, N, K):
    full_check(capi, M, N, K, seed=M + N, edge=True)


@pytest.mark.parametrize("NK", [(14336, 5120), (5120, 14336), (34816, 5120)])
@pytest.mark.parametrize("M", [1, 4, 16, 32, 64])
def test_decode_sweep(capi, M, NK):
    N, K = NK
    full_check(capi, M, N, K, seed=M * 7 + N, w_lo=-8, w_hi=2, outliers=0.01)


@pytest.mark.parametrize("M,N,K", [(8193, 1024, 5120), (8193, 1000, 5152)])
def test_tail_shapes_large_m(capi, M, N, K):
    x, wc, ws, b = make_problem(M, N, K, seed=M + N, edge=True)
    packed = pack_weights(capi, wc, ws, K)
    got = run_gemm(capi, x, packed, b, M, N, K)
    rows = sample_rows(M, seed=1)
    acc, mag = oracle_gemm_rows(x, rows, wc, ws, K, b)
    check_close(got[rows], acc, mag, n_acc(K), what=f"M={M}")


@pytest.mark.parametrize("NK", [(14336, 5120), (5120, 14336), (34816, 5120)])
@pytest.mark.parametrize("M", [2048, 8192])
def test_prefill_with_bias(capi, M, NK):
    N, K = NK
    x, wc, ws, b = make_problem(M, N, K, seed=M + N, with_bias=True)
    packed = pack_weights(capi, wc, ws, K)
    got = run_gemm(capi, x, packed, b, M, N, K)
    rows = sample_rows(M, seed=2, n_random=24, boundary_stride=8)
    acc, mag = oracle_gemm_rows(x, rows, wc, ws, K, b)
    check_close(got[rows], acc, mag, n_acc(K), what=f"prefill M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 2, 5, 8, 16, 300])
def test_prequantized_inputs_match_fused(capi, M):
    """bf16 input (quantized inside the GEMM kernel for M <= 8, by the
    quantizer kernel above) and the two pre-quantized forms give the same
    bits."""
    N, K = 640, 5152
    x, wc, ws, b = make_problem(M, N, K, seed=11, edge=True, with_bias=True)
    packed = pack_weights(capi, wc, ws, K)
    fused = run_gemm(capi, x, packed, b, M, N, K)
    c_ref, s_ref = ref.quantize_mxfp4(ref.bf16_bits_to_f64(x))
    rm = run_gemm(capi, x, packed, b, M, N, K, mode="pre",
                  pre=(dev_u8(c_ref), dev_u8(s_ref), capi.LAYOUT_ROWMAJOR))
    tc, ts = tiled_from_oracle(c_ref, s_ref, K)
    tiled = run_gemm(capi, x, packed, b, M, N, K, mode="pre", pre=(dev_u8(tc), dev_u8(ts), capi.LAYOUT_TILED))
    assert np.array_equal(fused, rm)
    assert np.array_equal(fused, tiled)


@pytest.mark.parametrize("M", [5, 200])
def test_padding_scales_never_change_results(capi, M):
    from oracle import tile_layout as tl
    N, K = 200, 288     # pads rows 200 -> 256 and K 288 -> 512
    x, wc, ws, b = make_problem(M, N, K, seed=5)
    packed = pack_weights(capi, wc, ws, K)
    base = run_gemm(capi, x, packed, b, M, N, K)
    offs = tl.weight_scale_offsets(N, K)
    pad = np.ones(offs.shape, bool)
    pad[:N, : -(-K // 32)] = False
    g = np.random.default_rng(0)
    for val in (0x00, 0x80, 0xFE, None):
        host = packed.cpu().numpy().copy()
        host[offs[pad]] = g.integers(0, 255, size=int(pad.sum())) if val is None else val
        got = run_gemm(capi, x, dev_u8(host), b, M, N, K)
        assert np.array_equal(got, base), val


@pytest.mark.parametrize("M,N,K", [(37, 14336, 5120), (64, 5120, 14336), (1, 34816, 5120), (2048, 1024, 5120)])
def test_run_to_run_bit_identical(capi, M, N, K):
    x, wc, ws, b = make_problem(M, N, K, seed=3, with_bias=True)
    packed = pack_weights(capi, wc, ws, K)
    first = run_gemm(capi, x, packed, b, M, N, K)
    for _ in range(3):
        assert np.array_equal(run_gemm(capi, x, packed, b, M, N, K), first)


def test_leading_dimension_of_output(capi):
    M, N, K = 20, 136, 256
    x, wc, ws, b = make_problem(M, N, K, seed=9, with_bias=True)
    packed = pack_weights(capi, wc, ws, K)
    got = run_gemm(capi, x, packed, b, M, N, K, ldo=N + 40)
    acc, mag = oracle_gemm_rows(x, np.arange(M), wc, ws, K, b)
    check_close(got, acc, mag, n_acc(K), K=K)


TINY = [(m, n, k) for m in (1, 2, 7, 16, 33, 64, 65, 129)
        for n in (1, 8, 127, 128, 129, 300) for k in (32, 64, 96, 256, 288, 512)]


def test_tiny_shape_sweep(capi):
    bad = []
    for i, (M, N, K) in enumerate(TINY):
        x, wc, ws, b = make_problem(M, N, K, seed=100 + i, w_lo=-8, w_hi=2, edge=True, with_bias=(i % 2 == 0))
        packed = pack_weights(capi, wc, ws, K)
        got = run_gemm(capi, x, packed, b, M, N, K)
        acc, mag = oracle_gemm_rows(x, np.arange(M), wc, ws, K, b)
        try:
            check_close(got, acc, mag, n_acc(K), what=f"{(M, N, K)}", K=K)
        except AssertionError as e:
            bad.append(str(e)[:200])
    assert not bad, f"{len(bad)} of {len(TINY)} shapes failed: {bad[:4]}"


@pytest.mark.parametrize("M,N,K", [(64, 256, 32768), (5, 300, 65536), (2, 256, 98560), (33, 256, 98560)])
def test_tiles_shared_by_many_ctas(capi, M, N, K):
    """One or two output tiles over a long K: for M <= 64 every tile's
    k-steps are split over a cluster of 8 CTAs whose parts are summed in
    shared memory (M = 2 and 5 quantized by the GEMM kernel itself, M = 33
    and 64 by the quantizer first); for larger M, stream-K parts."""
    full_check(capi, M, N, K, seed=21, with_bias=True)


@pytest.mark.parametrize("M,N,K", [(1, 40000, 512), (8, 39168, 1024), (12, 40960, 768), (64, 39000, 512)])
def test_more_tiles_than_sms(capi, M, N, K):
    """More 256-row weight tiles than SMs (152 on GB300): each decode CTA
    takes whole tiles in turn, draining the accumulator between them, with
    the activations quantized by four of its warps (M <= 8) or by the
    quantizer kernel first."""
    full_check(capi, M, N, K, seed=31, with_bias=True)


def test_one_workspace_for_every_shape_and_graph_replays(capi):
    """Calls of different shapes and input forms share one workspace (whatever
    one call leaves in it, the next may not depend on), eagerly and replayed
    from a CUDA graph, and give the bits of the same calls on fresh
    workspaces."""
    shapes = [(1, 14336, 5120), (64, 5120, 14336), (200, 1024, 5120), (16, 1000, 5152), (33, 128, 256),
              (2, 256, 98560)]
    probs, want = [], []
    for i, (M, N, K) in enumerate(shapes):
        x, wc, ws, b = make_problem(M, N, K, seed=40 + i, with_bias=(i % 2 == 1))
        packed = pack_weights(capi, wc, ws, K)
        probs.append((M, N, K, dev_bf16(x), packed, dev_bf16(b) if b is not None else None))
        want.append(run_gemm(capi, x, packed, b, M, N, K))
    wsb = max(capi.mxfp4_gemm_workspace_bytes(M, N, K) for M, N, K in shapes)
    work = gemm_workspace(capi, wsb)
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for M, N, K, *_ in probs]

    def calls(stream=None):
        for (M, N, K, x, packed, bias), out in zip(probs, outs):
            capi.mxfp4_gemm(x, K, None, None, 0, packed, bias, out, N, M, N, K, work, wsb, stream)

    for _ in range(3):
        for o in outs:
            o.fill_(float("nan"))
        calls()
        torch.cuda.synchronize()
        assert capi.mxfp4_get_device_error() == capi.OK
        for o, w in zip(outs, want):
            assert np.array_equal(host_bits(o), w)

    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        calls(s.cuda_stream)          # warm-up on the capture stream
        s.synchronize()
        with torch.cuda.graph(graph, stream=s):
            calls(s.cuda_stream)
    for _ in range(5):
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert capi.mxfp4_get_device_error() == capi.OK
        for o, w in zip(outs, want):
            assert np.array_equal(host_bits(o), w)


@pytest.mark.parametrize("M,N,K,pad", [(5, 300, 100, 0), (3, 520, 5120, 1), (16, 256, 1000, 3), (40, 700, 2056, 1)])
def test_unaligned_activation_rows(capi, M, N, K, pad):
    """bf16 rows that are not 16-byte aligned (lda = K + pad) or K % 8 != 0:
    the quantizing CTAs fall back to element loads, and the results must
    still match the oracle."""
    x, wc, ws, b = make_problem(M, N, K, seed=77, with_bias=True)
    packed = pack_weights(capi, wc, ws, K)
    lda = K + pad
    xpad = np.zeros((M, lda), dtype=np.uint16)
    xpad[:, :K] = x
    xd = dev_bf16(xpad)
    out = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    work = gemm_workspace(capi, wsb)
    capi.mxfp4_gemm(xd, lda, None, None, 0, packed, dev_bf16(b), out, N, M, N, K, work, wsb)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    acc, mag = oracle_gemm_rows(x, np.arange(M), wc, ws, K, b)
    check_close(host_bits(out), acc, mag, n_acc(K), what=f"M={M} N={N} K={K} lda={lda}")


def test_concurrent_host_threads(capi):
    """The entry points are re-entrant: four host threads (ctypes releases
    the GIL during the call) each run a different shape on their own stream
    and workspace, twenty calls each, and get the bits of the same calls made
    one after another."""
    import threading

    shapes = [(1, 14336, 5120), (16, 5120, 14336), (300, 1024, 5120), (64, 256, 32768)]
    jobs = []
    for i, (M, N, K) in enumerate(shapes):
        x, wc, ws, b = make_problem(M, N, K, seed=60 + i, with_bias=True)
        packed = pack_weights(capi, wc, ws, K)
        want = run_gemm(capi, x, packed, b, M, N, K)
        wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
        jobs.append(dict(M=M, N=N, K=K, x=dev_bf16(x), packed=packed, bias=dev_bf16(b), want=want,
                         ws=gemm_workspace(capi, wsb), wsb=wsb, stream=torch.cuda.Stream(),
                         out=torch.empty(M, N, dtype=torch.bfloat16, device="cuda")))
    torch.cuda.synchronize()
    errors = []

    def worker(j):
        try:
            for _ in range(20):
                capi.mxfp4_gemm(j["x"], j["K"], None, None, 0, j["packed"], j["bias"], j["out"], j["N"], j["M"],
                                j["N"], j["K"], j["ws"], j["wsb"], j["stream"])
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
        assert np.array_equal(host_bits(j["out"]), j["want"]), (j["M"], j["N"], j["K"])


def scaled_bf16(bits: np.ndarray, e: int) -> np.ndarray:
    """bf16 values times 2^e, rounded to bf16 (values pushed below the normal
    range lose bits; kernel and oracle see the same rounded inputs)."""
    return ref.f64_to_bf16_bits(ref.bf16_bits_to_f64(bits) * 2.0 ** e)


@pytest.mark.parametrize("M", [4, 16, 200])
@pytest.mark.parametrize("band", ["low", "high"])
def test_weight_scales_at_the_e8m0_extremes(capi, M, band):
    """Live weight blocks whose E8M0 scales sit at the ends of the format:
    bytes 0x00..0x06 (2^-127..2^-121) against activations near 2^100, and
    0xF0..0xFE (2^113..2^127) against activations near 2^-118, so that every
    product and sum stays inside the fp32 normal range while the scale
    exponents reach both limits.  Covers the in-kernel quantizer (M = 4),
    the decode kernel after the quantizer (M = 16) and the prefill kernel."""
    N, K = 520, 1024
    x, wc, _, b = make_problem(M, N, K, seed=M + (0 if band == "low" else 1))
    g = np.random.default_rng(M)
    nb = -(-K // 32)
    if band == "low":
        ws = g.integers(0x00, 0x07, size=(N, nb)).astype(np.uint8)
        ws[:, 0] = 0x00
        x = scaled_bf16(x, 100)
    else:
        ws = g.integers(0xF0, 0xFF, size=(N, nb)).astype(np.uint8)
        ws[:, 0] = 0xFE
        x = scaled_bf16(x, -118)
    packed = pack_weights(capi, wc, ws, K)
    got = run_gemm(capi, x, packed, None, M, N, K)
    acc, mag = oracle_gemm_rows(x, np.arange(M), wc, ws, K, None)
    assert np.isfinite(acc).all()
    check_close(got, acc, mag, n_acc(K), what=f"{band} scales M={M}", K=K)


@pytest.mark.parametrize("M", [4, 16, 200])
def test_nan_weight_scale_poisons_its_output_column(capi, M):
    """A live weight block with scale 0xFF (E8M0 NaN) makes that weight row's
    output NaN for every activation row, and nothing else."""
    N, K = 300, 512
    x, wc, ws, b = make_problem(M, N, K, seed=7 + M, with_bias=True)
    ws = ws.copy()
    ws[37, 5] = 0xFF
    ws[299, 15] = 0xFF
    packed = pack_weights(capi, wc, ws, K)
    got = run_gemm(capi, x, packed, b, M, N, K)
    acc, mag = oracle_gemm_rows(x, np.arange(M), wc, ws, K, b)
    assert np.isnan(acc[:, [37, 299]]).all() and np.isfinite(np.delete(acc, [37, 299], axis=1)).all()
    check_close(got, acc, mag, n_acc(K), what=f"NaN scale M={M}", K=K)


@pytest.mark.parametrize("M", [1, 16, 300])
def test_weights_refreshed_by_a_device_copy(capi, M):
    """The weight-update contract: a packed buffer rewritten by an ordinary
    device copy (not mxfp4_pack_weights), then mxfp4_weights_updated, then the
    GEMM: every call sees the weights of the copy just made, alternating
    between two weight sets."""
    N, K = 1024, 5120
    x, _, _, b = make_problem(M, N, K, seed=91 + M, with_bias=True)
    sets = []
    for k in range(2):
        wc = synth.weight_codes(N, K, seed=500 + k)
        ws = synth.weight_scales(N, K, -6, 0, seed=500 + k)
        sets.append((wc, ws, pack_weights(capi, wc, ws, K)))
    live = torch.empty_like(sets[0][2])
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    work = gemm_workspace(capi, wsb)
    xd, bd = dev_bf16(x), dev_bf16(b)
    want = []
    for wc, ws, _ in sets:
        acc, mag = oracle_gemm_rows(x, np.arange(M), wc, ws, K, b)
        want.append((acc, mag))
    torch.cuda.synchronize()
    for it in range(6):
        k = it % 2
        live.copy_(sets[k][2])            # an ordinary kernel writes the weights
        capi.mxfp4_weights_updated()
        capi.mxfp4_gemm(xd, K, None, None, 0, live, bd, out, N, M, N, K, work, wsb)
        torch.cuda.synchronize()
        assert capi.mxfp4_get_device_error() == capi.OK
        check_close(host_bits(out), *want[k], n_acc(K), what=f"refresh {it}")
