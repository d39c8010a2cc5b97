"""PyTorch custom operators over the library's C ABI (namespace ``mxfp4``).

Each operator has a fake (meta) implementation that only computes output
shapes, so FakeTensor tracing and ``torch.compile`` pass through the calls;
the real implementations marshal arguments to ``capi`` (every computation
runs in the library's CUDA kernels; output and scratch memory come from
torch's caching allocator, on the current stream).  The operations are those
the pages call from the layer code -- per_1x32_f4_quant, gemm_a4w4 with the
bias added, the pre-quantized tuple input, the one-time weight repack, and
the MLA absorbed BMM (sglang PR #39598 blog analysis, section 2,
apply_weights / process_weights_after_loading; PR #34317, Modifications) --
including the pages' flattening of 3-D activations to 2-D for the GEMM.

    torch.ops.mxfp4.pack_weights(codes, scales, K) -> packed
    torch.ops.mxfp4.quant_act(x, layout) -> (codes, scales)
    torch.ops.mxfp4.rmsnorm_quant_act(x, gamma, eps, layout, residual) -> (codes, scales)   # residual updated
    torch.ops.mxfp4.linear(x, w_packed, bias, N) -> out          # x [..., K] bf16
    torch.ops.mxfp4.linear_prequant(codes, scales, layout, w_packed, bias, M, N, K) -> out
    torch.ops.mxfp4.linear_mxfp4_out(x, w_packed, bias, N) -> (codes, scales)   # next layer's input
    torch.ops.mxfp4.linear_split_cat(x, w_packed, bias, z, s1, s2) -> (cat, split)   # per-group split + cat
    torch.ops.mxfp4.a16wfp4_bmm(x, w_packed, N, batch_major) -> out
"""

from __future__ import annotations

from typing import Optional

import torch
from torch import Tensor
from torch.library import custom_op

LAYOUT_ROWMAJOR, LAYOUT_TILED = 0, 1


def _capi():
    from . import capi
    return capi


def _stream(t: Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def _packed_weight_bytes(batch: int, N: int, K: int) -> int:
    # the packed layout of include/mxfp4.h: one 34816-byte block per
    # (256-row pair, 256-wide k-tile)
    return batch * _cdiv(N, 256) * _cdiv(K, 256) * 34816


def _check_args(where: str, *ts: Optional[Tensor], dtypes=()) -> None:
    """The tensors handed to the library must live on one CUDA device (the
    kernels dereference their pointers; a host pointer there would fault)
    and have the expected dtypes (None entries are skipped)."""
    dev = None
    for i, t in enumerate(ts):
        if t is None:
            continue
        if i < len(dtypes) and dtypes[i] is not None:
            torch._check(t.dtype == dtypes[i], lambda: f"{where}: argument {i} must be {dtypes[i]}, got {t.dtype}")
        if t.device.type == "meta":
            continue
        torch._check(t.device.type == "cuda", lambda: f"{where}: argument {i} is on {t.device}, not a CUDA device")
        dev = dev or t.device
        torch._check(t.device == dev, lambda: f"{where}: arguments are on different devices")


def _check_weights(where: str, w_packed: Tensor, batch: int, N: int, K: int) -> None:
    torch._check(K > 0 and K % 2 == 0, lambda: f"{where}: K = {K} must be positive and even")
    torch._check(N > 0, lambda: f"{where}: N = {N} must be positive")
    need = _packed_weight_bytes(batch, N, K)
    torch._check(w_packed.numel() >= need,
                 lambda: f"{where}: packed weights hold {w_packed.numel()} bytes, {need} needed")


def _check_bias(where: str, bias: Optional[Tensor], N: int) -> None:
    if bias is not None:
        torch._check(bias.numel() == N, lambda: f"{where}: bias has {bias.numel()} elements, N = {N}")


def _act_bytes(M: int, K: int, layout: int) -> tuple[int, int]:
    if layout == LAYOUT_ROWMAJOR:
        return M * (K // 2), M * _cdiv(K, 32)
    rp, kp = _cdiv(M, 128) * 128, _cdiv(K, 256) * 256
    return rp * kp // 2, rp * kp // 32


# ------------------------------------------------------------ weight repack
def _check_pack(where: str, codes: Tensor, scales: Tensor, K: int) -> None:
    _check_args(where, codes, scales, dtypes=(torch.uint8, torch.uint8))
    torch._check(codes.dim() in (2, 3) and scales.dim() == codes.dim(),
                 lambda: f"{where}: codes and scales must both be [N, *] or [B, N, *]")
    torch._check(K > 0 and K % 2 == 0, lambda: f"{where}: K = {K} must be positive and even")
    torch._check(codes.shape[-1] == K // 2 and scales.shape[-1] == _cdiv(K, 32),
                 lambda: f"{where}: codes [.., {codes.shape[-1]}] / scales [.., {scales.shape[-1]}] do not hold K = {K}")
    torch._check(codes.shape[:-1] == scales.shape[:-1], lambda: f"{where}: codes and scales differ in leading dims")


@custom_op("mxfp4::pack_weights", mutates_args=())
def pack_weights(codes: Tensor, scales: Tensor, K: int) -> Tensor:
    """codes [N, K/2] or [B, N, K/2] uint8, scales [.., N, ceil(K/32)] uint8
    -> the packed weight buffer (uint8)."""
    _check_pack("mxfp4::pack_weights", codes, scales, K)
    c = _capi()
    B = codes.shape[0] if codes.dim() == 3 else 1
    N = codes.shape[-2]
    packed = torch.empty(_packed_weight_bytes(B, N, K), dtype=torch.uint8, device=codes.device)
    c.mxfp4_pack_weights(codes.contiguous(), scales.contiguous(), B, N, K, packed, _stream(codes))
    return packed


@pack_weights.register_fake
def _(codes, scales, K):
    _check_pack("mxfp4::pack_weights", codes, scales, K)
    B = codes.shape[0] if codes.dim() == 3 else 1
    return codes.new_empty(_packed_weight_bytes(B, codes.shape[-2], K), dtype=torch.uint8)


# ---------------------------------------------------- activation quantizer
@custom_op("mxfp4::quant_act", mutates_args=())
def quant_act(x: Tensor, layout: int) -> tuple[Tensor, Tensor]:
    """x [..., K] bf16 -> (codes, scales): [M, K/2] and [M, ceil(K/32)] for
    the row-major layout, flat buffers of the TILED layout otherwise."""
    _check_args("mxfp4::quant_act", x, dtypes=(torch.bfloat16,))
    c = _capi()
    K = x.shape[-1]
    x2 = x.reshape(-1, K).contiguous()
    M = x2.shape[0]
    nc, ns = _act_bytes(M, K, layout)
    codes = torch.empty(nc, dtype=torch.uint8, device=x.device)
    scales = torch.empty(ns, dtype=torch.uint8, device=x.device)
    c.mxfp4_quant_act(x2, M, K, K, codes, scales, layout, _stream(x))
    if layout == LAYOUT_ROWMAJOR:
        return codes.view(M, K // 2), scales.view(M, _cdiv(K, 32))
    return codes, scales


@quant_act.register_fake
def _(x, layout):
    _check_args("mxfp4::quant_act", x, dtypes=(torch.bfloat16,))
    K = x.shape[-1]
    M = x.numel() // K
    nc, ns = _act_bytes(M, K, layout)
    if layout == LAYOUT_ROWMAJOR:
        return x.new_empty(M, K // 2, dtype=torch.uint8), x.new_empty(M, _cdiv(K, 32), dtype=torch.uint8)
    return x.new_empty(nc, dtype=torch.uint8), x.new_empty(ns, dtype=torch.uint8)


# --------------------------------------------- fused RMSNorm -> quantizer
@custom_op("mxfp4::rmsnorm_quant_act", mutates_args=("residual",))
def rmsnorm_quant_act(x: Tensor, gamma: Tensor, eps: float, layout: int,
                      residual: Optional[Tensor]) -> tuple[Tensor, Tensor]:
    """RMSNorm of x [..., K] (or of x + residual, stored back into residual)
    times gamma, quantized per 1x32 like quant_act; returns (codes, scales)."""
    _check_args("mxfp4::rmsnorm_quant_act", x, gamma, residual,
                dtypes=(torch.bfloat16, torch.bfloat16, torch.bfloat16))
    torch._check(gamma.numel() == x.shape[-1], lambda: "mxfp4::rmsnorm_quant_act: gamma must have K elements")
    c = _capi()
    K = x.shape[-1]
    x2 = x.reshape(-1, K).contiguous()
    M = x2.shape[0]
    res2 = None
    if residual is not None:
        torch._check(residual.is_contiguous() and residual.shape == x.shape,
                     lambda: "mxfp4::rmsnorm_quant_act: residual must be contiguous and shaped like x")
        res2 = residual.view(M, K)
    nc, ns = _act_bytes(M, K, layout)
    codes = torch.empty(nc, dtype=torch.uint8, device=x.device)
    scales = torch.empty(ns, dtype=torch.uint8, device=x.device)
    c.mxfp4_rmsnorm_quant_act(x2, K, res2, K, gamma.contiguous(), eps, M, K, codes, scales, layout, None, 0,
                              _stream(x))
    if layout == LAYOUT_ROWMAJOR:
        return codes.view(M, K // 2), scales.view(M, _cdiv(K, 32))
    return codes, scales


@rmsnorm_quant_act.register_fake
def _(x, gamma, eps, layout, residual):
    _check_args("mxfp4::rmsnorm_quant_act", x, gamma, residual,
                dtypes=(torch.bfloat16, torch.bfloat16, torch.bfloat16))
    torch._check(gamma.numel() == x.shape[-1], lambda: "mxfp4::rmsnorm_quant_act: gamma must have K elements")
    K = x.shape[-1]
    M = x.numel() // K
    nc, ns = _act_bytes(M, K, layout)
    if layout == LAYOUT_ROWMAJOR:
        return x.new_empty(M, K // 2, dtype=torch.uint8), x.new_empty(M, _cdiv(K, 32), dtype=torch.uint8)
    return x.new_empty(nc, dtype=torch.uint8), x.new_empty(ns, dtype=torch.uint8)


# ----------------------------------------------------------------- GEMMs
def _workspace(M: int, N: int, K: int, device) -> tuple[Tensor, int]:
    nbytes = _capi().mxfp4_gemm_workspace_bytes(M, N, K)
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device), nbytes


@custom_op("mxfp4::linear", mutates_args=())
def linear(x: Tensor, w_packed: Tensor, bias: Optional[Tensor], N: int) -> Tensor:
    """y = x W^T + bias with x [..., K] bf16 quantized per 1x32 inside the
    call, W the packed FP4 weights of N rows; y [..., N] bf16."""
    _check_args("mxfp4::linear", x, w_packed, bias, dtypes=(torch.bfloat16, torch.uint8, torch.bfloat16))
    _check_weights("mxfp4::linear", w_packed, 1, N, x.shape[-1])
    _check_bias("mxfp4::linear", bias, N)
    c = _capi()
    K = x.shape[-1]
    x2 = x.reshape(-1, K).contiguous()
    M = x2.shape[0]
    out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    ws, nbytes = _workspace(M, N, K, x.device)
    b = bias.contiguous() if bias is not None else None
    c.mxfp4_gemm(x2, K, None, None, LAYOUT_ROWMAJOR, w_packed, b, out, N, M, N, K, ws, nbytes, _stream(x))
    return out.view(*x.shape[:-1], N)


@linear.register_fake
def _(x, w_packed, bias, N):
    _check_args("mxfp4::linear", x, w_packed, bias, dtypes=(torch.bfloat16, torch.uint8, torch.bfloat16))
    _check_weights("mxfp4::linear", w_packed, 1, N, x.shape[-1])
    _check_bias("mxfp4::linear", bias, N)
    return x.new_empty(*x.shape[:-1], N, dtype=torch.bfloat16)


def _check_prequant(codes, scales, layout, w_packed, bias, M, N, K) -> None:
    where = "mxfp4::linear_prequant"
    _check_args(where, codes, scales, w_packed, bias, dtypes=(torch.uint8, torch.uint8, torch.uint8, torch.bfloat16))
    _check_weights(where, w_packed, 1, N, K)
    _check_bias(where, bias, N)
    torch._check(layout in (LAYOUT_ROWMAJOR, LAYOUT_TILED), lambda: f"{where}: layout {layout}")
    torch._check(M > 0, lambda: f"{where}: M = {M} must be positive")
    nc, ns = _act_bytes(M, K, layout)
    torch._check(codes.numel() >= nc and scales.numel() >= ns,
                 lambda: f"{where}: codes / scales hold {codes.numel()} / {scales.numel()} bytes, {nc} / {ns} needed")


@custom_op("mxfp4::linear_prequant", mutates_args=())
def linear_prequant(codes: Tensor, scales: Tensor, layout: int, w_packed: Tensor, bias: Optional[Tensor], M: int,
                    N: int, K: int) -> Tensor:
    """The pages' pre-quantized (x_fp4, x_scales) input: codes and scales in
    `layout` (as from quant_act) against the packed weights; [M, N] bf16."""
    _check_prequant(codes, scales, layout, w_packed, bias, M, N, K)
    c = _capi()
    out = torch.empty(M, N, dtype=torch.bfloat16, device=codes.device)
    ws, nbytes = _workspace(M, N, K, codes.device)
    b = bias.contiguous() if bias is not None else None
    c.mxfp4_gemm(None, 0, codes.contiguous(), scales.contiguous(), layout, w_packed, b, out, N, M, N, K, ws, nbytes,
                 _stream(codes))
    return out


@linear_prequant.register_fake
def _(codes, scales, layout, w_packed, bias, M, N, K):
    _check_prequant(codes, scales, layout, w_packed, bias, M, N, K)
    return codes.new_empty(M, N, dtype=torch.bfloat16)


@custom_op("mxfp4::linear_mxfp4_out", mutates_args=())
def linear_mxfp4_out(x: Tensor, w_packed: Tensor, bias: Optional[Tensor], N: int) -> tuple[Tensor, Tensor]:
    """linear() with the MXFP4 output epilogue: the bf16 result quantized per
    1x32 along N, row-major codes [M, N/2] and scales [M, ceil(N/32)] (M =
    the flattened leading dims of x), ready for linear_prequant."""
    _check_args("mxfp4::linear_mxfp4_out", x, w_packed, bias, dtypes=(torch.bfloat16, torch.uint8, torch.bfloat16))
    _check_weights("mxfp4::linear_mxfp4_out", w_packed, 1, N, x.shape[-1])
    _check_bias("mxfp4::linear_mxfp4_out", bias, N)
    torch._check(N % 2 == 0, lambda: f"mxfp4::linear_mxfp4_out: N = {N} must be even")
    c = _capi()
    K = x.shape[-1]
    x2 = x.reshape(-1, K).contiguous()
    M = x2.shape[0]
    codes = torch.empty(M, N // 2, dtype=torch.uint8, device=x.device)
    scales = torch.empty(M, _cdiv(N, 32), dtype=torch.uint8, device=x.device)
    ws, nbytes = _workspace(M, N, K, x.device)
    b = bias.contiguous() if bias is not None else None
    c.mxfp4_gemm_mxfp4_out(x2, K, None, None, LAYOUT_ROWMAJOR, w_packed, b, codes, scales, M, N, K, ws, nbytes,
                           _stream(x))
    return codes, scales


@linear_mxfp4_out.register_fake
def _(x, w_packed, bias, N):
    _check_args("mxfp4::linear_mxfp4_out", x, w_packed, bias, dtypes=(torch.bfloat16, torch.uint8, torch.bfloat16))
    _check_weights("mxfp4::linear_mxfp4_out", w_packed, 1, N, x.shape[-1])
    _check_bias("mxfp4::linear_mxfp4_out", bias, N)
    torch._check(N % 2 == 0, lambda: f"mxfp4::linear_mxfp4_out: N = {N} must be even")
    M = x.numel() // x.shape[-1]
    return x.new_empty(M, N // 2, dtype=torch.uint8), x.new_empty(M, _cdiv(N, 32), dtype=torch.uint8)


def _check_split_cat(where: str, x: Tensor, w_packed: Tensor, bias: Optional[Tensor], z: Tensor, s1: int,
                     s2: int) -> tuple[int, int, int]:
    _check_args(where, x, w_packed, bias, z, dtypes=(torch.bfloat16, torch.uint8, torch.bfloat16, torch.bfloat16))
    torch._check(s1 >= 0 and s2 >= 0 and s1 + s2 > 0 and s1 % 8 == 0 and s2 % 8 == 0,
                 lambda: f"{where}: s1 = {s1}, s2 = {s2} must be multiples of 8, not both 0")
    torch._check(z.dim() == 3, lambda: f"{where}: z must be [M, H, s3]")
    M, H, s3 = z.shape
    torch._check(M == x.numel() // x.shape[-1], lambda: f"{where}: z has {M} rows, x {x.numel() // x.shape[-1]}")
    torch._check(s3 % 8 == 0, lambda: f"{where}: s3 = {s3} must be a multiple of 8")
    N = H * (s1 + s2)
    _check_weights(where, w_packed, 1, N, x.shape[-1])
    _check_bias(where, bias, N)
    return M, H, s3


@custom_op("mxfp4::linear_split_cat", mutates_args=())
def linear_split_cat(x: Tensor, w_packed: Tensor, bias: Optional[Tensor], z: Tensor, s1: int,
                     s2: int) -> tuple[Tensor, Tensor]:
    """linear() with the split + cat epilogue: the output's N = H (s1 + s2)
    columns as H groups; returns cat [M, H, s1 + s3] (each group's first s1
    columns, then z[m, h]) and split [M, H, s2] (its other s2 columns), with
    z [M, H, s3]."""
    M, H, s3 = _check_split_cat("mxfp4::linear_split_cat", x, w_packed, bias, z, s1, s2)
    c = _capi()
    K = x.shape[-1]
    N = H * (s1 + s2)
    x2 = x.reshape(-1, K).contiguous()
    cat = torch.empty(M, H, s1 + s3, dtype=torch.bfloat16, device=x.device)
    split = torch.empty(M, H, s2, dtype=torch.bfloat16, device=x.device)
    ws, nbytes = _workspace(M, N, K, x.device)
    b = bias.contiguous() if bias is not None else None
    zc = z.contiguous() if s3 else None
    c.mxfp4_gemm_split_cat(x2, K, None, None, LAYOUT_ROWMAJOR, w_packed, b, M, N, K, s1, s2, zc, s3,
                           cat if s1 + s3 else None, split if s2 else None, ws, nbytes, _stream(x))
    return cat, split


@linear_split_cat.register_fake
def _(x, w_packed, bias, z, s1, s2):
    M, H, s3 = _check_split_cat("mxfp4::linear_split_cat", x, w_packed, bias, z, s1, s2)
    return x.new_empty(M, H, s1 + s3), x.new_empty(M, H, s2)


@custom_op("mxfp4::a16wfp4_bmm", mutates_args=())
def a16wfp4_bmm(x: Tensor, w_packed: Tensor, N: int, batch_major: bool) -> Tensor:
    """x [B, M, K] bf16 against B packed FP4 weight matrices of N rows:
    [B, M, N], or [M, B, N] when batch_major (the V-up projection)."""
    _check_args("mxfp4::a16wfp4_bmm", x, w_packed, dtypes=(torch.bfloat16, torch.uint8))
    B, M, K = x.shape
    _check_weights("mxfp4::a16wfp4_bmm", w_packed, B, N, K)
    c = _capi()
    out = torch.empty(*((M, B, N) if batch_major else (B, M, N)), dtype=torch.bfloat16, device=x.device)
    c.a16wfp4_bmm(x.contiguous(), w_packed, out, B, M, N, K, c.OUT_MBN if batch_major else c.OUT_BMN, _stream(x))
    return out


@a16wfp4_bmm.register_fake
def _(x, w_packed, N, batch_major):
    _check_args("mxfp4::a16wfp4_bmm", x, w_packed, dtypes=(torch.bfloat16, torch.uint8))
    B, M, K = x.shape
    _check_weights("mxfp4::a16wfp4_bmm", w_packed, B, N, K)
    return x.new_empty(*((M, B, N) if batch_major else (B, M, N)), dtype=torch.bfloat16)
