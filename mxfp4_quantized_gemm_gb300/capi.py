"""ctypes binding of ``libmxfp4_gb300.so`` (declared in ``include/mxfp4.h``).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  Arguments that are device buffers accept a torch tensor (its
``data_ptr()``) or a raw integer address; ``stream`` accepts a
``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or ``None`` for torch's
current stream on the current device.  A non-OK status raises
``Mxfp4Error``.  Importing this module fails loudly when the library has not
been built (``python -m mxfp4_quantized_gemm_gb300.build``).  The environment
variable ``MXFP4_GB300_LIB`` selects another build of the same library (the
timeline build of ``bench.py --timeline``).
"""

from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.environ.get("MXFP4_GB300_LIB") or os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                               "libmxfp4_gb300.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build it with `python -m mxfp4_quantized_gemm_gb300.build` "
        "(there is no CPU fallback)")
lib = ctypes.CDLL(_LIB_PATH)

# status codes (mxfp4_status)
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_MISALIGNED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, \
    ERR_NO_DEVICE = range(8)
LAYOUT_ROWMAJOR, LAYOUT_TILED = 0, 1
OUT_BMN, OUT_MBN = 0, 1

_p, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t

_SIGNATURES = {
    "mxfp4_abi_version": (_i, []),
    "mxfp4_status_string": (ctypes.c_char_p, [_i]),
    "mxfp4_packed_weight_bytes": (_sz, [_i, _i, _i]),
    "mxfp4_pack_weights": (_i, [_p, _p, _i, _i, _i, _p, _p]),
    "mxfp4_weights_updated": (_i, [_p]),
    "mxfp4_act_code_bytes": (_sz, [_i, _i, _i]),
    "mxfp4_act_scale_bytes": (_sz, [_i, _i, _i]),
    "mxfp4_quant_act": (_i, [_p, _i, _i, _i, _p, _p, _i, _p]),
    "mxfp4_rmsnorm_quant_act": (_i, [_p, _i, _p, _i, _p, ctypes.c_float, _i, _i, _p, _p, _i, _p, _i, _p]),
    "mxfp4_gemm_workspace_bytes": (_sz, [_i, _i, _i]),
    "mxfp4_gemm": (_i, [_p, _i, _p, _p, _i, _p, _p, _p, _i, _i, _i, _i, _p, _sz, _p]),
    "mxfp4_gemm_mxfp4_out": (_i, [_p, _i, _p, _p, _i, _p, _p, _p, _p, _i, _i, _i, _p, _sz, _p]),
    "mxfp4_gemm_split_cat": (_i, [_p, _i, _p, _p, _i, _p, _p, _i, _i, _i, _i, _i, _p, _i, _p, _p, _p, _sz, _p]),
    "a16wfp4_bmm": (_i, [_p, _p, _p, _i, _i, _i, _i, _i, _p]),
    "mxfp4_get_device_error": (_i, [_p]),
    "mxfp4_gemm_noalloc": (_i, [_p, _i, _p, _p, _p, _i, _i, _i, _i, _p]),
    "mxfp4_gemm_noalloc_max_scratch_bytes": (_sz, []),
    "mxfp4_diag_max_units": (_i, []),
    "mxfp4_diag_tensor_rate_variants": (_i, []),
    "mxfp4_diag_tensor_rate_info": (_i, [_i, ctypes.POINTER(_i)]),
    "mxfp4_diag_tensor_rate": (_i, [_i, _i, _i, _i, _p, ctypes.POINTER(_i), _p]),
    "mxfp4_diag_pair_alloc_probe": (_i, [_p, _p]),
    "mxfp4_diag_set_wait_cycles": (_i, [ctypes.c_longlong]),
    "mxfp4_diag_decode_timeline": (_i, [_p, _sz, ctypes.POINTER(_i)]),
    "mxfp4_diag_gemm_pair": (_i, [_p, _i, _p, _p, _i, _p, _p, _p, _i, _i, _i, _i, _p, _sz, _p]),
}
for _name, (_res, _args) in _SIGNATURES.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class Mxfp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.mxfp4_status_string(status).decode()}")


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str) -> None:
    if status != OK:
        raise Mxfp4Error(status, where)


def mxfp4_abi_version() -> int:
    return lib.mxfp4_abi_version()


def mxfp4_status_string(status: int) -> str:
    return lib.mxfp4_status_string(status).decode()


def mxfp4_packed_weight_bytes(batch: int, N: int, K: int) -> int:
    return lib.mxfp4_packed_weight_bytes(batch, N, K)


def mxfp4_act_code_bytes(M: int, K: int, layout: int) -> int:
    return lib.mxfp4_act_code_bytes(M, K, layout)


def mxfp4_act_scale_bytes(M: int, K: int, layout: int) -> int:
    return lib.mxfp4_act_scale_bytes(M, K, layout)


def mxfp4_rmsnorm_quant_act(x, ldx: int, residual, ldr: int, gamma, eps: float, M: int, K: int, codes, scales,
                            layout: int, y=None, ldy: int = 0, stream=None) -> None:
    _check(lib.mxfp4_rmsnorm_quant_act(_ptr(x), ldx, _ptr(residual), ldr, _ptr(gamma), eps, M, K, _ptr(codes),
                                       _ptr(scales), layout, _ptr(y), ldy, _stream(stream)),
           "mxfp4_rmsnorm_quant_act")


def mxfp4_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib.mxfp4_gemm_workspace_bytes(M, N, K)


def mxfp4_pack_weights(w_codes, w_scales, batch: int, N: int, K: int, packed, stream=None) -> None:
    _check(lib.mxfp4_pack_weights(_ptr(w_codes), _ptr(w_scales), batch, N, K, _ptr(packed), _stream(stream)),
           "mxfp4_pack_weights")


def mxfp4_weights_updated(stream=None) -> None:
    _check(lib.mxfp4_weights_updated(_stream(stream)), "mxfp4_weights_updated")


def mxfp4_quant_act(x, M: int, K: int, ldx: int, codes, scales, layout: int, stream=None) -> None:
    _check(lib.mxfp4_quant_act(_ptr(x), M, K, ldx, _ptr(codes), _ptr(scales), layout, _stream(stream)),
           "mxfp4_quant_act")


def mxfp4_gemm(a_bf16, lda: int, a_codes, a_scales, a_layout: int, w_packed, bias, out, ldo: int,
               M: int, N: int, K: int, workspace, workspace_bytes: int, stream=None) -> None:
    _check(lib.mxfp4_gemm(_ptr(a_bf16), lda, _ptr(a_codes), _ptr(a_scales), a_layout, _ptr(w_packed),
                          _ptr(bias), _ptr(out), ldo, M, N, K, _ptr(workspace), workspace_bytes,
                          _stream(stream)),
           "mxfp4_gemm")


def mxfp4_gemm_mxfp4_out(a_bf16, lda: int, a_codes, a_scales, a_layout: int, w_packed, bias, out_codes,
                         out_scales, M: int, N: int, K: int, workspace, workspace_bytes: int, stream=None) -> None:
    _check(lib.mxfp4_gemm_mxfp4_out(_ptr(a_bf16), lda, _ptr(a_codes), _ptr(a_scales), a_layout, _ptr(w_packed),
                                    _ptr(bias), _ptr(out_codes), _ptr(out_scales), M, N, K, _ptr(workspace),
                                    workspace_bytes, _stream(stream)),
           "mxfp4_gemm_mxfp4_out")


def mxfp4_gemm_split_cat(a_bf16, lda: int, a_codes, a_scales, a_layout: int, w_packed, bias, M: int, N: int,
                         K: int, s1: int, s2: int, z, s3: int, out_cat, out_split, workspace, workspace_bytes: int,
                         stream=None) -> None:
    _check(lib.mxfp4_gemm_split_cat(_ptr(a_bf16), lda, _ptr(a_codes), _ptr(a_scales), a_layout, _ptr(w_packed),
                                    _ptr(bias), M, N, K, s1, s2, _ptr(z), s3, _ptr(out_cat), _ptr(out_split),
                                    _ptr(workspace), workspace_bytes, _stream(stream)),
           "mxfp4_gemm_split_cat")


def a16wfp4_bmm(x, w_packed, out, B: int, M: int, N: int, K: int, out_layout: int, stream=None) -> None:
    _check(lib.a16wfp4_bmm(_ptr(x), _ptr(w_packed), _ptr(out), B, M, N, K, out_layout, _stream(stream)),
           "a16wfp4_bmm")


def mxfp4_gemm_noalloc(a_bf16, lda: int, w_packed, bias, out, ldo: int, M: int, N: int, K: int,
                       stream=None) -> None:
    _check(lib.mxfp4_gemm_noalloc(_ptr(a_bf16), lda, _ptr(w_packed), _ptr(bias), _ptr(out), ldo, M, N, K,
                                  _stream(stream)),
           "mxfp4_gemm_noalloc")


def mxfp4_gemm_noalloc_max_scratch_bytes() -> int:
    return lib.mxfp4_gemm_noalloc_max_scratch_bytes()


def mxfp4_get_device_error(stream=None) -> int:
    return lib.mxfp4_get_device_error(_stream(stream))


# ---- diagnostics (include/mxfp4_diag.h): measurements of the hardware, not the linear

def mxfp4_diag_max_units() -> int:
    return lib.mxfp4_diag_max_units()


def mxfp4_diag_tensor_rate_variants() -> int:
    return lib.mxfp4_diag_tensor_rate_variants()


def mxfp4_diag_tensor_rate_info(variant: int) -> dict:
    """The instruction mix of one measurement variant."""
    info = (_i * 7)()
    _check(lib.mxfp4_diag_tensor_rate_info(variant, info), "mxfp4_diag_tensor_rate_info")
    return dict(zip(("pair", "kind", "mmas", "copies", "form", "issuers", "split"), list(info)))


def mxfp4_diag_tensor_rate(variant: int, mma_n: int, steps: int, depth: int, ns_dev, stream=None) -> int:
    """Launches the issue-rate measurement; returns the number of units (CTAs or pairs) whose
    elapsed nanoseconds land in ``ns_dev`` once the stream has finished."""
    units = _i(0)
    _check(lib.mxfp4_diag_tensor_rate(variant, mma_n, steps, depth, _ptr(ns_dev), ctypes.byref(units),
                                      _stream(stream)),
           "mxfp4_diag_tensor_rate")
    return units.value


def mxfp4_diag_pair_alloc_probe(addr_dev, stream=None) -> None:
    _check(lib.mxfp4_diag_pair_alloc_probe(_ptr(addr_dev), _stream(stream)), "mxfp4_diag_pair_alloc_probe")


def mxfp4_diag_set_wait_cycles(cycles: int) -> None:
    _check(lib.mxfp4_diag_set_wait_cycles(cycles), "mxfp4_diag_set_wait_cycles")


def mxfp4_diag_gemm_pair(a_bf16, lda: int, a_codes, a_scales, a_layout: int, w_packed, bias, out, ldo: int,
                         M: int, N: int, K: int, workspace, workspace_bytes: int, stream=None) -> None:
    """mxfp4_gemm on the CTA-pair kernel; raises Mxfp4Error (MXFP4_ERR_UNSUPPORTED_SHAPE) where it
    does not apply."""
    _check(lib.mxfp4_diag_gemm_pair(_ptr(a_bf16), lda, _ptr(a_codes), _ptr(a_scales), a_layout, _ptr(w_packed),
                                    _ptr(bias), _ptr(out), ldo, M, N, K, _ptr(workspace), workspace_bytes,
                                    _stream(stream)),
           "mxfp4_diag_gemm_pair")


def mxfp4_diag_decode_timeline():
    """(stamps [64 calls][256 CTAs][8 points] uint64 ns as a numpy array, next call slot) from the
    timeline build; raises Mxfp4Error on the default build."""
    import numpy as np
    buf = np.zeros((64, 256, 8), dtype=np.uint64)
    nxt = _i(0)
    _check(lib.mxfp4_diag_decode_timeline(buf.ctypes.data, buf.nbytes, ctypes.byref(nxt)),
           "mxfp4_diag_decode_timeline")
    return buf, nxt.value
