"""MXFP4 block-scaled dense linear for GB300 (sm_103a).

The compute lives in ``libmxfp4_gb300.so`` (hand-written CUDA behind a C ABI,
declared in ``include/mxfp4.h``).  ``capi`` is its thin ctypes binding; its
import fails loudly when the library has not been built.  ``ops`` registers
the same calls as PyTorch custom operators (``torch.ops.mxfp4.*``) with shape
-only fake implementations; it loads the library on the first real call.
``synth`` makes seeded synthetic inputs and does not need the library.
"""

import importlib


def __getattr__(name):
    # Binding names resolve through ``capi`` on first use, so that importing
    # ``mxfp4_quantized_gemm_gb300.synth`` does not require the built library.
    if name.startswith("_") or name in ("synth", "capi", "build", "ops"):
        raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
    capi = importlib.import_module(".capi", __name__)
    try:
        return getattr(capi, name)
    except AttributeError:
        raise AttributeError(f"module {__name__!r} has no attribute {name!r}") from None
