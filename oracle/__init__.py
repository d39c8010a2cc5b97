"""CPU oracle for the MXFP4 dense linear: test infrastructure, never product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.
"""

from . import mxfp4_ref, tile_layout  # noqa: F401
