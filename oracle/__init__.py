"""fp64 CPU oracle for softcapped / sink / masked attention -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, loads or calls it, and the two share no code.

The arithmetic lives in ``attn_oracle.c`` (plain fp64 loops, one function per
quantity of the method); this module only compiles it with gcc and marshals
numpy arrays through ctypes.  See the header of ``attn_oracle.c`` for the
definition it writes out and the passages it follows.
"""
from .oracle import (  # noqa: F401
    Problem,
    build,
    forward,
    backward,
    rowdot,
    count_visible,
    capped,
    cap_factor,
    visible,
    row_visible,
    col_visible,
)
