"""CPU oracle for the flash-attention backward (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never touches it.
It wraps ``fa_oracle.c`` (plain C, double precision, one thread per core),
which is compiled here with gcc and shares no code with the CUDA path.
"""
from .oracle import (  # noqa: F401
    build, lib_path, half_to_double, dequant, fa_back, fa_forward, default_threads,
)
