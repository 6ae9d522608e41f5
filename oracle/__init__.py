"""CPU oracle for the transposed convolution -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product path (the CUDA
library and its Python binding) never imports, loads or calls it.

The arithmetic lives in ``ct_oracle.c`` (plain C, double precision, single
threaded); this module only builds it with gcc and marshals numpy arrays.
``ct_oracle_mt.c`` is the same scatter definition split over the host cores
by output slice: the benchmark's all-cores CPU baseline, never used to check
results (a test compares it with the parity oracle).
"""
from .oracle import (  # noqa: F401
    build_oracle,
    out_len,
    conv_transpose,
    conv_transpose_at,
    conv_direct,
    add_hswish,
    oracle_library_path,
    build_oracle_mt,
    conv_transpose_mt,
    host_cores,
)
