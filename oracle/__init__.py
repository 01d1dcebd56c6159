"""fp64 CPU oracle for paged GQA decode attention — TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library (``paged_gqa_decode_kvd_gb300``) and neither imports the other.

Parity pins (all in ``tests/test_oracle.py``, run with ``-m "not gpu"``):
e4m3 and e5m2 decode/encode, row quantise in both formats, the mixed-precision
pool, half-precision rounding, the low-bit (INT4 / 2-bit) group quantise and
its pool, the angle-domain key rows and query and their pool, the paged gather, decode
attention, the
split-free softmax statistics, the importance-score update and the block tier
plan are each pinned
to something other than the oracle itself; no function here is "parity
unpinned".
"""

from .oracle import (  # noqa: F401
    build,
    lib_path,
    e4m3_decode,
    e4m3_encode,
    quantize_rows,
    quantize_rows_fmt,
    e5m2_decode,
    e5m2_encode,
    FMT_BF16,
    FMT_E4M3,
    FMT_E5M2,
    round_half_sat,
    quantize_rows_lowbit,
    angle_key_rows,
    angle_query,
    OraclePool,
    decode,
    score_update,
    tier_plan,
    decode_dense_inputs,
)
