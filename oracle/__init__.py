"""CPU oracle for the W4A16 layer: TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package; the product path never does.
"""
from .w4a16_oracle import (  # noqa: F401
    dequantize,
    pack_cols,
    pack_rows,
    reference,
    reference_cols,
    reference_rows,
    round_to_act,
    unpack_cols,
    unpack_rows,
    widen,
)
