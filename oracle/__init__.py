"""fp64 CPU oracle for the exact attention forward (test infrastructure only).

Imported by the tests, the smoke check and the benchmark's CPU-baseline leg;
never by the product path, which runs only the CUDA library.
"""
from .attention import (  # noqa: F401
    attention_forward,
    attention_rows,
    combine,
    lse_to_row_order,
    sequences,
    split_forward,
    visible_count,
    visible_mask,
    widen,
)
from .kvcache import dequant_kv, fp8_to_float, gather_pages, plain_kv  # noqa: F401,E402
from .backward import attention_backward  # noqa: F401,E402
