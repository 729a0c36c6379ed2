"""Float64 CPU oracle for the sample · filter · capture step.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may import it. The CUDA path never does.
"""
from .philox import philox4x32_10, race_uniform  # noqa: F401
from .sfc_oracle import (  # noqa: F401
    DT_BF16,
    DT_F32,
    ROW_BADPARAM,
    ROW_OK,
    ROW_OVERFLOW,
    BatchResult,
    RowResult,
    row_params_ok,
    sample_filter_capture,
    greedy_row,
    pack_results,
    sample_row,
    support_bits,
    widen_logits,
)
from .replay import ROW_OUTSIDE, ReplayResult, replay_logprob, replay_row  # noqa: F401
from .pack import pack_supports  # noqa: F401
