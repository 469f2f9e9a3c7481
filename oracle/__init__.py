"""fp64 CPU oracle for exact attention -- test infrastructure only.

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg and reference arm.  It shares no code with the CUDA path.
"""
from .attention import (  # noqa: F401
    BF16_U,
    FP32_STEP,
    NEG_INF,
    backward,
    backward_rows,
    backward_dropout,
    backward_rows_dq,
    decode,
    decode_split,
    decode_visible,
    dropout_bytes,
    dropout_keep,
    dropout_threshold,
    e4m3_decode,
    forward_dropout,
    forward_error_bound,
    forward_fp8,
    fp8_error_model,
    grad_error_model,
    forward,
    forward_rows,
    dilated_block_mask,
    head_probs,
    merge_stats,
    philox4x32_10,
    tiled_forward,
    visible,
    window_block_mask,
)
