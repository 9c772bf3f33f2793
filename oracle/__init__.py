"""Float64 CPU oracle for exact tiled attention, flash-decoding and RMSNorm.

TEST INFRASTRUCTURE ONLY. This package is the slow, obviously correct
definition that the CUDA path is checked against. Only the tests, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it; the library (``exact_tiled_attention_attn_gb300``) never does, and
this package imports nothing from the library.

Every function works in float64 on inputs decoded exactly from bfloat16, and
cites the passage of the source pages it writes out. The pages are:

* "Module 07: Fused operators and FlashAttention" (LLM Inference Systems course)
* "FlashAttention: attention without the n x n matrix" (GPU-internals lesson)
* "Attention from the kernel's side: FlashAttention, online softmax and fused
  dequantisation" (note, in Polish)
* "Chapter 5. Operators and runtime", sections 5.3.3 "FlashAttention: tiling
  and online softmax" and 5.4.3 (rounding and FP8 scales; book chapter)
* "How does FlashAttention-3 work mathematically" (Q&A page), section 6 (FP8)

Parity status: every function here is pinned by the tests in
``tests/test_oracle_pins.py`` and ``tests/test_oracle_fp8_pins.py`` (worked
examples printed on the pages, closed forms, brute force on tiny inputs, the
recurrence-equals-three-pass identity, and the FP8 format's defining values). No function is "parity unpinned".
"""
from .attention import (  # noqa: F401
    scores_softmax_weighted,
    online_softmax_blocks,
    online_normalizer,
    online_weighted_stream,
    attention,
    attention_rows,
    attention_online,
    decode,
    decode_split_merge,
    count_blocks,
    attention_backward,
    attention_backward_rows,
)
from .rmsnorm import rmsnorm, rmsnorm_residual  # noqa: F401
from .fp8 import (  # noqa: F401
    E4M3_MAX,
    e4m3_value,
    e4m3_table,
    e4m3_encode,
    head_scale,
    quantize_block,
    quantize_kv,
    dequantize_kv,
    decode_fp8,
)
