"""Plain fp64 CPU oracle for row-indexed attention over a unified KV pool.

TEST INFRASTRUCTURE ONLY.  Nothing in the product library imports, links or
runs this package; only the tests, the smoke check and the benchmark's CPU
baseline leg do.  It shares no code with the CUDA path: it widens the raw
16-bit inputs itself, gathers rows with numpy indexing and uses a two-pass
softmax written out step by step.

What it follows ("llama.cpp 0.9.0 inference boundaries", section 1, the
``ggml_flash_attn_ext_rows`` paragraph): K/V stay in one shared pool; each
query slice carries an integer ``kv_rows`` list of the pool rows it needs; a
negative row index is padding and its mask entry is minus infinity.  The next
paragraph of the same section fixes that the result is exact attention over
the listed rows (no lossy summary, no importance-based dropping).  The old
path it replaces built a dense mask over the whole unified cache; that form is
written out separately as ``attend_dense`` and serves as a cross-check.

Paged INT8 KV with 64-token pages follows the v100llm article (sections 1-2);
the sinks + recent + top-k row-list builder its section 5 (``select_rows``).

Every function here is pinned by tests in ``tests/test_oracle_*.py`` against
closed forms, invariants, brute force on tiny inputs and the dense-mask form;
the page-table expansion and the INT8 codec are pinned by hand-worked cases and
exact rational checks.  Functions that carry no such pin say so in their
docstring with the words "parity unpinned".
"""
from .attention import attend_rows, attend_dense, visible_positions  # noqa: F401
from .kvcache import (  # noqa: F401
    widen_bf16, widen_f16, widen, quantize_int8, dequantize_int8, pack_scales, unpack_scales,
    page_table_to_rows, quantize_int4, dequantize_int4, append_rows,
    e4m3_value, e4m3_encode, quantize_fp8, dequantize_fp8,
)
from .sparse import select_rows  # noqa: F401
