"""CPU oracle for the fused dequantize-and-matvec path. TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product (the CUDA library and its
Python binding) never imports it and shares no code, table or constant with it.

Everything here is plain NumPy in float64 (float64 accumulation, IEEE
division, round-half-even), written from the pages' definitions:

* ``ternary``   - block-128 absmean ternary quantizer ("Ternary Bonsai 2",
                  section 1.2 ``block_ternary``; all-zero blocks section 3.4).
* ``int4``      - symmetric group-128 absmax/7 INT4 quantizer ("GPT-5.4 ...",
                  section 3.2).
* ``cassandra`` - lossless bf16 split ("Cassandra", sections 3.1-3.3): Wanda
                  value pruning into a bitmap, mantissa truncation, exponent
                  unary coding by per-tensor frequency rank, draft and exact
                  reconstruction.
* ``matvec``    - y = W_hat x in float64 and the per-row error bound term
                  sum_k |w_hat_k x_k|.
* ``moe``       - top-k routing, softmax over the selected experts, SwiGLU
                  experts and the weighted combine ("Nemotron 3.5 Bolt",
                  expert top-K routing section).
* ``layout``    - the packed byte layout of each format, written from its
                  specification (section offsets, bit positions).

Pins live in ``tests/test_oracle_*.py``. Every function has one; the exponent
entropy and mean unary code length (``cassandra.exponent_stats``) are pinned by
closed forms and the source-coding bound (the pages' own figures for them come
from trained models and are quoted as context only).
"""
