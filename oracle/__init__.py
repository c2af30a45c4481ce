"""CPU oracle for QuantMLA low-bit MLA decode attention -- TEST INFRASTRUCTURE.

This package is test infrastructure, not part of the library. Only the test
suite, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import or run it. The CUDA library never imports it and it
never imports the library: the two share no code, tables or helpers.

Everything here is a plain, slow, obviously correct restatement of what the
QuantMLA pages describe (see ``oracle/quantmla.py`` for citations):
  * per-token asymmetric affine quantizer, group size 64, fp16 (scale, min);
  * canonical bit packing of codes (for accounting and export comparisons);
  * dequantization in fp64;
  * the mixed-precision token selection rule (4 sink + 128 recent in BF16);
  * single-softmax MLA decode attention in fp64, plus the log-sum-exp merge of
    split partials;
  * the contents a fused writer must leave in the BF16 sink/recent ring.

Parity status of each function is listed in its docstring; every function is
pinned by ``tests/test_oracle.py`` to something other than itself.
"""

from .quantmla import *  # noqa: F401,F403
