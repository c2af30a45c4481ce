"""libmlaq: QuantMLA low-bit MLA decode attention over a paged dual-path cache.

The compute runs in the CUDA library ``libmlaq.so`` (built in-tree by
``bit_mla_kv_gb300.build.build()``); this package only marshals arguments.
Importing the package does not load the library; ``bit_mla_kv_gb300.mlaq``
does, and raises if it is missing.
"""

MODES = {"C4R4": 0, "C2R4": 1, "BF16": 2}
