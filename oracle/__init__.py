"""CPU oracle for the rotated low-bit KV cache — TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct restatement of what the source pages
define (SJ-KVaRN; KV Cache Precision Tail; KV cache math; HAL #582), written with numpy.
Codec arithmetic follows the fixed fp32 rules of the format specification (one IEEE
rounding per operation, halving-tree sums, round-half-even); attention is the plain
softmax definition evaluated in fp64 over the dequantized values.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import anything from here. The product path (the CUDA library and its
Python binding) never imports, links or executes this package, and the oracle imports
nothing from the product.

Parity pins: every function is pinned by a ``-m "not gpu"`` test against something other
than itself (library routines, closed forms, printed numbers, brute force). The only
function without an external pin of its exact output is the KVarN balancing schedule
(``kvarn.balance``): the pages print no worked example, so its exact scales are
"parity unpinned" and only its invariants are pinned.
"""

from . import fp, tables, rotation, codecs, kvarn, sizes, attention, cache  # noqa: F401
