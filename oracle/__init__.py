"""fp64 CPU oracle for MLA decode with matrix absorption.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arms of ``bench.py`` use it.  It shares no code with the CUDA
library (no kernels, headers, helpers or constants).

Modules
-------
``oracle.mla``         the decode step written out as its plain definition
                       (un-absorbed: K and V are reconstructed per cached token),
                       also over one block range of the keys, and the
                       log-sum-exp merge of such pieces
``oracle.prefill``     prefill in the standard order: K and V rebuilt from the
                       latents, then causal attention over d_k and d_v
``oracle.upstream``    down-projection and RoPE, used only to synthesise the
                       inputs of the tiny fp32 workload
``oracle.accounting``  closed-form cache sizes and FLOP counts

Every function is pinned by ``tests/test_oracle_*.py`` to numbers the pages
print, to closed forms, to textbook special cases or brute force on tiny
inputs, or to invariants that tie it to a pinned function.
"""

from . import accounting, mla, prefill, upstream  # noqa: F401
