"""Plain, slow CPU oracle for the partitioned mixed-precision ZeRO step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library under
``zero_partitioned_mixed_gb300/csrc``.

Every function cites the passage of the ZeRO pages it restates; the
numerics the pages leave open (Adam's exact form, loss scaling, clipping)
follow the readings written at the top of :mod:`oracle.zero_oracle`.
"""

from .zero_oracle import *  # noqa: F401,F403
