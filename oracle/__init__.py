"""Float64 CPU oracle for the DeMo / FlexDeMo per-shard optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code,
tables or constants with the CUDA library.
"""

from .demo_ref import *  # noqa: F401,F403
