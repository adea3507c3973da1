"""Float64 CPU oracle for the Variational Linear Attention (VLA) forward scan.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may import or run it.  It shares no code with
the CUDA path; the two meet only in the seeded inputs of ``workloads``.

Modules
-------
``vla_ref``   the sequential recurrence, step by step, as the pages state it
              (additive state write, and the delta-rule variant with
              ``rule="delta"``), and the direction projection ``project_u``.
``woodbury``  the same recurrence taken a chunk of steps at a time in exact
              Woodbury / LDL^T form (the design the chunked GPU kernel follows),
              checked against ``vla_ref`` by the tests.
"""
from .vla_ref import GUARD_EPS, READOUT_EPS, phi, scan, errors, project_u  # noqa: F401
from .woodbury import scan_chunked, ldl_unit  # noqa: F401
