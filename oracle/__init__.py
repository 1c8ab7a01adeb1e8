"""fp64 CPU oracle for the LOCKS decode step — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
path (the CUDA library and its Python binding) never imports, calls or links it,
and the two share no code: no kernels, helpers, tables or pre/post-processing.
The only thing both sides use is the seeded input generator in ``synth``.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
to closed forms, invariants, textbook routines or brute force, except the
constants of the output-error bound of Theorem 1 (not printed on the pages):
that bound itself is "parity unpinned"; only its monotone consequence is tested.
"""

from .locks_oracle import *  # noqa: F401,F403
