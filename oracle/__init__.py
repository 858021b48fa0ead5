"""Plain fp64 CPU oracle for the Muon step over stacked parameter banks.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package; only the test suite, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, helpers or constant
tables); its inputs come from the seeded generators in ``synth``.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, invariants, library routines or brute force, except the
NorMuon variant, whose formula the speedrun pages name but never define.  Its
invariants are pinned, but its formula is a reading of the published NorMuon
method and is "parity unpinned" relative to the pages.
"""
from .muon_oracle import *  # noqa: F401,F403
