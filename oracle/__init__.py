"""CPU oracle of the layer-range stage forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
anything here: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may.  The oracle shares no code with the CUDA path; the two
meet only in the seeded inputs of ``synth``.

It is a plain, slow, float64 restatement of what a stage computes, each function
citing the passage it follows.  Parity pins for every function live in
``tests/test_oracle_*.py``; see ``model.py`` for the list of what pins what.
"""
from .model import *  # noqa: F401,F403
