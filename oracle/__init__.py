"""CPU oracle of the ParisKV retrieval path -- test infrastructure only.

Imported by the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline
and reference legs of ``bench.py``; never by the CUDA library or its binding.
"""
from . import pariskv  # noqa: F401
