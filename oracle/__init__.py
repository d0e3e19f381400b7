"""CPU oracle of the GPT-2 training step -- test infrastructure only.

Imported by the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg; never by the CUDA library or its Python binding.
"""
