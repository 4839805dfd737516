"""CPU oracle for the DSA sparse-attention path -- test infrastructure only.

Importable by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg; never by the product package.
"""
