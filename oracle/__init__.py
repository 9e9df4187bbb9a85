"""CPU oracle for MoE dispatch / combine: test infrastructure only.

Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of bench.py
use this package. The CUDA library never imports, links or calls it.
"""
