"""CPU oracle for the MoE speculative verify step.

TEST INFRASTRUCTURE ONLY: plain, slow, fp64 (fp32 where the method fixes the
precision) Python/numpy code written from the EcoSpec and S2-MoE write-ups.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA library, and the
CUDA library never imports it.
"""
