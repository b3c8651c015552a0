"""CPU oracle for MXFP8 block-scaled attention.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the
CUDA library in ``block_scaled_mxfp8_gb300/`` and never imports it.
"""
