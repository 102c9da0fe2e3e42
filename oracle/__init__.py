"""Float64 CPU oracle for speculative-decoding verification.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs may import this package. It shares no code with the CUDA path.
"""
