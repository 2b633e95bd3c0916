"""CPU oracle for the CSA2 layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
``--impl reference`` leg may import this package.  The product path (the
``sparse_attention_prefill_gb300`` package and its CUDA library) never does.
The oracle shares no code with the CUDA path; see ``csa2_oracle.c``.
"""
