"""Oracle for the paged KV cache hot path: plain, slow, fp64, CPU only.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and bench.py's
cpu_baseline / reference leg may import, call or run anything under this package.
It shares no code with the CUDA library and never imports it.
"""
