"""fp64 CPU oracle of the batch-1 decode layer (test infrastructure only).

Only tests/, ``__graft_entry__.smoke()`` and the benchmark's cpu_baseline /
reference leg may import this package; the CUDA library never does.
"""
