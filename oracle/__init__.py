"""CPU oracle (float64 NumPy) for KV-cached grouped-query attention — test infrastructure only.

Only `tests/`, `__graft_entry__.smoke()` and the CPU baseline leg of `bench.py` may import it.
"""
