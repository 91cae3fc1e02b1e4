"""Stream-K GEMM with online ABFT for GB300 (sm_103a).

The compute path is the C-ABI library ``libskgemm.so`` built from ``csrc/``;
``skgemm`` is its thin ctypes binding (argument marshalling only).
"""
