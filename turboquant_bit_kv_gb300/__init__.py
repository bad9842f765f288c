"""GB300-native TurboQuant KV-cache compression.

The compute path lives in the C-ABI library ``libtq.so`` (hand-written CUDA
for sm_103a, declared in ``include/tq.h``); ``turboquant_bit_kv_gb300.tq``
is the thin ctypes binding over it and ``workloads`` draws seeded inputs.
"""
