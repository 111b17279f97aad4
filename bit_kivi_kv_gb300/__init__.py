"""KIVI-style low-bit KV cache with decode attention on GB300 (sm_103a).

``bit_kivi_kv_gb300.kivi`` is the ctypes binding of the C ABI (include/kivi.h);
it loads libkivi.so on import.  ``bit_kivi_kv_gb300.synth`` draws the seeded
synthetic inputs.  ``bit_kivi_kv_gb300.build`` compiles the CUDA library.
Importing the package itself loads nothing.
"""
