"""ParisKV decode-time KV-cache retrieval for GB300 (sm_103a).

The compute path lives in a C-ABI CUDA library (``csrc/``, declared in
``include/paris.h``); ``paris`` is its thin ctypes binding.
"""
