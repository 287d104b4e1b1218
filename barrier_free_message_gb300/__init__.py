"""barrier_free_message_gb300: barrier-free small-message AllReduce for simulated
ranks on one GB300 (sm_103a).

The compute path is the CUDA library ``libsfar`` behind a C ABI
(``include/sfar.h``); :mod:`barrier_free_message_gb300.sfar` is the thin
ctypes binding.  The library is loaded on first use and its absence is an
error: there is no CPU fallback.
"""
