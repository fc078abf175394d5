"""CSA / HCA single-token decode over a low-bit compressed KV cache, on B300.

The compute path is the CUDA library ``libdsv4.so`` (built for sm_103a from
``csrc/``); ``dsv4`` is its thin ctypes binding. ``workloads`` describes the
measured shapes and ``synth`` draws seeded inputs.
"""
