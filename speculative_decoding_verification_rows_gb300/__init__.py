"""GB300-native speculative-decoding verify step.

The compute path is the C-ABI library ``libsv.so`` (hand-written sm_103a CUDA
kernels behind ``include/sv.h``); ``sv`` is its thin Python binding and
``workloads`` builds seeded synthetic inputs.
"""
