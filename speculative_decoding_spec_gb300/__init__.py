"""GB300 (sm_103a) MTP speculative decoding: drafter -> one-pass verify -> greedy accept.

The hot path lives in libspec_gb300.so (C ABI in include/spec.h), built from
csrc/ by build.py; binding.py is its ctypes binding.
"""
