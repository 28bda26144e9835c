"""Batch-invariant per-token policy statistics over a wide vocabulary on GB300.

The computation lives in ``libpstat.so`` (hand-written sm_103a CUDA behind the
C ABI of ``include/pstat.h``).  ``vocab_wide_token_gb300.pstat`` is its ctypes
binding; importing it raises when the library has not been built (there is no
CPU fallback).  ``vocab_wide_token_gb300.tp`` runs the vocabulary-parallel
path over a torch.distributed group, ``vocab_wide_token_gb300.inputs`` holds
the seeded synthetic workloads and ``vocab_wide_token_gb300.build`` the nvcc
build.
"""

__all__ = ["pstat", "tp", "inputs", "build"]
