"""Paged-KV GQA attention hot path for GB300 (sm_103a).

The compute path is the C-ABI library ``libpa.so`` built from ``csrc/``;
``pa`` is its thin ctypes binding.  ``workloads`` draws seeded synthetic
inputs.
"""
