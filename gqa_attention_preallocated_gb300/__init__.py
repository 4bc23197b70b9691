"""GQA attention over a preallocated KV cache, native to GB300 (sm_103a).

The compute path is the C-ABI library ``libkvc.so`` built from ``csrc/``;
this package only marshals arguments to it.  ``workloads`` holds the seeded
synthetic input generators.
"""
