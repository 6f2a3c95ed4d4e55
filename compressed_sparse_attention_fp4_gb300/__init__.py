"""GB300 (sm_103a) CSA2 decode hot path: FP4 main-KV codec, hierarchical
sparse indexer and sparse MLA decode attention, as a C-ABI CUDA library.

Modules:
  csa2   -- ctypes binding of libcsa2.so (loads the library; raises if absent)
  step   -- decode-step runner over a layer schedule (optionally CUDA-graphed)
  synth  -- seeded synthetic inputs (no method arithmetic)
  build  -- nvcc build of libcsa2.so
"""
