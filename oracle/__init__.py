"""CPU oracle for the CSA2 decode hot path (test infrastructure only).

This package is the slow, plain, fp64 statement of what the CUDA library
computes.  It exists to check that library: only the test-suite, the smoke
check of ``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  The product path never calls into it and
it never calls into the product path; the two share no code, tables or
constants.  The only thing both sides consume is the seeded synthetic inputs
made by ``compressed_sparse_attention_fp4_gb300.synth``, which holds none of the
method's arithmetic.

Sources (web pages, cited by title and section):

* [P1] newsaint.id, "DeepSeek-V4.1-Flash 2026: Arsitektur Causal
  Encoder-Decoder (CED), Compressed Sparse Attention 2 (CSA2), FP4 KV Caching,
  dan SWA Bounded Replay untuk 1M Context Window" -- section 3 (Hierarchical
  Sparse Indexer), section 4 (FP4 main KV), section 8 (PyTorch simulation:
  ``FP4Quantizer``, ``HierarchicalSparseIndexer``).
* [P2] stamatios.com, "DeepSeek-V4.1 Flash comprime cache KV para 890 bytes por
  token" -- section "CSA2: compressão em três dimensões".
* [P3] foosynaptic mechanism atlas, "DeepSeek-V4.1-Flash 梗概" -- section 3.2
  (CSA2 mode table, Hierarchical Sparse Indexer, FP4 main KV).
* [P4] abrarakhunji.com, "DeepSeek-V4.1-Flash Architecture: Causal
  Encoder-Decoder (CED), 890-Byte KV Cache, Engram Memory, and CSA2" --
  section 3 (CSA2 layer modes, FP4 E2M1).

Modules:

* ``codec``     -- E2M1 / E4M3 formats, FP4 KV quantize / dequantize.
* ``indexer``   -- indexer scores, block scores, pool and Top-K selection.
* ``indexer_fp4`` -- the indexer with FP4 query and key (a next row: pinned,
  no kernel yet).
* ``attention`` -- joint softmax over the selected main KV and the SWA window.
* ``schedule``  -- Full / Reindex / Reuse layer schedules.

Parity status: every function here is pinned by a ``-m "not gpu"`` test
against something other than itself (exact rational arithmetic, brute force,
closed forms, textbook dense attention).  No function is "parity unpinned".
"""
