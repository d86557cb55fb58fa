"""Oracle for the Prof-K top-k engine.  TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU statement of what the engine computes,
written from the Prof-K paper ("Prof-K: Probabilistic One-Pass Filtering for
Efficient Top-k Selection") and the GPU.js top-k / radix-sort / compaction
exercises it is checked against.  It shares no code with the CUDA path and
neither imports the other.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or execute anything here.

Modules:
  plain   -- exact top-k by definition (C++ nth_element + sort, via ctypes),
             the rank R of a threshold element, the t-th sampled order statistic.
  params  -- Algorithm 1 (adaptive (S, t, M)) as printed, and the exact-tail
             reading of its t and M that the engine uses by default.
  philox  -- Philox4x32-10 (Salmon et al., SC'11) and the uniform index sampler.

Parity status per function is stated in each module's header.
"""
