"""Plain, slow, fp64 CPU oracle for split-KV sparse-MLA decode and dense FP8 SDPA decode.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it. It shares no code, headers, tables or helpers with the
CUDA library; the two meet only at the seeded inputs of
``split_kv_sparse_gb300.workloads`` (which holds no attention arithmetic).

Modules:
  codecs -- bf16 and FP8 e4m3 round-to-nearest-even encoders written from the
            formats' definitions (1-8-7 and 1-4-3/bias 7/no infinities).
  mla    -- sparse-MLA attention as its plain definition, the split-KV row
            partition, per-split partials, the log-sum-exp combine, the
            attention sink, the output casts and the workspace formula.
  sdpa   -- dense GQA causal decode attention on FP8 codes with per-tensor
            descales, its split-KV chunking and the combine's amax.

Pins (tests/test_oracle_*.py) tie every function to something other than
itself: torch's fp64 SDPA and logsumexp library routines, closed forms,
the workspace sizes printed in FlashMLA PR #25 ("Measured"), exhaustive
codec checks against torch's own float8/bfloat16 conversions, and split
invariance. The attention values themselves are not printed on any page,
so no page-printed attention value pins them.
"""
