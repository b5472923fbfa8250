"""CPU oracle of the ZeRO-3 per-step shard data path.  TEST INFRASTRUCTURE.

Only the tests, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or calls it, and this package shares no
code with the product: the only module both sides use is `synth`, which
draws the synthetic inputs and holds none of the step's arithmetic.

The oracle is plain and slow on purpose: integer logic in plain Python,
floating point in numpy float32 element-wise operations in exactly the order
the method states (each operation rounds to float32; numpy does not contract
a*b+c into an FMA), the gradient norm in float64 with an exactly rounded sum.

Sources.  Citations name the page and the section on it:
  [ZeRO-3 chapter]  "03 · ZeRO-3：参数分片与 all-gather 调度"
                    (DeepSpeed code-reading chapter, ai-reference-codex)
  [Grok blog]       "DeepSpeed ZeRO Stage 3：参数分区，让大模型训练“零负担”"
  [Core flow]       "ZeRO-3 核心流程：把参数也切开的那一档" (llmnex)

Modules
  plan  - A1: partition sizes, padding, layouts, reduce / gather buckets,
          sub-groups, per-rank memory accounting.
  bf16  - float32 <-> bfloat16 conversion (round to nearest even).
  step  - A1 data movement (partition of full weights), A2 reduce-scatter,
          A3 global norm and clip coefficient, A4 AdamW / Adam-L2 with the
          bf16 cast, A5 all_gather_coalesced, and the whole step.

Parity status: every function is pinned by tests/test_oracle_*.py against
the pages' worked example, closed forms, invariants, brute force or a
library routine (torch.optim.AdamW, torch's bfloat16 cast,
torch.nn.utils.clip_grad_norm_, numpy.linalg.norm).  The choices the pages
leave open (listed as readings in the design notes) are conventions that
both sides follow; no external value fixes them.
"""
