"""CPU oracle for batch-invariant split-KV decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code, constants or helpers with the
CUDA library; the two meet only on the seeded inputs of
``invariant_decode_attention_gb300.workloads``.

What it computes and where that is stated:

* ``attention.attend`` -- plain softmax attention of one query row over its
  own KV list (contiguous, paged or top-k index-gathered), in fp64.  Source:
  "Sparse MLA decode is not batch-invariant" (FlashMLA issue #212), Summary
  and Measurement sections (the call ``flash_mla_with_kvcache(q, indices,
  topk_length, ...)`` and its per-row output + LSE).
* ``attention.lse_merge`` -- the log-sum-exp merge of per-split partials.
  Source: same page, "Where it comes from" (the ``combine.cu`` loop that
  rescales each split's partial by its LSE weight and sums in fp32).
* ``plan.plan_invariant`` -- per-row split plan whose count and boundaries
  depend only on the row's own length.  Source: same page, "Question" (the
  proposed opt-in mode).
* ``plan.plan_balanced`` -- batch-wide quota + greedy packing.  Source: same
  page, "Where it comes from" (``payload = ceil_div(total_num_blocks,
  num_sm_parts) + fixed_overhead_num_blocks`` and the greedy packing loop).
* ``fp8`` -- exact fp64 decode of an FP8 E4M3 key/value cache with one
  scale per cache (the reading of the pages' low-precision checkpoints,
  stated in the module).
* ``nvfp4`` -- exact fp64 decode of an NVFP4 weight matrix (E2M1 codes, one
  E4M3 scale per 16 weights, one fp32 scale per matrix) and the product
  ``bf16(x) @ W^T`` that both kernel shapes of a weight matmul agree on.
  Source: "Greedy outputs depend on batch composition" (gllm issue #98),
  Candidate cause and Next steps.
* ``bf16`` -- exact fp64 -> bf16 round-to-nearest-even, used to state the
  output rounding and the tolerance in units of bf16 ULP (same page,
  Measurement: "1-2 ULP of bf16 near 1.0").

Parity pins (``tests/test_oracle_*.py``) tie every function to closed forms,
brute force and invariants; no function here is "parity unpinned".
"""

from . import attention, plan, bf16, fp8, nvfp4  # noqa: F401
