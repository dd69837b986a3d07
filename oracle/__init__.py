"""CPU oracle for the grouped-contiguous FP8 x MXFP4 MoE expert GEMM and its routing plan.

TEST INFRASTRUCTURE ONLY. This package is the slow, plain, obviously-correct
statement of what the GPU path computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  The product path (the CUDA library and
its Python binding) never imports, links or calls anything here, and nothing
here imports the product path.  The two share no code: the seeded input
generator in ``synth/`` feeds both sides and holds none of the method's
arithmetic.

Sources (web pages on the subject, cited by title and section):

* humming PR #129, "perf(sm90): size grouped W4A8 tiles per expert" -- the
  benchmark command names the operand formats: ``--a_dtype float8e4m3``,
  ``--b_dtype float4e2m1``, ``--c_dtype bfloat16``, ``--bs_dtype float8e8m0``,
  ``--input_scale_group_size 128``, ``--weight_scale_group_size 32``,
  ``--gemm_type grouped_contiguous``; its first section describes rows routed
  to each expert as contiguous ranges.
* MoonEP PR #38, "fit planning block size to device SMEM limit" -- the
  routing-plan kernel (per-expert histogram, per-warp scratch, column
  placement) and its check against an independent reference plus planning
  invariants.

Modules:

* ``formats``  -- decode tables for E2M1, E4M3, E8M0 written from the format
  definitions, and float64 -> bfloat16 round-to-nearest-even.
* ``plan``     -- histogram, exclusive scan, stable permutation.
* ``gemm``     -- per-expert float64 dequantise + matmul, BF16 rounding once;
  and a sampled variant computing chosen output elements one by one.

Every function here is pinned by ``tests/test_oracle_*.py`` against facts
fixed independently of this code (exhaustive decode against closed forms and
library conversions, identity / one-hot / all-ones weights with closed-form
outputs, brute force on tiny shapes, plan invariants).  The GEMM's agreement
with the pages' own numbers is "parity unpinned": the pages print timings,
not output values.
"""
