"""Float64 CPU oracle for the MLA forward_absorb decode step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls, links
or executes anything in this package; only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference arm may.  It shares no code with the
CUDA path: the two meet only in the seeded input generator
(``mla_decode_attention_08_gb300.inputs``), which holds none of the method's
arithmetic.

Modules
  fp8        e4m3fn decode / encode written from the format's definition.
  quant      per-tensor absmax FP8 quantisation of the bf16 latent cache.
  qsplit     the two-term e4m3 query and probability operands of the
             e4m3-cache step (per-token power-of-two scale, hi / lo split).
  mxfp4      MXFP4 (E2M1 elements, E8M0 scale per 32) codec, block
             quantiser and the decode step over an MXFP4 cache.
  attention  exact softmax attention over the dequantised e4m3 cache or the
             bf16 cache (float64), and the split-KV partial / log-sum-exp
             combine restated.
  schedule   the token-balanced split schedule restated with plain loops.

Every function names the page passage it follows.  The pages are the three
kernelbot-amd-mixed-mla leaderboard submissions (663509 "v_ae",
722089 "v60", 738050); where they are silent the reading taken is stated.
"""
