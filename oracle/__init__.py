"""CPU oracle of the batch-1 decode step: plain, slow, fp64.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call, link
or execute this package: only the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs use it. It shares no code with the
CUDA path (no kernels, headers, helpers, tables or pre/post-processing);
both sides receive the same seeded inputs from ``synth``.

What it computes is the plain definition of one decode step of a
pre-norm transformer whose weights are their quantised values and whose KV
cache holds bfloat16, every product and sum taken in fp64:

* the step is matrix-vector work over all active weights plus the KV cache
  (Kog, "3k tokens/s per request", section "what limits decode speed on
  GPUs": batch-1 decode is matrix-vector dominated);
* the new token's key/value are written to the cache, then attention reads it
  (Muse Spark Open megakernel article, section "where the kernel boundary
  sits": attention of a layer reads KV history written by earlier steps);
* MoE layers route each token to 8 of 512 experts plus 1 shared expert
  (Ling-3.0-flash on DGX Spark, section "model and baseline configuration");
* the LM head may be the bf16 matrix or its dynamic FP8 quantisation
  (same article, section "optimisation 2: online FP8 LM head");
* a verify window of k tokens is checked in one pass and the correct prefix
  accepted (same article, section "optimisation 3: MTP speculative decoding");
* optionally the KV cache holds FP8 e4m3 codes with a scale per layer, K/V and
  kv head, 1.0 unless given (Kimi-K3 on 8xB300: fp8_e4m3 caches whose missing
  scaling factors fall back to 1.0).

Modules: ``formats`` (number formats and the FP8 / MXFP4 quantisers),
``ops`` (one function per operation), ``model`` (the whole step and verify).

Parity status: every function is pinned by the CPU tests to closed forms,
brute force, library conversions or invariants, except three conventions the
pages leave open and that no property can decide: the RoPE pairing
(rotate-half), the routing score (softmax over the selected experts) and the
RMSNorm gain distribution. Those three are "parity unpinned" by the pages.
"""
