"""Oracle for the block text-diffusion denoising path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow CPU restatement of
what the GPU path computes, used to check it.  Only the test suite, the smoke
check and the benchmark's CPU-baseline leg may import it; the product path
(the C-ABI library and its Python binding) never does, and shares no code,
header, table or constant with it.

Sources (DiffusionGemma Technical Report and the accompanying blog post):
  * canvas of C tokens, uniform prior x_1 ~ Unif(V^C): report §2.1
    "Probability Paths and Denoising";
  * clean prefix in a read-only KV cache, bidirectional attention inside the
    256-token canvas, causal attention for context encoding: report §1,
    blog "Once Written, a Prefix Becomes History", report §4;
  * top-k mixture-of-experts FFN: report abstract and §6 "GPU time breakdown";
  * high-confidence positions lock in first, the rest keep being revised:
    blog "Once Written, a Prefix Becomes History";
  * adaptive stopping under a budget N: report §3.3 / Figure 5;
  * Eq. 7-10 efficiency metrics and the K-1 extra KV-append forwards:
    report §3.4.

Where the pages are silent (the sampler's exact commit rule, RoPE and RMSNorm
conventions, the reduction order that makes the sampler reproducible) the
modules state the reading they implement.

Modules
  philox   -- Philox4x32-10 counter-based generator (Salmon et al., SC'11)
  dgmath   -- the fp32 exp/log the sampler uses (Cody-Waite + series)
  weights  -- seeded synthetic weights (Irwin-Hall(4) over Philox words)
  model    -- fp64 forward passes: prefill, canvas denoise, commit
  sampler  -- canonical vocab-tile partials, tree merge, commit/re-noise/stop
  metrics  -- Eq. 7-10
  generate -- the canvas loop that ties them together
"""
