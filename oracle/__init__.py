"""CPU oracle for block speculative decoding with target-context injection.

THIS PACKAGE IS TEST INFRASTRUCTURE, NOT THE PRODUCT.  Only the test suite,
the smoke check and the CPU-baseline leg of the benchmark may import it.  The
product path (the CUDA library and its Python binding) never calls into it and
shares no code with it: no kernels, no helpers, no tables, no constants.

What it computes, and where each step comes from:

* ``philox``    Philox-4x32-10 counter-based generator (Salmon, Moraes, Dror,
                Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11).
                The pages name no generator; this one supplies the uniforms
                that the accept/resample rule consumes.
* ``fixedpoint`` exact integer inverse-CDF sampling used by every draw.
* ``sampling``  temperature / top-p preparation of a distribution and the
                drafter's own draw y ~ q.
* ``verify``    greedy prefix match and lossless rejection sampling
                ("DFlash vs DFlash 2" blog, section "The problem: one expensive
                token at a time": accept with min(1, p/q), resample from the
                normalised [p - q]+, bonus token when every draft survives).
* ``quant``     FP8 (E4M3) drafter weights with one float32 scale per output
                row, and their exact dequantization (product doc "Speculative
                decoding", introduction, and model card section "Serve": the
                models are served in FP8; format and scaling are readings).
* ``model``     the drafter: target-feature fusion H_t = RMSNorm(W_c[...]),
                context K/V injection, the non-causal block pass over
                [anchor, MASK, ...] with a sliding-window context, the shared
                LM head, per-position top-k and log-sum-exp ("DFlash vs
                DFlash 2", sections "DFlash: generate the block all at once" and
                "Conditioning on the target model"; model card
                "Beam-1.0-501B-A23B-DFlash2", section "Model").

Floating point is accumulated in float64 throughout.  Integer decisions
(argmax, accept, inverse-CDF index) are taken exactly as the function
docstrings state so that a second implementation can match them bit for bit.

Parity unpinned (conventions the pages do not fix; parity with the oracle is
parity with these readings): RoPE placement and base, the pre-norm layer
layout, the RMSNorm epsilon, the MASK token id, and the Philox counter layout.
"""

from . import philox, fixedpoint, sampling, verify, model, quant  # noqa: F401
