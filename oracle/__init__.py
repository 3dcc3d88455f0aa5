"""fp64 CPU oracle for the Transformer-stack forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs use it.  It shares no code with the
CUDA path; the only module both sides use is ``synth`` (seeded random inputs).

The oracle is the plain definition of what the pages' method computes, in
float64, with no blocking, fusion or online softmax:

* Attention is the textbook five-step form -- scores Q K^T, scale by
  1/sqrt(d_k), mask, row softmax, times V -- from "TikTok TechJam 2026 --
  Problem 3: GPU Transformer Optimization", section 2.1 (Flash Attention),
  steps (1)-(5).  The flash form of the same section (running max m, running
  normaliser l, rescaled O) reaches the same result in exact arithmetic, so
  the oracle does not use it.
* Layer order follows the same page, section 1.A: a fused QKV projection
  reading the normed activations, attention, o_proj + residual + LayerNorm,
  FFN (GELU) + residual + LayerNorm of the next layer, and a tail of final
  LayerNorm + pad-mask + output cast.  The first LayerNorm has nothing to add
  to (the layer_norm_cast item), so the residual stream starts as x.  This is
  the pre-LN reading; ``norm_placement=1`` gives the post-LN reading.
* Masks: right-padded key mask mask[b, j] = (j < len_b) (section 2.1, "the
  mask trick"); causal allows j <= i.  Output rows at padded positions are
  zero (section 1.A, post_attn_chain_tail and final_layernorm).
* GELU is the exact erf form (section 2.3, the per-shape bias+GELU epilogue:
  the tanh form was only a candidate).
* The residual stream, LayerNorm statistics and softmax are exact here
  (float64); the pages keep them in fp32 on the GPU ("Transformerkernel",
  How we built it, first pass).

Readings where the pages are silent: LayerNorm eps = 1e-5 with the biased
variance (divide by D) inside the square root; a query with no allowed key
(only possible when len_b = 0) gets a zero attention output; padded output
rows are written as exact zeros.

Parity of each function is pinned in ``tests/test_oracle_pins.py`` against
library routines (torch float64 ``layer_norm``, ``gelu``,
``scaled_dot_product_attention`` and ``TransformerEncoder``), closed forms
and invariants.
"""
from .stack import (attention, attention_backward, attention_batched, attention_lse, forward,
                    forward_batched, gate, gelu, layer_norm, sequence_forward)

__all__ = ["attention", "attention_backward", "attention_batched", "attention_lse", "forward", "forward_batched",
           "gate", "gelu", "layer_norm", "sequence_forward"]
