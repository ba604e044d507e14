"""fp64 CPU oracle for the attention backward pass -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct statement of what the
backward pass computes.  It materialises S, P, dP and dS as full [Sq, Sk]
arrays per (batch, head) slice and uses numpy (fp64) matrix products as its
only library steps.  It shares no code with the CUDA library: neither imports
the other.

Only the tests, the smoke check of ``__graft_entry__`` and the CPU-baseline
leg of ``bench.py`` may import it.  The product path never calls it.

Sources (the three pages the method is taken from):
  * "rustytorch flash_attention_backward_dq.metal" -- dQ of a [B,H,S,D]
    causal MHA backward, Delta = rowsum(dO*O), P = exp(scale*q.k - LSE).
  * "ferrotensor-backend flash_attention_v2_backward.wgsl" -- two-pass
    backward with GQA, causal offset, sliding window, additive mask with a
    -1e30 hard sentinel, dropout multiplier M, dS = P*(M*(dO.V) - Delta).
  * "rullama attention_backward_dq.wgsl" -- single-query decode backward with
    given probabilities and unscaled scores.

Every function here is pinned by a test under tests/ against something other
than itself (finite differences, torch autograd, closed forms, invariants,
published known-answer vectors); the one exception is the dropout bit
pattern relative to the pages' own (unpublished) hash, which is "parity
unpinned" -- parity there is only against the Philox4x32-10 spec below.
"""
