"""fp64 decode backward (oracle; test infrastructure only).

Follows the four numbered steps of the decode page
("rullama attention_backward_dq.wgsl", header comment), for one query per
head, given probabilities, unscaled scores, kv = h / heads_per_kv:
  1. d_probs_j  = d_out_h . v_hist[j, kv]
  2. sum_pd     = sum_j probs_hj d_probs_j
  3. d_scores_j = probs_hj (d_probs_j - sum_pd)
  4. d_q_h      = sum_j d_scores_j k_hist[j, kv]
Batched over an outer sequence axis: k_hist, v_hist [N, history, n_kv, D],
probs [N, n_heads, history], d_out [N, n_heads, D].  decode_backward_kv is
the history's gradients (the page's pass 2, plain reading).
"""
from __future__ import annotations

import numpy as np


def decode_backward(k_hist, v_hist, probs, d_out, seqs=None):
    """Returns (d_scores [N, n_heads, history], d_q [N, n_heads, D]) in fp64
    for the requested sequences (all by default; others stay zero)."""
    k_hist = np.asarray(k_hist)
    v_hist = np.asarray(v_hist)
    probs = np.asarray(probs)
    d_out = np.asarray(d_out)
    N, hist, n_kv, D = k_hist.shape
    n_heads = probs.shape[1]
    heads_per_kv = n_heads // n_kv
    d_scores = np.zeros((N, n_heads, hist), dtype=np.float64)
    d_q = np.zeros((N, n_heads, D), dtype=np.float64)
    for n in (range(N) if seqs is None else seqs):
        for h in range(n_heads):
            kv = h // heads_per_kv
            v = v_hist[n, :, kv, :].astype(np.float64)
            k = k_hist[n, :, kv, :].astype(np.float64)
            pr = probs[n, h].astype(np.float64)
            dp = v @ d_out[n, h].astype(np.float64)      # step 1
            sum_pd = float(pr @ dp)                      # step 2
            ds = pr * (dp - sum_pd)                      # step 3
            d_scores[n, h] = ds
            d_q[n, h] = ds @ k                           # step 4
    return d_scores, d_q


def decode_backward_kv(q, probs, d_out, d_scores, n_kv, seqs=None):
    """Pass 2 of the decode backward, the gradients of the history, in fp64.

    The decode page's pass 1 stages d_scores for a pass 2 that also takes q
    (the pass-2 file itself is not on the pages).  Plain reading, the
    gradients of the forward out_h = sum_j probs_hj v_j with unscaled scores
    score_hj = q_h . k_j, for KV head kv and its query heads h:
      d_k_hist[j, kv] = sum_h d_scores_hj q_h
      d_v_hist[j, kv] = sum_h probs_hj d_out_h
    q, d_out [N, n_heads, D]; probs, d_scores [N, n_heads, history].
    Returns (d_k_hist, d_v_hist) [N, history, n_kv, D] for the requested
    sequences (all by default; others stay zero)."""
    q = np.asarray(q)
    probs = np.asarray(probs)
    d_out = np.asarray(d_out)
    d_scores = np.asarray(d_scores)
    N, n_heads, hist = probs.shape
    D = q.shape[-1]
    heads_per_kv = n_heads // n_kv
    d_k = np.zeros((N, hist, n_kv, D), dtype=np.float64)
    d_v = np.zeros((N, hist, n_kv, D), dtype=np.float64)
    for n in (range(N) if seqs is None else seqs):
        for kv in range(n_kv):
            hs = range(kv * heads_per_kv, (kv + 1) * heads_per_kv)
            for h in hs:
                d_k[n, :, kv, :] += np.outer(d_scores[n, h].astype(np.float64),
                                             q[n, h].astype(np.float64))
                d_v[n, :, kv, :] += np.outer(probs[n, h].astype(np.float64),
                                             d_out[n, h].astype(np.float64))
    return d_k, d_v


def softmax_rows(logits) -> np.ndarray:
    """Row softmax in fp64 (forms the decode probabilities from logits)."""
    x = np.asarray(logits, dtype=np.float64)
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)
