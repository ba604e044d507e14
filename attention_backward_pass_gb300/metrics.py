"""Work counted by the throughput metric.

The metric credits the five dense contractions of the backward pass
(S = Q K^T, dP = dO V^T, dV = P^T dO, dK = dS^T Q, dQ = dS K): 2*D flops
each per visible (query, key) pair, i.e. 10*D flops per pair per query head.
Visibility follows the causal / causal-offset / sliding-window rule of the
WGSL two-pass backward page (``fab2_visible``); the additive mask and dropout
are not subtracted.  Recomputation is not credited.
"""
from __future__ import annotations


def visible_pairs(seq_q, seq_k, causal, causal_offset, window) -> int:
    """Number of (query, key) pairs of one head allowed by the causal/window
    rule, counted row by row as a key interval per query."""
    total = 0
    for i in range(seq_q):
        qa = i + causal_offset
        lo, hi = 0, seq_k  # [lo, hi)
        if causal:
            hi = min(hi, qa + 1)
        if window > 0:
            lo = max(lo, qa - window + 1)
            hi = min(hi, qa + window)
        if hi > lo:
            total += hi - lo
    return total


def counted_flops(p) -> float:
    """10 * D flops per visible pair per query head, over the whole batch."""
    pairs = visible_pairs(p.seq_q, p.seq_k, p.causal, p.causal_offset, p.window)
    return 10.0 * p.head_dim * pairs * p.batch * p.num_heads


def lse_flops(p) -> float:
    """2 * D flops per visible pair per query head (the score product of the
    LSE sweep), over the whole batch."""
    pairs = visible_pairs(p.seq_q, p.seq_k, p.causal, p.causal_offset, p.window)
    return 2.0 * p.head_dim * pairs * p.batch * p.num_heads


def decode_bytes(p) -> int:
    """Minimum HBM bytes of the decode backward: K and V history read once per
    sequence (shared by the query heads of a KV head), probs and d_out read,
    d_scores and d_q written; all fp32."""
    kv = 2 * p.num_seqs * p.history_len * p.n_kv_heads * p.head_dim
    probs = p.num_seqs * p.n_heads * p.history_len
    dout = p.num_seqs * p.n_heads * p.head_dim
    return 4 * (kv + 2 * probs + 2 * dout)


def decode_kv_bytes(p) -> int:
    """Minimum HBM bytes of the decode pass 2: d_k_hist and d_v_hist written,
    probs and d_scores read, q and d_out read; all fp32."""
    hist = 2 * p.num_seqs * p.history_len * p.n_kv_heads * p.head_dim
    rows = 2 * p.num_seqs * p.n_heads * p.history_len
    vecs = 2 * p.num_seqs * p.n_heads * p.head_dim
    return 4 * (hist + rows + vecs)


def decode_flops(p) -> float:
    """2 flops per multiply-add of d_probs = d_out.v and d_q = sum d_scores k,
    per query head: 4 * history * D per head."""
    return 4.0 * p.num_seqs * p.n_heads * p.history_len * p.head_dim
