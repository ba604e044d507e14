"""fp64 definition of the attention backward pass (oracle; test infrastructure only).

Each (batch, query head) slice is handled on its own, with S, P, dP and dS
materialised as full [Sq, Sk] fp64 arrays.  The only library step is the
numpy matrix product.  Nothing is blocked, fused or reordered.

Notation follows the WGSL two-pass backward page
("flash_attention_v2_backward.wgsl"):
  s_ij   = scale * q_i . k_j + mask_ij
  P_ij   = exp(s_ij - LSE_i)          (0 for invisible or hard-masked pairs)
  M_ij   = dropout multiplier          (header comment; dropout_scale)
  Delta_i = dO_i . O_i                 (flash_bwd_dq, "delta4")
  dS_ij  = P_ij * (M_ij * (dO_i . V_j) - Delta_i)   (header comment)
  dQ_i   = scale * sum_j dS_ij K_j     (flash_bwd_dq, sweep 2)
  dK_j   = scale * sum_i dS_ij Q_i     summed over the query heads that share
  dV_j   = sum_i P_ij M_ij dO_i        the KV head (flash_bwd_dk_dv, loop g)
The Metal page ("flash_attention_backward_dq.metal") is the special case
without mask, window, dropout or GQA, in [B,H,S,D] layout, with the scale
applied to dQ at the end; the result is the same up to rounding.
"""
from __future__ import annotations

import numpy as np

from . import philox

MASKED = -1.0e30          # hard sentinel of page 2 (FAB_MASKED)
EMPTY_ROW_LSE = 3.0e38    # LSE of a row with no probability mass (flash_bwd_dq)
LAYOUT_BHSD = 0
LAYOUT_BSHD = 1


# --------------------------------------------------------------------------
# Masking rules
# --------------------------------------------------------------------------

def visible(seq_q: int, seq_k: int, causal: int, causal_offset: int, window: int) -> np.ndarray:
    """Visibility of key kj to query qi, page 2 ``fab2_visible``.

    qa = qi + causal_offset; a pair is visible iff (not causal or kj <= qa)
    and (window == 0 or |qa - kj| < window).  (Indices beyond seq_q / seq_k
    do not exist in the [Sq, Sk] array.)
    """
    qi = np.arange(seq_q, dtype=np.int64)[:, None]
    kj = np.arange(seq_k, dtype=np.int64)[None, :]
    qa = qi + int(causal_offset)
    vis = np.ones((seq_q, seq_k), dtype=bool)
    if causal:
        vis &= kj <= qa
    if window > 0:
        vis &= np.abs(qa - kj) < int(window)
    return vis


def mask_slice(p, mask_flat: np.ndarray, b: int, h: int) -> np.ndarray:
    """Additive mask of one (b, h) slice, page 2 ``fab2_mask_at``:
    mask[b*sb + h*sh + qi*sq + kj*sk] (element strides; sh = 0 broadcasts)."""
    qi = np.arange(p.seq_q, dtype=np.int64)[:, None]
    kj = np.arange(p.seq_k, dtype=np.int64)[None, :]
    idx = (b * p.mask_stride_b + h * p.mask_stride_h
           + qi * p.mask_stride_q + kj * p.mask_stride_k)
    return np.asarray(mask_flat, dtype=np.float64).reshape(-1)[idx]


def hard_and_bias(p, mask, b: int, h: int):
    """(hard, bias): hard marks pairs that carry no probability (invisible, or
    the additive mask is at or below the -1e30 sentinel); bias is the additive
    mask (0 without one).  Reading: the page tests s <= -1e30 after adding the
    mask in fp32, which for |scale*q.k| far below 1e22 is the same as testing
    the mask value itself; the oracle tests the mask value."""
    vis = visible(p.seq_q, p.seq_k, p.causal, p.causal_offset, p.window)
    if p.has_mask:
        bias = mask_slice(p, mask, b, h)
        hard = ~vis | (bias <= MASKED)
        bias = np.where(hard, 0.0, bias)
    else:
        bias = np.zeros((p.seq_q, p.seq_k))
        hard = ~vis
    return hard, bias


def multiplier(p, b: int, h: int) -> np.ndarray:
    """Dropout multiplier M for slice (b, h); bh = b * num_heads + h."""
    return philox.dropout_multiplier(p.seed, b * p.num_heads + h, p.seq_q, p.seq_k,
                                     p.dropout_prob)


# --------------------------------------------------------------------------
# Layout helpers
# --------------------------------------------------------------------------

def _q_slice(p, X, b, h):
    X = np.asarray(X)
    return X[b, h] if p.layout == LAYOUT_BHSD else X[b, :, h]


def _kv_slice(p, X, b, kvh):
    X = np.asarray(X)
    return X[b, kvh] if p.layout == LAYOUT_BHSD else X[b, :, kvh]


def _set_q(p, X, b, h, val):
    if p.layout == LAYOUT_BHSD:
        X[b, h] = val
    else:
        X[b, :, h] = val


def _add_kv(p, X, b, kvh, val):
    if p.layout == LAYOUT_BHSD:
        X[b, kvh] += val
    else:
        X[b, :, kvh] += val


def kv_head(p, h: int) -> int:
    """GQA mapping of page 2: kvh = h / (num_heads / num_kv_heads)."""
    return h // (p.num_heads // p.num_kv_heads)


def _groups(p, groups):
    if groups is None:
        return [(b, g) for b in range(p.batch) for g in range(p.num_kv_heads)]
    return list(groups)


# --------------------------------------------------------------------------
# Scores, Delta, forward (input synthesis) and backward
# --------------------------------------------------------------------------

def scores(p, Q, K, mask, b, h):
    """s = scale * Q_h K_kvh^T + mask, fp64 [Sq, Sk]; also returns hard."""
    q = _q_slice(p, Q, b, h).astype(np.float64)
    k = _kv_slice(p, K, b, kv_head(p, h)).astype(np.float64)
    hard, bias = hard_and_bias(p, mask, b, h)
    s = float(p.scale) * (q @ k.T) + bias
    return s, hard


def delta(dO_rows: np.ndarray, O_rows: np.ndarray) -> np.ndarray:
    """Delta_i = sum_d dO_id * O_id (the Metal page's "D = rowsum(dO * O)")."""
    return np.sum(np.asarray(dO_rows, np.float64) * np.asarray(O_rows, np.float64), axis=-1)


def row_lse(s: np.ndarray, hard: np.ndarray) -> np.ndarray:
    """LSE_i = log sum over non-hard j of exp(s_ij), shifted by the row
    maximum; 3e38 for a row with no non-hard key (page 2, flash_bwd_dq sweep 1:
    lse = m + log l, "fully masked row")."""
    sm = np.where(hard, -np.inf, s)
    m = np.max(sm, axis=1, initial=-np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.where(hard, 0.0, np.exp(np.where(hard, 0.0, s - m_safe[:, None])))
    l = e.sum(axis=1)
    return np.where(empty, EMPTY_ROW_LSE, m_safe + np.log(np.where(empty, 1.0, l)))


def lse(p, Q, K, mask=None, groups=None):
    """Row log-sum-exp of the scores for callers without a saved LSE (page 2,
    flash_bwd_dq sweep 1), fp64 [B, H, Sq]; only the requested (b, kv-head)
    groups are filled (all by default).  Dropout does not enter."""
    LSE = np.zeros(p.lse_shape(), dtype=np.float64)
    G = p.num_heads // p.num_kv_heads
    for b, kvh in _groups(p, groups):
        for h in range(kvh * G, (kvh + 1) * G):
            s, hard = scores(p, Q, K, mask, b, h)
            LSE[b, h] = row_lse(s, hard)
    return LSE


def forward(p, Q, K, V, mask=None, groups=None):
    """O and LSE consistent with the backward's conventions (used only to
    synthesise backward inputs).  LSE_i = log sum over non-hard j of
    exp(s_ij) (max-shifted); a row with no non-hard key gets LSE = 3e38 and
    O = 0 (flash_bwd_dq, "fully masked row").  O_i = sum_j P_ij M_ij V_j.
    Returns (O, LSE) as fp64 arrays in the problem's layout, with only the
    requested (b, kv-head) groups filled (all by default)."""
    O = np.zeros(p.q_shape(), dtype=np.float64)
    LSE = np.zeros(p.lse_shape(), dtype=np.float64)
    G = p.num_heads // p.num_kv_heads
    for b, kvh in _groups(p, groups):
        v = _kv_slice(p, V, b, kvh).astype(np.float64)
        for h in range(kvh * G, (kvh + 1) * G):
            s, hard = scores(p, Q, K, mask, b, h)
            lse_row = row_lse(s, hard)
            empty = lse_row == EMPTY_ROW_LSE
            P = np.where(hard, 0.0, np.exp(np.where(hard, 0.0, s - lse_row[:, None])))
            P[empty] = 0.0
            Mdrop = multiplier(p, b, h)
            _set_q(p, O, b, h, (P * Mdrop) @ v)
            LSE[b, h] = lse_row
    return O, LSE


def backward(p, Q, K, V, O, dO, LSE, mask=None, groups=None, return_parts=False):
    """dQ, dK, dV of the attention backward pass, by definition, in fp64.

    For each (b, query head h) with kvh = h / (H / Hkv):
      P   = exp(s - LSE) on non-hard pairs, 0 elsewhere
      dP' = M * (dO V^T);  dS = P * (dP' - Delta);  Delta = rowsum(dO * O)
      dQ  = scale * dS K;  dK[kvh] += scale * dS^T Q;  dV[kvh] += (P M)^T dO
    dQ/dK/dV are returned in the problem's layout; only the requested
    (b, kv-head) groups are computed (all by default).  With
    ``return_parts`` the per-slice P, dS and Delta are also returned as a
    dict keyed by (b, h).
    """
    dQ = np.zeros(p.q_shape(), dtype=np.float64)
    dK = np.zeros(p.kv_shape(), dtype=np.float64)
    dV = np.zeros(p.kv_shape(), dtype=np.float64)
    parts = {}
    G = p.num_heads // p.num_kv_heads
    LSE = np.asarray(LSE, dtype=np.float64)
    for b, kvh in _groups(p, groups):
        k = _kv_slice(p, K, b, kvh).astype(np.float64)
        v = _kv_slice(p, V, b, kvh).astype(np.float64)
        for h in range(kvh * G, (kvh + 1) * G):
            q = _q_slice(p, Q, b, h).astype(np.float64)
            o = _q_slice(p, O, b, h).astype(np.float64)
            do = _q_slice(p, dO, b, h).astype(np.float64)
            s, hard = scores(p, Q, K, mask, b, h)
            lse = LSE[b, h]
            # P = 0 on hard pairs whatever LSE holds (an empty row's LSE never
            # enters exp on a non-hard pair because there is none)
            P = np.where(hard, 0.0, np.exp(np.where(hard, 0.0, s - lse[:, None])))
            Mdrop = multiplier(p, b, h)
            D = delta(do, o)
            dPp = Mdrop * (do @ v.T)
            dS = P * (dPp - D[:, None])
            _set_q(p, dQ, b, h, float(p.scale) * (dS @ k))
            _add_kv(p, dK, b, kvh, float(p.scale) * (dS.T @ q))
            _add_kv(p, dV, b, kvh, (P * Mdrop).T @ do)
            if return_parts:
                parts[(b, h)] = {"P": P, "dS": dS, "Delta": D, "M": Mdrop}
    if return_parts:
        return dQ, dK, dV, parts
    return dQ, dK, dV


def loss(p, Q, K, V, dO, mask=None):
    """L = sum(dO * O(Q, K, V)) with mask and dropout pattern held fixed; its
    gradient with respect to Q, K, V is (dQ, dK, dV) when O and LSE come from
    the same forward.  Used by the finite-difference pin."""
    O, _ = forward(p, Q, K, V, mask)
    return float(np.sum(np.asarray(dO, np.float64) * O))
