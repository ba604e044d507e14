"""Seeded synthetic workloads for the attention backward pass.

This module only draws random numbers and describes shapes.  It holds none of
the backward pass's arithmetic: O and LSE (which depend on the forward pass)
are produced elsewhere.  Both the parity tests (which feed the fp64 oracle)
and the benchmark draw their inputs from here, so both sides always see the
same arrays for the same seed.

The five workloads mirror the problem shapes of the three source pages
("flash_attention_backward_dq.metal": [B,H,S,D] MHA with causal masking;
"flash_attention_v2_backward.wgsl": [B,S,H,D] with GQA, causal offset,
sliding window, additive mask and dropout; "attention_backward_dq.wgsl":
single-query decode with given probabilities).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

LAYOUT_BHSD = 0  # page 1: Q,O,dO,dQ [B,H,Sq,D]; K,V [B,Hkv,Sk,D]
LAYOUT_BSHD = 1  # page 2: Q,O,dO,dQ [B,Sq,H,D]; K,V [B,Sk,Hkv,D]
DTYPE_F32 = 0
DTYPE_BF16 = 1
MASKED = -1.0e30  # hard-mask sentinel of page 2 (FAB_MASKED)


@dataclasses.dataclass
class AttnProblem:
    """Shape and masking rules of one backward-pass problem."""

    batch: int
    num_heads: int
    num_kv_heads: int
    seq_q: int
    seq_k: int
    head_dim: int
    scale: float
    causal: int = 0
    causal_offset: int = 0
    window: int = 0
    dropout_prob: float = 0.0
    seed: int = 0
    has_mask: int = 0
    # mask element strides for [B,1,Sq,Sk] broadcast over heads
    mask_stride_b: int = 0
    mask_stride_h: int = 0
    mask_stride_q: int = 0
    mask_stride_k: int = 0
    layout: int = LAYOUT_BHSD
    dtype: int = DTYPE_F32
    deterministic: int = 0

    def q_shape(self):
        if self.layout == LAYOUT_BHSD:
            return (self.batch, self.num_heads, self.seq_q, self.head_dim)
        return (self.batch, self.seq_q, self.num_heads, self.head_dim)

    def kv_shape(self):
        if self.layout == LAYOUT_BHSD:
            return (self.batch, self.num_kv_heads, self.seq_k, self.head_dim)
        return (self.batch, self.seq_k, self.num_kv_heads, self.head_dim)

    def lse_shape(self):
        return (self.batch, self.num_heads, self.seq_q)

    def mask_shape(self):
        return (self.batch, 1, self.seq_q, self.seq_k)


@dataclasses.dataclass
class DecodeProblem:
    """Batched single-query decode backward (page 3 layout, plus a sequence axis)."""

    num_seqs: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    history_len: int


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    # keep NaN/inf payloads as they are (none are generated here)
    return r.astype(np.uint32).view(np.float32)


def round_io(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round an array once to the problem's I/O dtype (values kept in float32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == DTYPE_BF16:
        return _to_bf16_values(x)
    return x


def make_inputs(p: AttnProblem, seed: int, q_std=1.0, kv_std=1.0, do_std=0.1,
                mask_frac: float = 0.1):
    """Draw Q, K, V, dO (and the additive mask) for problem ``p``.

    Q, K, V ~ N(0, q_std^2 / kv_std^2), dO ~ N(0, do_std^2), rounded to the
    I/O dtype.  The mask, when present, has shape [B,1,Sq,Sk] with entries
    -1e30 with probability ``mask_frac`` and 0 otherwise.
    """
    g = _rng(seed)
    Q = round_io(g.standard_normal(p.q_shape(), dtype=np.float32) * q_std, p.dtype)
    K = round_io(g.standard_normal(p.kv_shape(), dtype=np.float32) * kv_std, p.dtype)
    V = round_io(g.standard_normal(p.kv_shape(), dtype=np.float32) * kv_std, p.dtype)
    dO = round_io(g.standard_normal(p.q_shape(), dtype=np.float32) * do_std, p.dtype)
    mask = None
    if p.has_mask:
        u = g.random(p.mask_shape(), dtype=np.float32)
        mask = np.where(u < mask_frac, np.float32(MASKED), np.float32(0.0)).astype(np.float32)
    return Q, K, V, dO, mask


def make_decode_inputs(p: DecodeProblem, seed: int):
    """k_hist, v_hist [N,history,n_kv,D], d_out [N,n_heads,D] ~ N(0,1);
    logits [N,n_heads,history] ~ N(0,1) (probabilities are the softmax of
    these logits, formed by the caller)."""
    g = _rng(seed)
    k = g.standard_normal((p.num_seqs, p.history_len, p.n_kv_heads, p.head_dim), dtype=np.float32)
    v = g.standard_normal((p.num_seqs, p.history_len, p.n_kv_heads, p.head_dim), dtype=np.float32)
    d_out = g.standard_normal((p.num_seqs, p.n_heads, p.head_dim), dtype=np.float32)
    logits = g.standard_normal((p.num_seqs, p.n_heads, p.history_len), dtype=np.float32)
    return k, v, d_out, logits


def make_decode_queries(p: DecodeProblem, seed: int):
    """q [N,n_heads,D] ~ N(0,1) for the decode pass 2 (its own stream: the
    pass-1 inputs of the same seed are unchanged)."""
    g = _rng(seed + 0x51)
    return g.standard_normal((p.num_seqs, p.n_heads, p.head_dim), dtype=np.float32)


# --------------------------------------------------------------------------
# The five workloads (shapes, masking rules, value distributions).
# --------------------------------------------------------------------------

def tiny() -> AttnProblem:
    """B=1, H=Hkv=2, S=64, D=64, fp32, non-causal, no mask/dropout."""
    return AttnProblem(1, 2, 2, 64, 64, 64, scale=1.0 / 8.0)


def causal_mha() -> AttnProblem:
    """B=4, H=Hkv=16, S=1024, D=64, fp32 [B,H,S,D], causal."""
    return AttnProblem(4, 16, 16, 1024, 1024, 64, scale=1.0 / 8.0, causal=1)


def gqa_window(dtype: int = DTYPE_F32) -> AttnProblem:
    """B=2, Hq=32, Hkv=8, S=4096, D=128, [B,S,H,D], causal, window 1024."""
    return AttnProblem(2, 32, 8, 4096, 4096, 128, scale=1.0 / math.sqrt(128.0), causal=1,
                       window=1024, layout=LAYOUT_BSHD, dtype=dtype)


def masked_dropout() -> AttnProblem:
    """B=2, H=Hkv=16, Sq=512, Sk=2048, D=64, causal offset 1536, additive
    mask [B,1,Sq,Sk] (10% -1e30), dropout 0.1."""
    sq, sk = 512, 2048
    return AttnProblem(2, 16, 16, sq, sk, 64, scale=1.0 / 8.0, causal=1, causal_offset=1536,
                       dropout_prob=0.1, seed=0x5EED0004, has_mask=1,
                       mask_stride_b=sq * sk, mask_stride_h=0, mask_stride_q=sk, mask_stride_k=1)


def decode() -> DecodeProblem:
    """64 sequences, 8 query heads, 1 KV head, D=256, history 4096."""
    return DecodeProblem(64, 8, 1, 256, 4096)


WORKLOADS = {
    "tiny": (tiny, 0),
    "causal_mha": (causal_mha, 1),
    "gqa_window": (gqa_window, 2),
    "masked_dropout": (masked_dropout, 3),
}

