"""The row log-sum-exp sweep on the tensor cores (attn_bwd_lse) against the
fp64 oracle, row by row, and the backward pass without a saved LSE.

Bar for the LSE: every row within the bound parity_helpers.lse_bound derives
from the arithmetic (input rounding to TF32, fp32 accumulation, fp32
reduction); rows without a visible non-hard key are exactly 3e38 on both
sides.  Bar for the gradients with the LSE recomputed: the backward's own
(max|err|/max|ref| <= 2e-3 fp32, <= 2e-2 bf16).
"""
import copy

import numpy as np
import pytest

from attention_backward_pass_gb300 import workloads as W
from oracle import attention as OA

from parity_helpers import TOL, compare, lse_bound, make_case, run_lse_gpu

pytestmark = pytest.mark.gpu


def P(**kw):
    base = dict(batch=1, num_heads=2, num_kv_heads=2, seq_q=64, seq_k=64, head_dim=64,
                scale=0.125)
    base.update(kw)
    p = W.AttnProblem(**base)
    if p.has_mask:
        p.mask_stride_b, p.mask_stride_h = p.seq_q * p.seq_k, 0
        p.mask_stride_q, p.mask_stride_k = p.seq_k, 1
    return p


CASES = {
    "tiny": W.tiny(),
    "causal_ragged_d64": P(seq_q=300, seq_k=300, causal=1),
    "noncausal_rect_d64": P(seq_q=200, seq_k=333),
    "gqa_window_bshd_d128": P(num_heads=4, num_kv_heads=2, seq_q=384, seq_k=384, head_dim=128,
                              causal=1, window=100, layout=W.LAYOUT_BSHD,
                              scale=1 / np.sqrt(128)),
    "window_only_offset": P(seq_q=150, seq_k=260, window=40, causal_offset=60),
    "long_keys_offset": P(seq_q=300, seq_k=1000, causal=1, causal_offset=700, head_dim=128,
                          scale=1 / np.sqrt(128)),
    "mask_vec_offset": P(seq_q=200, seq_k=520, causal=1, causal_offset=320, has_mask=1),
    "mask_unaligned_rows": P(seq_q=130, seq_k=333, window=50, has_mask=1, num_heads=3,
                             num_kv_heads=1),
    "negative_scale": P(seq_q=100, seq_k=170, scale=-0.2),
    "single_query_key": P(seq_q=1, seq_k=1),
    "empty_rows": P(seq_q=100, seq_k=90, window=5, causal_offset=80),
}


def _inputs(p, seed, real_mask=True):
    Q, K, V, dO, mask = W.make_inputs(p, seed)
    if mask is not None and real_mask:
        real = np.random.default_rng(seed + 7).standard_normal(mask.shape).astype(np.float32)
        mask = np.where(mask < -1.0e29, mask, real).astype(np.float32)
    return Q, K, mask


def _check(p, Q, K, mask, got, groups=None):
    ref = OA.lse(p, Q.astype(np.float64), K.astype(np.float64), mask, groups=groups)
    heads = None
    if groups is not None:
        G = p.num_heads // p.num_kv_heads
        heads = [(b, h) for b, g in groups for h in range(g * G, (g + 1) * G)]
    bound = lse_bound(p, Q, K, mask, ref)
    for b in range(p.batch):
        for h in range(p.num_heads):
            if heads is not None and (b, h) not in heads:
                continue
            r, g, bd = ref[b, h], got[b, h], bound[b, h]
            empty = r == OA.EMPTY_ROW_LSE
            assert np.all(g[empty] == np.float32(3.0e38)), (b, h)
            err = np.abs(g[~empty] - r[~empty])
            assert np.all(np.isfinite(g[~empty])), (b, h)
            assert np.all(err <= bd[~empty]), (b, h, float(err.max()),
                                               float(bd[~empty][err.argmax()]))


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("name", sorted(CASES))
def test_lse_parity(name, dtype):
    p = copy.copy(CASES[name])
    p.dtype = dtype
    Q, K, mask = _inputs(p, seed=2468)
    got = run_lse_gpu(p, Q, K, mask)
    _check(p, Q, K, mask, got)


FULL = {
    "causal_mha": (W.causal_mha, [(0, 0), (3, 15)]),
    "gqa_window_f32": (lambda: W.gqa_window(W.DTYPE_F32), [(1, 7)]),
    "gqa_window_bf16": (lambda: W.gqa_window(W.DTYPE_BF16), [(0, 2)]),
    "masked_dropout": (W.masked_dropout, [(1, 9)]),
}


@pytest.mark.parametrize("name", sorted(FULL))
def test_lse_full_size_sampled(name):
    make, groups = FULL[name]
    p = make()
    Q, K, mask = _inputs(p, seed=W.WORKLOADS.get(name, (None, 2))[1], real_mask=False)
    got = run_lse_gpu(p, Q, K, mask)
    _check(p, Q, K, mask, got, groups=groups)


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("name", ["causal_ragged_d64", "gqa_window_bshd_d128",
                                  "mask_vec_offset", "empty_rows"])
def test_backward_without_lse(name, dtype):
    p = copy.copy(CASES[name])
    p.dtype = dtype
    if name == "mask_vec_offset":
        p.dropout_prob, p.seed = 0.1, 0x5EED0009
    case = make_case(p, seed=1357)
    errs = compare(p, case, recompute_lse=True)
    assert all(e <= TOL[dtype] for e in errs.values()), errs


def test_backward_without_lse_full_size_sampled():
    p = W.causal_mha()
    groups = [(2, 5)]
    case = make_case(p, seed=W.WORKLOADS["causal_mha"][1], groups=groups)
    errs = compare(p, case, groups=groups, recompute_lse=True)
    assert all(e <= TOL[p.dtype] for e in errs.values()), errs
