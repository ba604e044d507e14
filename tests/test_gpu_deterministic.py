"""Deterministic dQ (attn_bwd_params.deterministic = 1): every key tile
stores its dQ contribution in its own workspace slice and a final kernel sums
the slices in key-tile order.  Checked against the fp64 oracle with the
backward's bars, and for bit-for-bit equality of dQ across repeated calls
(fresh workspace each time, filled with 0xFF bytes, so nothing unwritten can
be read back as data)."""
import copy

import numpy as np
import pytest

from attention_backward_pass_gb300 import workloads as W

from parity_helpers import TOL, compare, make_case, run_gpu

pytestmark = pytest.mark.gpu


def P(**kw):
    base = dict(batch=1, num_heads=2, num_kv_heads=2, seq_q=64, seq_k=64, head_dim=64,
                scale=0.125, deterministic=1)
    base.update(kw)
    p = W.AttnProblem(**base)
    if p.has_mask:
        p.mask_stride_b, p.mask_stride_h = p.seq_q * p.seq_k, 0
        p.mask_stride_q, p.mask_stride_k = p.seq_k, 1
    return p


CASES = {
    "causal_ragged_d64": P(seq_q=300, seq_k=300, causal=1),
    "noncausal_rect_d64": P(seq_q=200, seq_k=333),
    "gqa_window_bshd_d128": P(num_heads=4, num_kv_heads=2, seq_q=384, seq_k=384, head_dim=128,
                              causal=1, window=100, layout=W.LAYOUT_BSHD,
                              scale=1 / np.sqrt(128)),
    "mask_dropout_offset": P(seq_q=200, seq_k=520, causal=1, causal_offset=320, has_mask=1,
                             dropout_prob=0.1, seed=0x5EED0004),
    "empty_rows": P(seq_q=100, seq_k=90, window=5, causal_offset=80),
}


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("name", sorted(CASES))
def test_deterministic_parity_and_repeatability(name, dtype):
    p = copy.copy(CASES[name])
    p.dtype = dtype
    case = make_case(p, seed=97)
    errs = compare(p, case)
    assert all(e <= TOL[dtype] for e in errs.values()), errs
    first = run_gpu(p, case)
    for _ in range(2):
        again = run_gpu(p, case)
        for a, b in zip(first, again):
            assert np.array_equal(a, b)


def test_deterministic_full_size_sampled():
    p = W.causal_mha()
    p.deterministic = 1
    groups = [(1, 4)]
    case = make_case(p, seed=W.WORKLOADS["causal_mha"][1], groups=groups)
    errs = compare(p, case, groups=groups)
    assert all(e <= TOL[p.dtype] for e in errs.values()), errs
