"""Fused forward (attn_fwd) against the fp64 oracle forward: O within the
backward's bars (max|err|/max|ref|: 2e-3 fp32 with TF32 products, 2e-2 bf16),
LSE row by row within parity_helpers.lse_bound, empty rows 3e38 / O = 0."""
import copy

import numpy as np
import pytest

from attention_backward_pass_gb300 import workloads as W
from oracle import attention as OA

from parity_helpers import TOL, lse_bound, rel_err, run_fwd_gpu

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
    "mask_dropout_offset": P(seq_q=200, seq_k=520, causal=1, causal_offset=320, has_mask=1,
                             dropout_prob=0.1, seed=0x5EED0004),
    "single_query_key": P(seq_q=1, seq_k=1),
    "empty_rows": P(seq_q=100, seq_k=90, window=5, causal_offset=80),
    "long_keys": P(seq_q=130, seq_k=1500, causal=1, causal_offset=1400, head_dim=128,
                   scale=1 / np.sqrt(128)),
}


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("name", sorted(CASES))
def test_forward_parity(name, dtype):
    p = copy.copy(CASES[name])
    p.dtype = dtype
    Q, K, V, _, mask = W.make_inputs(p, 4242)
    O, LSE = run_fwd_gpu(p, Q, K, V, mask)
    f = lambda a: a.astype(np.float64)  # noqa: E731
    O_ref, LSE_ref = OA.forward(p, f(Q), f(K), f(V), mask)
    assert np.all(np.isfinite(O))
    assert rel_err(O, O_ref) <= TOL[dtype], rel_err(O, O_ref)
    empty = LSE_ref == OA.EMPTY_ROW_LSE
    assert np.all(LSE[empty] == np.float32(3.0e38))
    bound = lse_bound(p, Q, K, mask, LSE_ref)
    assert np.all(np.abs(LSE[~empty] - LSE_ref[~empty]) <= bound[~empty])


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_forward_everything_per_head_mask(head_dim, dtype):
    """GQA, causal with an offset, a sliding window, dropout and a different
    real-valued mask per (batch, query head) stored transposed, on ragged
    query and key tails."""
    from parity_helpers import strided_mask
    p = P(batch=2, num_heads=6, num_kv_heads=2, seq_q=211, seq_k=345, head_dim=head_dim,
          scale=1 / np.sqrt(head_dim), causal=1, causal_offset=134, window=150,
          dropout_prob=0.2, seed=0x5EED000C, layout=W.LAYOUT_BSHD)
    p.dtype = dtype
    Q, K, V, _, _ = W.make_inputs(p, 808)
    mask, _ = strided_mask(p, "per_head_transposed", 809)
    mask = mask.astype(np.float32)
    O, LSE = run_fwd_gpu(p, Q, K, V, mask)
    f = lambda a: a.astype(np.float64)  # noqa: E731
    O_ref, LSE_ref = OA.forward(p, f(Q), f(K), f(V), mask)
    assert np.all(np.isfinite(O))
    assert rel_err(O, O_ref) <= TOL[dtype], rel_err(O, O_ref)
    empty = LSE_ref == OA.EMPTY_ROW_LSE
    assert np.all(LSE[empty] == np.float32(3.0e38))
    bound = lse_bound(p, Q, K, mask, LSE_ref)
    assert np.all(np.abs(LSE[~empty] - LSE_ref[~empty]) <= bound[~empty])


def _tf32_values(x):
    """Round float32 values to TF32-representable ones (10-bit mantissa,
    nearest), so that the kernel's TF32 operand rounding is exact."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_forward_lazy_rescale(head_dim, dtype):
    """Queries with standard deviation 4 make a row's running maximum grow by
    more than 2^8 from one key tile to a later one, so the O accumulator is
    rescaled in tensor memory, in tiles where only some rows of a warp need
    it.  fp32 inputs are TF32-representable, so the error stays that of the
    fp32 sums and the approximate exponentials."""
    p = P(num_heads=4, num_kv_heads=2, seq_q=300, seq_k=700, head_dim=head_dim,
          scale=1 / np.sqrt(head_dim), causal=1, causal_offset=400)
    p.dtype = dtype
    Q, K, V, _, _ = W.make_inputs(p, 909, q_std=4.0)
    if dtype == W.DTYPE_F32:
        Q, K, V = _tf32_values(Q), _tf32_values(K), _tf32_values(V)
    O, LSE = run_fwd_gpu(p, Q, K, V, None)
    f = lambda a: a.astype(np.float64)  # noqa: E731
    O_ref, LSE_ref = OA.forward(p, f(Q), f(K), f(V), None)
    assert np.all(np.isfinite(O))
    assert rel_err(O, O_ref) <= TOL[dtype], rel_err(O, O_ref)
    bound = lse_bound(p, Q, K, None, LSE_ref)
    assert np.all(np.abs(LSE - LSE_ref) <= bound)
