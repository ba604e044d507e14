"""CUDA path vs the fp64 oracle, element by element, on seeded inputs.

Small problems span several tiles and a ragged tail and are compared in full;
the full-size workloads are compared on seeded (batch, kv-head) groups.
Bars: max|err|/max|ref| <= 2e-3 (fp32 I/O, TF32 products) and <= 2e-2
(bf16 I/O); dropout keep masks bit-exact.
"""
import numpy as np
import pytest

from attention_backward_pass_gb300 import workloads as W
from oracle import decode as OD
from oracle import philox

from parity_helpers import (TOL, compare, decode_case, make_case, rel_err, run_decode_gpu,
                            run_decode_kv_gpu, strided_mask)

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


SMALL = {
    "tiny": W.tiny(),
    "causal_ragged_d64": P(seq_q=300, seq_k=300, causal=1),
    "noncausal_rect_d64": P(seq_q=200, seq_k=333),
    "gqa_window_bshd_d128": P(num_heads=4, num_kv_heads=2, seq_q=384, seq_k=384, head_dim=128,
                              causal=1, window=100, layout=W.LAYOUT_BSHD,
                              scale=1 / np.sqrt(128)),
    "window_only_offset": P(seq_q=150, seq_k=260, window=40, causal_offset=60),
    "mask_dropout_offset": P(seq_q=200, seq_k=520, causal=1, causal_offset=320, has_mask=1,
                             dropout_prob=0.1, seed=0x5EED0004),
    "single_query_key": P(seq_q=1, seq_k=1),
    "empty_rows": P(seq_q=100, seq_k=90, window=5, causal_offset=80),
    # mask + dropout on the D = 128 tile configurations
    "mask_dropout_d128": P(seq_q=200, seq_k=333, head_dim=128, scale=1 / np.sqrt(128), causal=1,
                           causal_offset=133, has_mask=1, dropout_prob=0.15, seed=0x5EED0006),
    # GQA with mask + dropout, D = 64, [B,H,S,D]
    "gqa_mask_dropout_d64_bhsd": P(num_heads=4, num_kv_heads=2, seq_q=190, seq_k=300, causal=1,
                                   causal_offset=110, has_mask=1, dropout_prob=0.1,
                                   seed=0x5EED0007),
    "gqa_mask_dropout_d128_bshd": P(batch=2, num_heads=4, num_kv_heads=1, seq_q=150, seq_k=270,
                                    head_dim=128, scale=1 / np.sqrt(128), causal=1,
                                    causal_offset=120, has_mask=1, dropout_prob=0.2,
                                    seed=0x5EED0008, layout=W.LAYOUT_BSHD),
    # more work items (key tile, batch, KV head) than SMs, so CTAs walk several
    # items: D = 64 causal (192 items), GQA window D = 128 (176 items), items
    # without query tiles mixed in (448 of 576 see no query: their dK / dV are
    # zeros), mask + dropout across items (192 items)
    "many_items_d64": P(batch=8, num_heads=8, num_kv_heads=8, seq_q=380, seq_k=380, causal=1),
    "many_items_gqa_window_d128": P(batch=4, num_heads=8, num_kv_heads=4, seq_q=1300,
                                    seq_k=1300, head_dim=128, scale=1 / np.sqrt(128), causal=1,
                                    window=500, layout=W.LAYOUT_BSHD),
    "many_items_empty_keys": P(batch=4, num_heads=16, num_kv_heads=16, seq_q=200, seq_k=1100,
                               causal=1),
    "many_items_mask_dropout": P(batch=4, num_heads=8, num_kv_heads=8, seq_q=256, seq_k=700,
                                 causal=1, causal_offset=444, has_mask=1, dropout_prob=0.1,
                                 seed=0x5EED0009),
}


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_parity(name, dtype):
    import copy
    p = copy.copy(SMALL[name])
    p.dtype = dtype
    case = make_case(p, seed=1234)
    errs = compare(p, case)
    assert all(e <= TOL[dtype] for e in errs.values()), errs


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("kind", ["dense", "partial"])
def test_real_valued_mask(kind, dtype):
    """An additive mask with arbitrary finite values (N(0,1)) besides the
    hard-mask sentinel.  "partial" keeps real values only for the first 96
    queries, so that some query tiles of a key tile have only 0 / -1e30 entries
    and others do not."""
    from oracle import attention as OA
    p = P(seq_q=256, seq_k=300, causal=1, causal_offset=100, has_mask=1, dropout_prob=0.1,
          seed=0x5EED0005)
    p.dtype = dtype
    Q, K, V, dO, mask = W.make_inputs(p, 4321)
    real = np.random.default_rng(77).standard_normal(mask.shape).astype(np.float32)
    if kind == "partial":
        real[:, :, 96:, :] = 0.0
    mask = np.where(mask < -1.0e29, mask, real).astype(np.float32)
    O, LSE = OA.forward(p, Q, K, V, mask)
    case = dict(Q=Q, K=K, V=V, dO=dO, mask=mask, O=W.round_io(O.astype(np.float32), p.dtype),
                LSE=LSE.astype(np.float32))
    errs = compare(p, case)
    assert all(e <= TOL[dtype] for e in errs.values()), errs


def _strided_mask_case(p, kind, seed):
    """Seeded inputs with a per-(batch, query head) real-valued mask stored in
    the layout ``kind`` (see parity_helpers.strided_mask); O and LSE from the
    oracle forward."""
    from oracle import attention as OA
    Q, K, V, dO, _ = W.make_inputs(p, seed)
    store, _ = strided_mask(p, kind, seed + 1)
    store = store.astype(np.float32)
    O, LSE = OA.forward(p, Q, K, V, store)
    return dict(Q=Q, K=K, V=V, dO=dO, mask=store, O=W.round_io(O.astype(np.float32), p.dtype),
                LSE=LSE.astype(np.float32))


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("kind", ["per_head", "per_head_transposed", "head_major"])
def test_strided_per_head_mask(kind, head_dim, dtype):
    """A different mask for every (batch, query head) of a GQA problem, with
    contiguous, transposed and head-major storage (mask strides b/h/q/k of
    page 2's fab2_mask_at), plus dropout, on a ragged causal shape."""
    p = P(batch=2, num_heads=4, num_kv_heads=2, seq_q=150, seq_k=270, head_dim=head_dim,
          scale=1 / np.sqrt(head_dim), causal=1, causal_offset=120, dropout_prob=0.1,
          seed=0x5EED000A, layout=W.LAYOUT_BSHD)
    p.dtype = dtype
    case = _strided_mask_case(p, kind, seed=606)
    errs = compare(p, case)
    assert all(e <= TOL[dtype] for e in errs.values()), errs


@pytest.mark.parametrize("recompute_lse", [False, True], ids=["lse_given", "lse_recomputed"])
@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_everything_mix(head_dim, dtype, recompute_lse):
    """Every rule of page 2 at once: GQA (3 query heads per KV head), causal
    with an offset, a sliding window, a real-valued per-head additive mask
    with sentinels, dropout, [B,S,H,D], on a shape with ragged query and key
    tails."""
    p = P(batch=2, num_heads=6, num_kv_heads=2, seq_q=211, seq_k=345, head_dim=head_dim,
          scale=1 / np.sqrt(head_dim), causal=1, causal_offset=134, window=150,
          dropout_prob=0.2, seed=0x5EED000B, layout=W.LAYOUT_BSHD)
    p.dtype = dtype
    case = _strided_mask_case(p, "per_head", seed=707)
    errs = compare(p, case, recompute_lse=recompute_lse)
    assert all(e <= TOL[dtype] for e in errs.values()), errs


def test_keep_mask_bit_exact():
    import torch
    import attention_backward_pass_gb300 as ab
    p = W.masked_dropout()
    for b, h in [(0, 0), (1, 15), (0, 7)]:
        keep = torch.empty((p.seq_q, p.seq_k), dtype=torch.uint8, device="cuda")
        ab.dropout_keep_mask(p, b, h, keep)
        ref = philox.keep_mask(p.seed, b * p.num_heads + h, p.seq_q, p.seq_k, p.dropout_prob)
        assert np.array_equal(keep.cpu().numpy().astype(bool), ref)


def test_repeat_calls_overwrite():
    p = SMALL["causal_ragged_d64"]
    case = make_case(p, seed=5)
    errs = compare(p, case, repeat=3)
    assert all(e <= TOL[p.dtype] for e in errs.values()), errs


# ------------------------------------------------------------- full sizes

FULL = {
    "tiny": (W.tiny, None),
    "causal_mha": (W.causal_mha, [(0, 0), (3, 15), (2, 6)]),
    "gqa_window_f32": (lambda: W.gqa_window(W.DTYPE_F32), [(0, 0), (0, 5), (1, 7)]),
    "gqa_window_bf16": (lambda: W.gqa_window(W.DTYPE_BF16), [(0, 0), (1, 3), (1, 7)]),
    "masked_dropout": (W.masked_dropout, [(0, 0), (1, 9)]),
}


@pytest.mark.parametrize("name", sorted(FULL))
def test_full_size_sampled(name):
    make, groups = FULL[name]
    p = make()
    seed = W.WORKLOADS.get(name, (None, 2))[1]
    case = make_case(p, seed=seed, groups=groups)
    errs = compare(p, case, groups=groups)
    assert all(e <= TOL[p.dtype] for e in errs.values()), errs


# ------------------------------------------------------------- decode

DECODE = {
    "small_g8_d256": W.DecodeProblem(2, 8, 1, 256, 300),
    "g2_kv2_d64_ragged": W.DecodeProblem(3, 4, 2, 64, 17),
    "g1_d128": W.DecodeProblem(2, 4, 4, 128, 1000),
    "g16_d64": W.DecodeProblem(1, 16, 1, 64, 77),
    # many short sequences: CTAs cover several (sequence, KV head) pairs
    "many_seqs_g4_kv2_d128": W.DecodeProblem(300, 8, 2, 128, 100),
    "many_seqs_g2_kv4_d64_odd": W.DecodeProblem(260, 8, 4, 64, 37),
    # few long sequences: each pair is split over many CTAs
    "long_g8_d256": W.DecodeProblem(3, 8, 1, 256, 20000),
}


@pytest.mark.parametrize("name", sorted(DECODE))
def test_decode_parity(name):
    p = DECODE[name]
    case = decode_case(p, seed=7)
    ds, dq = run_decode_gpu(p, case)
    rds, rdq = OD.decode_backward(case["k"], case["v"], case["probs"], case["d_out"])
    assert rel_err(ds, rds) <= 2e-3 and rel_err(dq, rdq) <= 2e-3, (rel_err(ds, rds),
                                                                    rel_err(dq, rdq))


@pytest.mark.parametrize("name", sorted(DECODE))
def test_decode_kv_parity(name):
    """Pass 2 (history gradients) on pass 1's GPU d_scores, against the oracle
    of both passes in fp64."""
    p = DECODE[name]
    case = decode_case(p, seed=7)
    q = W.make_decode_queries(p, seed=7)
    ds, _ = run_decode_gpu(p, case)
    d_k, d_v = run_decode_kv_gpu(p, case, q, ds)
    rds, _ = OD.decode_backward(case["k"], case["v"], case["probs"], case["d_out"])
    rdk, rdv = OD.decode_backward_kv(q, case["probs"], case["d_out"], rds, p.n_kv_heads)
    assert np.all(np.isfinite(d_k)) and np.all(np.isfinite(d_v))
    assert rel_err(d_k, rdk) <= 2e-3 and rel_err(d_v, rdv) <= 2e-3, (rel_err(d_k, rdk),
                                                                    rel_err(d_v, rdv))


def test_decode_kv_full_size_sampled():
    p = W.decode()
    case = decode_case(p, seed=4)
    q = W.make_decode_queries(p, seed=4)
    ds, _ = run_decode_gpu(p, case)
    d_k, d_v = run_decode_kv_gpu(p, case, q, ds)
    seqs = [0, 31, 63]
    rds, _ = OD.decode_backward(case["k"], case["v"], case["probs"], case["d_out"], seqs=seqs)
    rdk, rdv = OD.decode_backward_kv(q, case["probs"], case["d_out"], rds, p.n_kv_heads, seqs=seqs)
    assert np.all(np.isfinite(d_k)) and np.all(np.isfinite(d_v))
    assert rel_err(d_k[seqs], rdk[seqs]) <= 2e-3 and rel_err(d_v[seqs], rdv[seqs]) <= 2e-3


def test_decode_full_size_sampled():
    p = W.decode()
    case = decode_case(p, seed=4)
    ds, dq = run_decode_gpu(p, case, repeat=2)
    seqs = [0, 31, 63]
    rds, rdq = OD.decode_backward(case["k"], case["v"], case["probs"], case["d_out"], seqs=seqs)
    assert rel_err(ds[seqs], rds[seqs]) <= 2e-3
    assert rel_err(dq[seqs], rdq[seqs]) <= 2e-3
