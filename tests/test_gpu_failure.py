"""Failure detection on the GPU without a fault, and stray-write detection.

* A self-test kernel waits on an mbarrier that nothing arrives on: the bounded
  wait gives up after about a second, the device error word reads
  ATTN_ERR_TIMEOUT, clearing it works, and the context then runs a backward
  pass that matches the oracle.
* Every output of the backward (default and deterministic dQ), the LSE sweep,
  the fused forward and both decode passes is written into the middle of a
  larger buffer whose
  guard regions hold a sentinel bit pattern; the guards must be untouched and
  the outputs must match the oracle (the parity suites' shapes: ragged tiles,
  Sq = Sk = 1, GQA with a window, mask with dropout).
"""
import copy

import numpy as np
import pytest

from attention_backward_pass_gb300 import workloads as W
from oracle import attention as OA
from oracle import decode as OD

from parity_helpers import TOL, compare, decode_case, lse_bound, make_case, rel_err

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements on each side (a multiple of 256 bytes for every dtype)


def _guarded(shape, torch_dtype, device="cuda"):
    import torch
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * GUARD, dtype=torch_dtype, device=device)
    if buf.element_size() == 4:
        buf.view(torch.int32).fill_(0x7FC0DEAD)
    else:
        buf.view(torch.int16).fill_(0x7FDE)
    return buf, buf[GUARD:GUARD + n].view(shape)


def _guards_intact(buf):
    import torch
    raw = buf.view(torch.int32) if buf.element_size() == 4 else buf.view(torch.int16)
    want = 0x7FC0DEAD if buf.element_size() == 4 else 0x7FDE
    n = raw.numel()
    head, tail = raw[:GUARD], raw[n - GUARD:]
    return bool((head == want).all()) and bool((tail == want).all())


def test_bounded_wait_runs_out_and_context_survives():
    import torch
    import attention_backward_pass_gb300 as ab
    assert ab.check_device_error() == 0
    ab.selftest_wait_timeout()
    torch.cuda.synchronize()
    try:
        assert ab.check_device_error(clear=False) == ab.ATTN_ERR_TIMEOUT
    finally:
        ab.check_device_error(clear=True)
    assert ab.check_device_error() == 0
    p = W.AttnProblem(batch=1, num_heads=2, num_kv_heads=2, seq_q=300, seq_k=300, head_dim=64,
                      scale=0.125, causal=1)
    errs = compare(p, make_case(p, seed=3))
    assert all(e <= TOL[p.dtype] for e in errs.values()), errs


def P(**kw):
    base = dict(batch=1, num_heads=2, num_kv_heads=2, seq_q=64, seq_k=64, head_dim=64,
                scale=0.125)
    base.update(kw)
    p = W.AttnProblem(**base)
    if p.has_mask:
        p.mask_stride_b, p.mask_stride_h = p.seq_q * p.seq_k, 0
        p.mask_stride_q, p.mask_stride_k = p.seq_k, 1
    return p


# shapes of the parity suites (ragged tiles, Sq = Sk = 1, GQA + window + BSHD,
# mask + dropout + offset)
GUARD_CASES = {
    "causal_ragged_d64": (P(seq_q=300, seq_k=300, causal=1), (0, 1)),
    "single_query_key": (P(seq_q=1, seq_k=1), (0,)),
    "gqa_window_bshd_d128": (P(num_heads=4, num_kv_heads=2, seq_q=384, seq_k=384, head_dim=128,
                               causal=1, window=100, layout=W.LAYOUT_BSHD,
                               scale=1 / np.sqrt(128)), (0, 1)),
    "mask_dropout_offset": (P(seq_q=200, seq_k=520, causal=1, causal_offset=320, has_mask=1,
                              dropout_prob=0.1, seed=0x5EED0004), (0, 1)),
}
BWD_PARAMS = [(n, d) for n, (_, dets) in sorted(GUARD_CASES.items()) for d in dets]


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("name,det", BWD_PARAMS)
def test_backward_writes_stay_inside_outputs(name, det, dtype):
    import torch
    import attention_backward_pass_gb300 as ab
    p = copy.copy(GUARD_CASES[name][0])
    p.dtype, p.deterministic = dtype, det
    case = make_case(p, seed=77)
    tdt = torch.bfloat16 if dtype == W.DTYPE_BF16 else torch.float32
    to = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda().to(tdt)  # noqa: E731
    t = {k: to(case[k]) for k in ("Q", "K", "V", "O", "dO")}
    lse = torch.from_numpy(case["LSE"]).cuda()
    mask = torch.from_numpy(case["mask"]).cuda() if case["mask"] is not None else None
    bq, dQ = _guarded(p.q_shape(), tdt)
    bk, dK = _guarded(p.kv_shape(), tdt)
    bv, dV = _guarded(p.kv_shape(), tdt)
    ws = ab.alloc_workspace(p)
    ws.fill_(0xFF)
    ab.attn_bwd(p, t["Q"], t["K"], t["V"], t["O"], t["dO"], lse, mask, dQ, dK, dV, ws)
    torch.cuda.synchronize()
    assert ab.check_device_error() == 0
    assert _guards_intact(bq) and _guards_intact(bk) and _guards_intact(bv)
    f = lambda x: x.astype(np.float64)  # noqa: E731
    ref = OA.backward(p, f(case["Q"]), f(case["K"]), f(case["V"]), f(case["O"]), f(case["dO"]),
                      case["LSE"].astype(np.float64), case["mask"])
    for g, r in zip((dQ, dK, dV), ref):
        assert rel_err(g.float().cpu().numpy(), r) <= TOL[dtype]


LSE_CASES = {
    "causal_ragged_d64": P(seq_q=300, seq_k=300, causal=1),
    "single_query_key": P(seq_q=1, seq_k=1),
    "mask_unaligned_rows": P(seq_q=130, seq_k=333, window=50, has_mask=1, num_heads=3,
                             num_kv_heads=1),
}


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("name", sorted(LSE_CASES))
def test_lse_writes_stay_inside_output(name, dtype):
    import torch
    import attention_backward_pass_gb300 as ab
    p = copy.copy(LSE_CASES[name])
    p.dtype = dtype
    Q, K, _, _, mask = W.make_inputs(p, 78)
    tdt = torch.bfloat16 if dtype == W.DTYPE_BF16 else torch.float32
    q = torch.from_numpy(Q).cuda().to(tdt)
    k = torch.from_numpy(K).cuda().to(tdt)
    m = torch.from_numpy(mask).cuda() if mask is not None else None
    buf, out = _guarded((p.batch, p.num_heads, p.seq_q), torch.float32)
    ab.attn_bwd_lse(p, q, k, m, out)
    torch.cuda.synchronize()
    assert ab.check_device_error() == 0
    assert _guards_intact(buf)
    ref = OA.lse(p, Q.astype(np.float64), K.astype(np.float64), mask)
    got = out.cpu().numpy().astype(np.float64)
    empty = ref == OA.EMPTY_ROW_LSE
    assert np.all(got[empty] == np.float32(3.0e38))
    assert np.all(np.abs(got[~empty] - ref[~empty]) <= lse_bound(p, Q, K, mask, ref)[~empty])


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("name", sorted(GUARD_CASES))
def test_forward_writes_stay_inside_outputs(name, dtype):
    import torch
    import attention_backward_pass_gb300 as ab
    p = copy.copy(GUARD_CASES[name][0])
    p.dtype = dtype
    Q, K, V, _, mask = W.make_inputs(p, 79)
    tdt = torch.bfloat16 if dtype == W.DTYPE_BF16 else torch.float32
    to = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda().to(tdt)  # noqa: E731
    m = torch.from_numpy(mask).cuda() if mask is not None else None
    bo, O = _guarded(p.q_shape(), tdt)
    bl, LSE = _guarded((p.batch, p.num_heads, p.seq_q), torch.float32)
    ws = torch.empty(ab.fwd_workspace_size(p), dtype=torch.uint8, device="cuda")
    ab.attn_fwd(p, to(Q), to(K), to(V), m, O, LSE, ws)
    torch.cuda.synchronize()
    assert ab.check_device_error() == 0
    assert _guards_intact(bo) and _guards_intact(bl)
    f = lambda a: a.astype(np.float64)  # noqa: E731
    O_ref, LSE_ref = OA.forward(p, f(Q), f(K), f(V), mask)
    assert rel_err(O.float().cpu().numpy(), O_ref) <= TOL[dtype]
    got = LSE.cpu().numpy().astype(np.float64)
    empty = LSE_ref == OA.EMPTY_ROW_LSE
    assert np.all(got[empty] == np.float32(3.0e38))
    bound = lse_bound(p, Q, K, mask, LSE_ref)
    assert np.all(np.abs(got[~empty] - LSE_ref[~empty]) <= bound[~empty])


# shapes of the decode parity suite
@pytest.mark.parametrize("shape", [(3, 4, 2, 64, 17), (1, 16, 1, 64, 77), (2, 8, 1, 256, 300)])
def test_decode_writes_stay_inside_outputs(shape):
    import torch
    import attention_backward_pass_gb300 as ab
    dp = W.DecodeProblem(*shape)
    c = decode_case(dp, seed=5)
    t = {k: torch.from_numpy(np.ascontiguousarray(c[k])).cuda() for k in ("k", "v", "d_out", "probs")}
    bs, d_scores = _guarded((dp.num_seqs, dp.n_heads, dp.history_len), torch.float32)
    bq, d_q = _guarded((dp.num_seqs, dp.n_heads, dp.head_dim), torch.float32)
    ws = ab.alloc_decode_workspace(dp, "cuda")
    ab.attn_bwd_decode(dp, t["k"], t["v"], t["probs"], t["d_out"], d_scores, d_q, ws)
    q = torch.from_numpy(W.make_decode_queries(dp, 5)).cuda()
    hshape = (dp.num_seqs, dp.history_len, dp.n_kv_heads, dp.head_dim)
    bk, d_k = _guarded(hshape, torch.float32)
    bv, d_v = _guarded(hshape, torch.float32)
    ab.attn_bwd_decode_kv(dp, q, t["probs"], t["d_out"], d_scores, d_k, d_v)
    torch.cuda.synchronize()
    assert ab.check_device_error() == 0
    assert all(_guards_intact(b) for b in (bs, bq, bk, bv))
    rds, rdq = OD.decode_backward(c["k"], c["v"], c["probs"], c["d_out"])
    assert rel_err(d_scores.cpu().numpy(), rds) <= 2e-3 and rel_err(d_q.cpu().numpy(), rdq) <= 2e-3
    rdk, rdv = OD.decode_backward_kv(q.cpu().numpy(), c["probs"], c["d_out"],
                                     d_scores.cpu().numpy(), dp.n_kv_heads)
    assert rel_err(d_k.cpu().numpy(), rdk) <= 2e-3 and rel_err(d_v.cpu().numpy(), rdv) <= 2e-3
