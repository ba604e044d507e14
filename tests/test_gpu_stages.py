"""The three stages of the backward pass called one by one.

attn_bwd runs attn_bwd_prepare, attn_bwd_tiles and attn_bwd_finish on one
stream; inside attn_bwd the tile kernel may start while the prepare kernel
finishes (a programmatic dependent launch), while a direct attn_bwd_tiles call
launches normally.  These tests call the stages through the C ABI, check dQ,
dK, dV against the fp64 oracle at the parity bars, and check that they agree
with attn_bwd on the same inputs (dK, dV exactly; dQ, which is summed with
atomics or, deterministic, in a fixed order, within one rounding step).
"""
import copy

import numpy as np
import pytest

from attention_backward_pass_gb300 import workloads as W

from parity_helpers import TOL, _torch_io, make_case, oracle_grads, rel_err

pytestmark = pytest.mark.gpu


def _P(**kw):
    base = dict(batch=2, num_heads=4, num_kv_heads=2, seq_q=300, seq_k=300, head_dim=64,
                scale=0.125, causal=1)
    base.update(kw)
    return W.AttnProblem(**base)


CASES = {
    "gqa_causal_d64": _P(),
    "gqa_window_bshd_d128": _P(seq_q=400, seq_k=400, head_dim=128, scale=1 / np.sqrt(128),
                               window=150, layout=W.LAYOUT_BSHD),
    "mask_dropout_d64": _P(num_heads=2, num_kv_heads=2, seq_q=200, seq_k=333, causal_offset=133,
                           has_mask=1, mask_stride_b=200 * 333, mask_stride_q=333,
                           mask_stride_k=1, dropout_prob=0.1, seed=0x5EED0010),
}


def _run(p, case, staged):
    import torch
    import attention_backward_pass_gb300 as ab
    t = {k: _torch_io(case[k], p.dtype, "cuda") for k in ("Q", "K", "V", "O", "dO")}
    lse = torch.from_numpy(case["LSE"]).cuda()
    mask = torch.from_numpy(case["mask"]).cuda() if case["mask"] is not None else None
    tdt = torch.bfloat16 if p.dtype == W.DTYPE_BF16 else torch.float32
    dQ = torch.full(p.q_shape(), float("nan"), dtype=tdt, device="cuda")
    dK = torch.full(p.kv_shape(), float("nan"), dtype=tdt, device="cuda")
    dV = torch.full(p.kv_shape(), float("nan"), dtype=tdt, device="cuda")
    ws = ab.alloc_workspace(p, "cuda")
    ws.fill_(0xFF)
    if staged:
        ab.attn_bwd_prepare(p, t["Q"], t["K"], t["O"], t["dO"], lse, dQ, ws)
        ab.attn_bwd_tiles(p, t["Q"], t["K"], t["V"], t["dO"], mask, dQ, dK, dV, ws)
        ab.attn_bwd_finish(p, dQ, ws)
    else:
        ab.attn_bwd(p, t["Q"], t["K"], t["V"], t["O"], t["dO"], lse, mask, dQ, dK, dV, ws)
    torch.cuda.synchronize()
    assert ab.check_device_error() == 0
    return [x.float().cpu().numpy().astype(np.float64) for x in (dQ, dK, dV)]


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("name", sorted(CASES))
def test_stages_match_oracle_and_attn_bwd(name, dtype, deterministic):
    p = copy.copy(CASES[name])
    p.dtype = dtype
    p.deterministic = deterministic
    case = make_case(p, seed=77)
    staged = _run(p, case, staged=True)
    fused = _run(p, case, staged=False)
    ref = oracle_grads(p, case)
    for nm, s, f, r in zip(("dQ", "dK", "dV"), staged, fused, ref):
        assert np.all(np.isfinite(s)), nm
        assert rel_err(s, r) <= TOL[p.dtype], (nm, rel_err(s, r))
        if nm == "dQ" and not deterministic:
            # fp32 atomics: the order of the additions differs from run to run
            assert rel_err(s, f) <= (1e-5 if dtype == W.DTYPE_F32 else 1e-2), (nm, rel_err(s, f))
        else:
            assert np.array_equal(s, f), nm
