"""The decode backward entry point that allocates nothing.

Some callers cannot hand the library a workspace (no allocator available or
allowed where they run).  attn_bwd_decode_noalloc keeps its scratch in a
fixed device array inside the library instead.  These tests call it through
the C ABI and check that, on two calls in a row, it gives the same d_scores
and d_q as attn_bwd_decode (which takes a caller workspace), within the
fp32 parity tolerance, and that a problem too large for the array is
refused.  This file is collected last on purpose.
"""
import numpy as np
import pytest

from attention_backward_pass_gb300 import workloads as W

from parity_helpers import decode_case, rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _run_both(p, seed, oracle_seqs=()):
    import torch
    import attention_backward_pass_gb300 as ab
    case = decode_case(p, seed)
    t = {k: torch.from_numpy(np.ascontiguousarray(case[k])).cuda()
         for k in ("k", "v", "d_out", "probs")}
    shape_s = (p.num_seqs, p.n_heads, p.history_len)
    shape_q = (p.num_seqs, p.n_heads, p.head_dim)
    ref_s = torch.full(shape_s, float("nan"), device="cuda")
    ref_q = torch.full(shape_q, float("nan"), device="cuda")
    ws = ab.alloc_decode_workspace(p)
    ab.attn_bwd_decode(p, t["k"], t["v"], t["probs"], t["d_out"], ref_s, ref_q, ws)
    outs = []
    for _ in range(2):  # two calls in a row share the one scratch array
        s = torch.full(shape_s, float("nan"), device="cuda")
        q = torch.full(shape_q, float("nan"), device="cuda")
        ab.attn_bwd_decode_noalloc(p, t["k"], t["v"], t["probs"], t["d_out"], s, q)
        outs.append((s, q))
    torch.cuda.synchronize()
    assert ab.check_device_error() == 0
    ref_s, ref_q = ref_s.cpu().numpy(), ref_q.cpu().numpy()
    for s, q in outs:
        s, q = s.cpu().numpy(), q.cpu().numpy()
        assert np.all(np.isfinite(s)) and np.all(np.isfinite(q))
        assert rel_err(s, ref_s) <= TOL, rel_err(s, ref_s)
        assert rel_err(q, ref_q) <= TOL, rel_err(q, ref_q)
        if oracle_seqs:
            from oracle import decode as OD
            seqs = list(oracle_seqs)
            rds, rdq = OD.decode_backward(case["k"], case["v"], case["probs"], case["d_out"],
                                          seqs=seqs)
            assert rel_err(s[seqs], rds[seqs]) <= TOL, rel_err(s[seqs], rds[seqs])
            assert rel_err(q[seqs], rdq[seqs]) <= TOL, rel_err(q[seqs], rdq[seqs])


@pytest.mark.parametrize("prob", [W.decode(), W.DecodeProblem(3, 4, 2, 64, 17)],
                         ids=["64seq_8h_d256_4096", "3seq_4h_2kv_d64_17"])
def test_noalloc_matches_workspace_entry_point(prob):
    _run_both(prob, seed=11)


def test_noalloc_uses_fewer_splits_when_the_usual_ones_do_not_fit():
    """900 (sequence, KV head) pairs with D = 256, 8 query heads per KV head
    and a 64-key history: the partial sums of the usual split count (one
    split per SM, each holding a slot for every pair it touches) need more
    than the 8 MiB array, those of one split fit, so the entry point runs
    with fewer splits.  Checked against the workspace entry point and, on a
    few sequences, against the fp64 oracle."""
    import attention_backward_pass_gb300 as ab
    p = W.DecodeProblem(900, 8, 1, 256, 64)
    assert ab.decode_workspace_size(p) > (8 << 20)
    _run_both(p, seed=13, oracle_seqs=(0, 450, 899))


def test_noalloc_rejects_problem_beyond_scratch():
    import torch
    import attention_backward_pass_gb300 as ab
    # 4096 sequences x 8 heads x (256 + 8) floats = 34 MiB for one split > 8 MiB
    p = W.DecodeProblem(4096, 8, 1, 256, 16)
    dummy = torch.empty(16, device="cuda")
    with pytest.raises(ab.AttnError) as e:
        ab.attn_bwd_decode_noalloc(p, dummy, dummy, dummy, dummy, dummy, dummy)
    assert e.value.status == -6
