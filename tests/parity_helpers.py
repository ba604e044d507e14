"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs, and compare.

Metric (per output tensor, over the compared slice):
    max |gpu - oracle| / max |oracle|
Bars: 2e-3 for fp32 I/O (TF32 tensor-core products), 2e-2 for bf16 I/O.
"""
from __future__ import annotations

import numpy as np

from attention_backward_pass_gb300 import workloads as W
from oracle import attention as OA
from oracle import decode as OD

TOL = {W.DTYPE_F32: 2e-3, W.DTYPE_BF16: 2e-2}


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    gpu = np.asarray(gpu, dtype=np.float64)
    denom = float(np.max(np.abs(ref))) if ref.size else 0.0
    if denom == 0.0:
        return float(np.max(np.abs(gpu))) if gpu.size else 0.0
    return float(np.max(np.abs(gpu - ref))) / denom


def strided_mask(p, kind, seed):
    """Input synthesis for masked cases: a logical additive mask L [B, H, Sq, Sk] (N(0,1) values, 20 % at the
    -1e30 sentinel, every head different) and the storage the oracle reads
    through p's element strides:
      per_head            [B, H, Sq, Sk]   strides (H Sq Sk, Sq Sk, Sk, 1)
      per_head_transposed [B, H, Sk, Sq]   strides (H Sq Sk, Sq Sk, 1, Sq)
      head_major          [H, B, Sk, Sq]   strides (Sq Sk, B Sq Sk, 1, Sq)
    Sets the strides on p and returns (storage, L)."""
    rng = np.random.default_rng(seed)
    B, H, Sq, Sk = p.batch, p.num_heads, p.seq_q, p.seq_k
    L = rng.standard_normal((B, H, Sq, Sk))
    L[rng.random(L.shape) < 0.2] = W.MASKED
    if kind == "per_head":
        store = L.copy()
        strides = (H * Sq * Sk, Sq * Sk, Sk, 1)
    elif kind == "per_head_transposed":
        store = np.ascontiguousarray(L.transpose(0, 1, 3, 2))
        strides = (H * Sq * Sk, Sq * Sk, 1, Sq)
    elif kind == "head_major":
        store = np.ascontiguousarray(L.transpose(1, 0, 3, 2))
        strides = (Sq * Sk, B * Sq * Sk, 1, Sq)
    else:
        raise ValueError(kind)
    p.has_mask = 1
    p.mask_stride_b, p.mask_stride_h, p.mask_stride_q, p.mask_stride_k = strides
    return store, L


def _torch_io(x, dtype, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)
    return t.to(torch.bfloat16) if dtype == W.DTYPE_BF16 else t


def make_case(p, seed, groups=None, fill_lse=1.0e4):
    """Seeded inputs plus O and LSE from the oracle forward, rounded once to
    the I/O dtype (O) and fp32 (LSE).  When ``groups`` is given, the forward
    runs only for those (b, kv-head) groups; the other heads get random O and
    a large LSE (their outputs are not compared)."""
    Q, K, V, dO, mask = W.make_inputs(p, seed)
    O, LSE = OA.forward(p, Q, K, V, mask, groups=groups)
    if groups is not None:
        rng = np.random.default_rng(seed + 1)
        G = p.num_heads // p.num_kv_heads
        done = np.zeros((p.batch, p.num_heads), dtype=bool)
        for b, g in groups:
            done[b, g * G:(g + 1) * G] = True
        for b in range(p.batch):
            for h in range(p.num_heads):
                if not done[b, h]:
                    LSE[b, h] = fill_lse
                    if p.layout == W.LAYOUT_BHSD:
                        O[b, h] = rng.standard_normal(O[b, h].shape)
                    else:
                        O[b, :, h] = rng.standard_normal(O[b, :, h].shape)
    O = W.round_io(O.astype(np.float32), p.dtype)
    LSE = LSE.astype(np.float32)
    return dict(Q=Q, K=K, V=V, dO=dO, mask=mask, O=O, LSE=LSE)


def run_gpu(p, case, device="cuda", repeat=1, recompute_lse=False):
    """Runs attn_bwd through the C ABI; returns fp64 numpy dQ, dK, dV.
    recompute_lse: pass no LSE, so the pass computes it itself."""
    import torch
    import attention_backward_pass_gb300 as ab
    t = {k: _torch_io(case[k], p.dtype, device) for k in ("Q", "K", "V", "O", "dO")}
    lse = None if recompute_lse else torch.from_numpy(case["LSE"]).to(device)
    mask = torch.from_numpy(case["mask"]).to(device) if case["mask"] is not None else None
    tdt = torch.bfloat16 if p.dtype == W.DTYPE_BF16 else torch.float32
    dQ = torch.full(p.q_shape(), float("nan"), dtype=tdt, device=device)
    dK = torch.full(p.kv_shape(), float("nan"), dtype=tdt, device=device)
    dV = torch.full(p.kv_shape(), float("nan"), dtype=tdt, device=device)
    ws = ab.alloc_workspace(p, device)
    ws.fill_(0xFF)  # contents on entry must not matter
    for _ in range(repeat):
        ab.attn_bwd(p, t["Q"], t["K"], t["V"], t["O"], t["dO"], lse, mask, dQ, dK, dV, ws)
    torch.cuda.synchronize()
    assert ab.check_device_error() == 0
    return [x.float().cpu().numpy().astype(np.float64) for x in (dQ, dK, dV)]


def oracle_grads(p, case, groups=None):
    f = lambda x: x.astype(np.float64)  # noqa: E731
    return OA.backward(p, f(case["Q"]), f(case["K"]), f(case["V"]), f(case["O"]), f(case["dO"]),
                       case["LSE"].astype(np.float64), case["mask"], groups=groups)


def select_groups(p, arr, groups, side):
    """Stack the slices of `arr` that belong to the (b, kv-head) groups."""
    G = p.num_heads // p.num_kv_heads
    out = []
    for b, g in groups:
        heads = range(g * G, (g + 1) * G) if side == "q" else [g]
        for h in heads:
            out.append(arr[b, h] if p.layout == W.LAYOUT_BHSD else arr[b, :, h])
    return np.stack(out)


def compare(p, case, groups=None, repeat=1, recompute_lse=False):
    """Returns {name: rel_err} for dQ, dK, dV (on the sampled groups if given)."""
    gpu = run_gpu(p, case, repeat=repeat, recompute_lse=recompute_lse)
    ref = oracle_grads(p, case, groups)
    errs = {}
    for name, g, r, side in zip(("dQ", "dK", "dV"), gpu, ref, ("q", "k", "k")):
        assert np.all(np.isfinite(g if groups is None else select_groups(p, g, groups, side))), name
        if groups is None:
            errs[name] = rel_err(g, r)
        else:
            errs[name] = rel_err(select_groups(p, g, groups, side),
                                 select_groups(p, r, groups, side))
    return errs


def lse_bound(p, Q, K, mask, ref):
    """Per-row bound on |LSE_gpu - LSE_oracle| derived from the arithmetic.
    The LSE is a smooth maximum of the row's scores (its gradient is a
    probability vector), so its error is at most the largest score error plus
    the error of the reduction:
      score:  (2 u_in + D 2^-23) |scale| max_j sum_d |q_id k_jd|, u_in = 2^-10 for
              fp32 inputs read as TF32 (truncation or rounding), 0 for bf16
              inputs (exact products), fp32 accumulation over D terms;
      reduce: Sk 2^-24 (recursive fp32 sum of at most Sk terms) + 2^-20 (ex2 /
              log2 approximations) + 2^-22 (|LSE| + max|mask|) (rounding of the
              scaled scores and of the result).
    Returns an array shaped like ``ref`` ([B, H, Sq])."""
    G = p.num_heads // p.num_kv_heads
    u_in = 2.0 ** -10 if p.dtype == W.DTYPE_F32 else 0.0
    mmax = 0.0
    if mask is not None:
        mv = np.asarray(mask, dtype=np.float64)
        mv = mv[mv > -1e30]
        mmax = float(np.max(np.abs(mv))) if mv.size else 0.0
    out = np.zeros_like(ref)
    for b in range(p.batch):
        for h in range(p.num_heads):
            q = np.abs(Q[b, h] if p.layout == W.LAYOUT_BHSD else Q[b, :, h]).astype(np.float64)
            kk = K[b, h // G] if p.layout == W.LAYOUT_BHSD else K[b, :, h // G]
            a = (q @ np.abs(kk).astype(np.float64).T).max(axis=1)
            out[b, h] = ((2 * u_in + p.head_dim * 2.0 ** -23) * abs(p.scale) * a
                         + p.seq_k * 2.0 ** -24 + 2.0 ** -20
                         + 2.0 ** -22 * (np.abs(ref[b, h]) + mmax))
    return out


def run_lse_gpu(p, Q, K, mask, device="cuda"):
    """attn_bwd_lse through the C ABI; returns fp64 numpy LSE [B, H, Sq]."""
    import torch
    import attention_backward_pass_gb300 as ab
    q = _torch_io(Q, p.dtype, device)
    k = _torch_io(K, p.dtype, device)
    m = torch.from_numpy(mask).to(device) if mask is not None else None
    out = torch.full((p.batch, p.num_heads, p.seq_q), float("nan"), device=device)
    ab.attn_bwd_lse(p, q, k, m, out)
    torch.cuda.synchronize()
    assert ab.check_device_error() == 0
    return out.cpu().numpy().astype(np.float64)


def run_fwd_gpu(p, Q, K, V, mask, device="cuda"):
    """attn_fwd through the C ABI; returns fp64 numpy O (p's layout) and LSE."""
    import torch
    import attention_backward_pass_gb300 as ab
    q = _torch_io(Q, p.dtype, device)
    k = _torch_io(K, p.dtype, device)
    v = _torch_io(V, p.dtype, device)
    m = torch.from_numpy(mask).to(device) if mask is not None else None
    o = torch.full(p.q_shape(), float("nan"), dtype=q.dtype, device=device)
    lse = torch.full((p.batch, p.num_heads, p.seq_q), float("nan"), device=device)
    ws = torch.empty(ab.fwd_workspace_size(p), dtype=torch.uint8, device=device)
    ab.attn_fwd(p, q, k, v, m, o, lse, ws)
    torch.cuda.synchronize()
    assert ab.check_device_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def decode_case(p, seed):
    k, v, d_out, logits = W.make_decode_inputs(p, seed)
    probs = OD.softmax_rows(logits).astype(np.float32)
    return dict(k=k, v=v, d_out=d_out, probs=probs)


def run_decode_kv_gpu(p, case, q, d_scores, device="cuda"):
    """Decode pass 2 on the GPU from the given (fp32) d_scores."""
    import torch
    import attention_backward_pass_gb300 as ab
    t = {k: torch.from_numpy(np.ascontiguousarray(case[k])).to(device) for k in ("d_out", "probs")}
    tq = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).to(device)
    tds = torch.from_numpy(np.ascontiguousarray(d_scores, dtype=np.float32)).to(device)
    shape = (p.num_seqs, p.history_len, p.n_kv_heads, p.head_dim)
    d_k = torch.full(shape, float("nan"), device=device)
    d_v = torch.full(shape, float("nan"), device=device)
    ab.attn_bwd_decode_kv(p, tq, t["probs"], t["d_out"], tds, d_k, d_v)
    torch.cuda.synchronize()
    return d_k.cpu().numpy().astype(np.float64), d_v.cpu().numpy().astype(np.float64)


def run_decode_gpu(p, case, device="cuda", repeat=1):
    import torch
    import attention_backward_pass_gb300 as ab
    t = {k: torch.from_numpy(np.ascontiguousarray(case[k])).to(device)
         for k in ("k", "v", "d_out", "probs")}
    d_scores = torch.full((p.num_seqs, p.n_heads, p.history_len), float("nan"), device=device)
    d_q = torch.full((p.num_seqs, p.n_heads, p.head_dim), float("nan"), device=device)
    ws = ab.alloc_decode_workspace(p, device)
    for _ in range(repeat):
        ab.attn_bwd_decode(p, t["k"], t["v"], t["probs"], t["d_out"], d_scores, d_q, ws)
    torch.cuda.synchronize()
    assert ab.check_device_error() == 0
    return d_scores.cpu().numpy().astype(np.float64), d_q.cpu().numpy().astype(np.float64)
