"""Pins of the fp64 oracle against facts other than itself (CPU only).

* finite differences of L = sum(dO * O(Q, K, V)) with mask and dropout fixed
* torch autograd of a materialised softmax attention (library special case)
* invariants: sum_j dS_ij = 0, sum_j dK_j = 0, sum_j dV_j = sum_i dO_i,
  GQA == MHA on repeated K/V with dK/dV summed over the group
* closed forms: Sk = 1, Q = 0, fully masked rows, a hand-worked example
* visibility: special cases that reduce to numpy's triangle routines
* Philox4x32-10 known-answer vectors and keep-rate statistics
* decode: finite differences of the decode loss, one-hot probabilities,
  sum_pd == Delta
"""
import math
import os

import numpy as np
import pytest

from attention_backward_pass_gb300 import workloads as W
from oracle import attention as A
from oracle import decode as Dec
from oracle import philox

from parity_helpers import strided_mask

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(**kw):
    base = dict(batch=1, num_heads=2, num_kv_heads=2, seq_q=5, seq_k=7, head_dim=4,
                scale=0.7)
    base.update(kw)
    p = W.AttnProblem(**base)
    if p.has_mask and p.mask_stride_q == 0:
        p.mask_stride_b, p.mask_stride_h = p.seq_q * p.seq_k, 0
        p.mask_stride_q, p.mask_stride_k = p.seq_k, 1
    return p


def inputs64(p, seed, mask_frac=0.25):
    Q, K, V, dO, mask = W.make_inputs(p, seed, do_std=1.0, mask_frac=mask_frac)
    return [x.astype(np.float64) if x is not None else None for x in (Q, K, V, dO, mask)]


VARIANTS = {
    "plain": dict(),
    "causal": dict(causal=1),
    "causal_offset": dict(causal=1, causal_offset=2),
    "window": dict(window=3),
    "causal_window_offset": dict(causal=1, window=3, causal_offset=2),
    "mask": dict(has_mask=1),
    "dropout": dict(dropout_prob=0.3, seed=0x1234_0000_0042),
    "gqa_bshd": dict(num_heads=4, num_kv_heads=2, layout=W.LAYOUT_BSHD, causal=1),
    "everything": dict(num_heads=4, num_kv_heads=1, causal=1, causal_offset=3, window=4,
                       has_mask=1, dropout_prob=0.25, seed=99, layout=W.LAYOUT_BSHD),
}


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_finite_differences(name):
    p = small(**VARIANTS[name])
    Q, K, V, dO, mask = inputs64(p, seed=11)
    O, LSE = A.forward(p, Q, K, V, mask)
    dQ, dK, dV = A.backward(p, Q, K, V, O, dO, LSE, mask)
    h = 1e-6
    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        fd = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = X[idx]
            X[idx] = old + h
            lp = A.loss(p, Q, K, V, dO, mask)
            X[idx] = old - h
            lm = A.loss(p, Q, K, V, dO, mask)
            X[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - G)) / max(np.max(np.abs(G)), 1e-30)
        assert err < 1e-6, (name, err)


def _torch_reference(p, Q, K, V, dO, mask, M=None):
    torch = pytest.importorskip("torch")
    q = torch.tensor(Q, dtype=torch.float64, requires_grad=True)
    k = torch.tensor(K, dtype=torch.float64, requires_grad=True)
    v = torch.tensor(V, dtype=torch.float64, requires_grad=True)
    G = p.num_heads // p.num_kv_heads
    if p.layout == W.LAYOUT_BSHD:
        qh, kh, vh = q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2)
    else:
        qh, kh, vh = q, k, v
    kh = kh.repeat_interleave(G, dim=1)
    vh = vh.repeat_interleave(G, dim=1)
    s = p.scale * qh @ kh.transpose(-1, -2)
    i = torch.arange(p.seq_q)[:, None] + p.causal_offset
    j = torch.arange(p.seq_k)[None, :]
    allowed = torch.ones(p.seq_q, p.seq_k, dtype=torch.bool)
    if p.causal:
        allowed &= j <= i
    if p.window:
        allowed &= (i - j).abs() < p.window
    allowed = allowed.expand_as(s).clone()
    if mask is not None:
        m = torch.tensor(mask, dtype=torch.float64)
        allowed &= m > -1e30
        s = s + torch.where(m > -1e30, m, torch.zeros_like(m))
    s = s.masked_fill(~allowed, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    P = torch.softmax(s, dim=-1)
    if M is not None:
        P = P * torch.tensor(M, dtype=torch.float64)
    o = P @ vh
    if p.layout == W.LAYOUT_BSHD:
        o = o.transpose(1, 2)
    o.backward(torch.tensor(dO, dtype=torch.float64))
    return (o.detach().numpy(), lse.detach().numpy(), q.grad.numpy(), k.grad.numpy(),
            v.grad.numpy())


@pytest.mark.parametrize("name", ["plain", "causal", "causal_window_offset", "mask",
                                  "gqa_bshd", "dropout"])
def test_against_torch_autograd(name):
    p = small(**VARIANTS[name])
    Q, K, V, dO, mask = inputs64(p, seed=5)
    M = None
    if p.dropout_prob > 0:
        M = np.stack([np.stack([A.multiplier(p, b, h) for h in range(p.num_heads)])
                      for b in range(p.batch)])
    o_t, lse_t, dq_t, dk_t, dv_t = _torch_reference(p, Q, K, V, dO, mask, M)
    O, LSE = A.forward(p, Q, K, V, mask)
    dQ, dK, dV = A.backward(p, Q, K, V, O, dO, LSE, mask)
    np.testing.assert_allclose(O, o_t, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(LSE, lse_t, rtol=1e-12, atol=1e-12)
    for a, b in ((dQ, dq_t), (dK, dk_t), (dV, dv_t)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("kind", ["per_head", "per_head_transposed", "head_major"])
def test_strided_per_head_mask_against_torch_autograd(kind):
    """The mask is indexed with the query head (not its KV head) and with the
    q / k strides the caller gives (page 2, fab2_mask_at).  GQA with two query
    heads per KV head, two batches and a different mask per (b, h): a head
    index taken from the KV head, a swapped q / k stride or a dropped batch
    term reads another head's or the transposed values and fails here."""
    p = small(batch=2, num_heads=4, num_kv_heads=2, seq_q=5, seq_k=7, causal=1,
              causal_offset=3, layout=W.LAYOUT_BSHD, dropout_prob=0.2, seed=31)
    Q, K, V, dO, _ = inputs64(p, seed=9)
    store, L = strided_mask(p, kind, seed=17)
    M = np.stack([np.stack([A.multiplier(p, b, h) for h in range(p.num_heads)])
                  for b in range(p.batch)])
    o_t, lse_t, dq_t, dk_t, dv_t = _torch_reference(p, Q, K, V, dO, L, M)
    O, LSE = A.forward(p, Q, K, V, store)
    dQ, dK, dV = A.backward(p, Q, K, V, O, dO, LSE, store)
    np.testing.assert_allclose(O, o_t, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(LSE, lse_t, rtol=1e-12, atol=1e-12)
    for a, b in ((dQ, dq_t), (dK, dk_t), (dV, dv_t)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)
    # the LSE sweep reads the mask the same way
    np.testing.assert_allclose(A.lse(p, Q, K, store), lse_t, rtol=1e-12, atol=1e-12)


def test_mask_head_stride_reaches_every_query_head():
    """Brute force on the index rule alone: with a per-head mask that holds
    the flat element index, mask_slice returns b*sb + h*sh + i*sq + j*sk."""
    p = small(batch=2, num_heads=6, num_kv_heads=2, seq_q=3, seq_k=4, has_mask=1)
    sb, sh, sq, sk = 97, 13, 1, 3
    p.mask_stride_b, p.mask_stride_h, p.mask_stride_q, p.mask_stride_k = sb, sh, sq, sk
    flat = np.arange(2 * 97 + 6 * 13 + 10, dtype=np.float64)
    for b in range(p.batch):
        for h in range(p.num_heads):
            got = A.mask_slice(p, flat, b, h)
            for i in range(p.seq_q):
                for j in range(p.seq_k):
                    assert got[i, j] == b * sb + h * sh + i * sq + j * sk


@pytest.mark.parametrize("name", ["plain", "causal_window_offset", "mask", "dropout",
                                  "everything"])
def test_invariants(name):
    p = small(**VARIANTS[name], seq_q=6, seq_k=9)
    Q, K, V, dO, mask = inputs64(p, seed=3, mask_frac=0.2)
    O, LSE = A.forward(p, Q, K, V, mask)
    dQ, dK, dV, parts = A.backward(p, Q, K, V, O, dO, LSE, mask, return_parts=True)
    for (b, h), d in parts.items():
        rows = np.abs(d["dS"].sum(axis=1))
        assert np.max(rows) < 1e-12 * max(1.0, np.abs(d["dS"]).max()), (b, h)
    # sum_j dK_j = 0 per KV head (sum of the group's sum_j dS_ij Q_i terms)
    kv_axis = 2 if p.layout == W.LAYOUT_BHSD else 1
    assert np.max(np.abs(dK.sum(axis=kv_axis))) < 1e-11
    if p.dropout_prob == 0 and not p.has_mask and p.window == 0 and not p.causal:
        G = p.num_heads // p.num_kv_heads
        q_axis = kv_axis
        sdo = dO.sum(axis=q_axis)  # [B,H,D]
        sdo = sdo.reshape(p.batch, p.num_kv_heads, G, p.head_dim).sum(axis=2)
        np.testing.assert_allclose(dV.sum(axis=kv_axis), sdo, rtol=1e-12, atol=1e-12)


def test_sum_dv_equals_sum_do_with_causal_rows():
    p = small(causal=1, causal_offset=0, seq_q=6, seq_k=6)
    Q, K, V, dO, mask = inputs64(p, seed=8)
    O, LSE = A.forward(p, Q, K, V, mask)
    _, _, dV = A.backward(p, Q, K, V, O, dO, LSE, mask)
    np.testing.assert_allclose(dV.sum(axis=2), dO.sum(axis=2), rtol=1e-12, atol=1e-12)


def test_gqa_equals_repeated_mha():
    p = small(num_heads=6, num_kv_heads=2, causal=1, window=4, causal_offset=1, has_mask=1,
              dropout_prob=0.2, seed=7)
    Q, K, V, dO, mask = inputs64(p, seed=21)
    O, LSE = A.forward(p, Q, K, V, mask)
    dQ, dK, dV = A.backward(p, Q, K, V, O, dO, LSE, mask)
    G = 3
    pm = small(num_heads=6, num_kv_heads=6, causal=1, window=4, causal_offset=1, has_mask=1,
               dropout_prob=0.2, seed=7)
    pm.mask_stride_b, pm.mask_stride_q, pm.mask_stride_k = p.mask_stride_b, p.mask_stride_q, 1
    Kr, Vr = np.repeat(K, G, axis=1), np.repeat(V, G, axis=1)
    Om, LSEm = A.forward(pm, Q, Kr, Vr, mask)
    np.testing.assert_allclose(Om, O, rtol=1e-13, atol=1e-13)
    dQm, dKm, dVm = A.backward(pm, Q, Kr, Vr, Om, dO, LSEm, mask)
    np.testing.assert_allclose(dQm, dQ, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dKm.reshape(1, 2, G, 7, 4).sum(axis=2), dK, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dVm.reshape(1, 2, G, 7, 4).sum(axis=2), dV, rtol=1e-12, atol=1e-13)


def test_single_key_closed_form():
    # Sk = 1: P = 1, dS = 0 (so dQ = dK = 0) and dV = sum_i M_i dO_i
    p = small(seq_k=1, dropout_prob=0.5, seed=3)
    Q, K, V, dO, mask = inputs64(p, seed=2)
    O, LSE = A.forward(p, Q, K, V, mask)
    dQ, dK, dV = A.backward(p, Q, K, V, O, dO, LSE, mask)
    assert np.max(np.abs(dQ)) < 1e-13 and np.max(np.abs(dK)) < 1e-13
    for h in range(p.num_heads):
        M = A.multiplier(p, 0, h)[:, 0]
        np.testing.assert_allclose(dV[0, h, 0], (M[:, None] * dO[0, h]).sum(axis=0), rtol=1e-12)
        np.testing.assert_allclose(LSE[0, h], p.scale * Q[0, h] @ K[0, h, 0], rtol=1e-12)


def test_zero_queries_give_uniform_probabilities():
    p = small(causal=1, window=3, causal_offset=1)
    Q, K, V, dO, mask = inputs64(p, seed=4)
    Q[:] = 0.0
    O, LSE = A.forward(p, Q, K, V, mask)
    _, _, _, parts = A.backward(p, Q, K, V, O, dO, LSE, mask, return_parts=True)
    vis = A.visible(p.seq_q, p.seq_k, 1, 1, 3)
    expect = vis / vis.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(parts[(0, 0)]["P"], expect, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(LSE[0, 0], np.log(vis.sum(axis=1)), rtol=1e-14)


def test_fully_masked_rows():
    # window 1 with causal offset beyond seq_k leaves rows with no visible key
    p = small(causal=0, window=1, causal_offset=5, seq_q=4, seq_k=7)
    Q, K, V, dO, mask = inputs64(p, seed=9)
    O, LSE = A.forward(p, Q, K, V, mask)
    vis = A.visible(4, 7, 0, 5, 1)
    empty = ~vis.any(axis=1)
    assert empty.any() and (~empty).any()
    assert np.all(LSE[0, :, empty] == A.EMPTY_ROW_LSE)
    dQ, dK, dV = A.backward(p, Q, K, V, O, dO, LSE, mask)
    assert np.all(dQ[0, :, empty] == 0.0) and np.all(O[0, :, empty] == 0.0)
    assert np.all(np.isfinite(dK)) and np.all(np.isfinite(dV))


@pytest.mark.parametrize("name", ["plain", "causal", "causal_window_offset", "mask",
                                  "gqa_bshd", "everything"])
def test_lse_against_torch_logsumexp(name):
    # the LSE sweep alone (no forward): torch's logsumexp over the allowed
    # scores; rows with no allowed key are -inf there and 3e38 in the oracle
    p = small(**VARIANTS[name])
    Q, K, V, dO, mask = inputs64(p, seed=21)
    _, lse_t, _, _, _ = _torch_reference(p, Q, K, V, dO, mask)
    got = A.lse(p, Q, K, mask)
    empty = ~np.isfinite(lse_t)
    np.testing.assert_allclose(got[~empty], lse_t[~empty], rtol=1e-12, atol=1e-12)
    assert np.all(got[empty] == A.EMPTY_ROW_LSE)


def test_lse_online_recurrence_and_dropout_independence():
    # the page's sweep 1 taken key by key (running maximum m, running sum l
    # rescaled by exp(m - m_new)) in plain Python on a tiny case, with rows
    # that have no visible key; dropout does not change the LSE
    p = small(causal=1, causal_offset=1, window=2, has_mask=1, seq_q=6, seq_k=5)
    Q, K, V, dO, mask = inputs64(p, seed=4, mask_frac=0.4)
    # finite additive values where the mask is not hard
    mask = np.where(mask <= -1e30, mask, np.random.default_rng(3).normal(size=mask.shape))
    got = A.lse(p, Q, K, mask)
    G = p.num_heads // p.num_kv_heads
    for h in range(p.num_heads):
        for i in range(p.seq_q):
            m, l = -math.inf, 0.0
            for j in range(p.seq_k):
                qa = i + p.causal_offset
                if j > qa or abs(qa - j) >= p.window:
                    continue
                mv = mask[0, 0, i, j]
                if mv <= -1e30:
                    continue
                s = p.scale * sum(Q[0, h, i, d] * K[0, h // G, j, d] for d in range(4)) + mv
                m_new = max(m, s)
                l = l * math.exp(m - m_new) + math.exp(s - m_new)
                m = m_new
            want = m + math.log(l) if l > 0 else A.EMPTY_ROW_LSE
            assert abs(got[0, h, i] - want) <= 1e-12 * max(1.0, abs(want)), (h, i)
    pd = small(causal=1, causal_offset=1, window=2, has_mask=1, seq_q=6, seq_k=5,
               dropout_prob=0.5, seed=7)
    np.testing.assert_array_equal(A.lse(pd, Q, K, mask), got)


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, expr = line.split(None, 1)
            vals[k] = eval(expr, {"log": math.log})
    return vals


def test_hand_worked_example():
    g = _golden("worked_example_1x2.txt")
    p = W.AttnProblem(1, 1, 1, 1, 2, 1, scale=1.0)
    Q = np.array([1.0]).reshape(1, 1, 1, 1)
    K = np.array([0.0, math.log(3.0)]).reshape(1, 1, 2, 1)
    V = np.array([1.0, 5.0]).reshape(1, 1, 2, 1)
    dO = np.array([1.0]).reshape(1, 1, 1, 1)
    O, LSE = A.forward(p, Q, K, V)
    assert abs(LSE[0, 0, 0] - g["lse"]) < 1e-14 and abs(O[0, 0, 0, 0] - g["o"]) < 1e-14
    assert abs(A.delta(dO[0, 0], O[0, 0])[0] - g["delta"]) < 1e-14
    dQ, dK, dV = A.backward(p, Q, K, V, O, dO, LSE)
    assert abs(dQ[0, 0, 0, 0] - g["dq"]) < 1e-14
    np.testing.assert_allclose(dK[0, 0, :, 0], [g["dk0"], g["dk1"]], atol=1e-14)
    np.testing.assert_allclose(dV[0, 0, :, 0], [g["dv0"], g["dv1"]], atol=1e-14)


# ---------------------------------------------------------------- visibility

@pytest.mark.parametrize("sq,sk", [(1, 1), (5, 5), (4, 9), (9, 4)])
def test_visibility_special_cases(sq, sk):
    ones = np.ones((sq, sk), dtype=bool)
    assert np.array_equal(A.visible(sq, sk, 0, 0, 0), ones)
    for off in range(0, sk + 2):
        # causal with offset: bottom-right style alignment == tril with diagonal offset
        assert np.array_equal(A.visible(sq, sk, 1, off, 0), np.tril(ones, k=off))
    for w in range(1, sk + 2):
        band = np.tril(ones, k=w - 1) & np.triu(ones, k=-(w - 1))
        assert np.array_equal(A.visible(sq, sk, 0, 0, w), band)
        assert np.array_equal(A.visible(sq, sk, 1, 0, w), np.tril(ones) & np.triu(ones, k=-(w - 1)))
        for off in range(0, 3):
            sb = np.tril(ones, k=off + w - 1) & np.triu(ones, k=off - (w - 1))
            assert np.array_equal(A.visible(sq, sk, 0, off, w), sb)


def test_mask_sentinel_and_broadcast():
    p = small(has_mask=1, num_heads=3, num_kv_heads=3)
    mask = np.zeros((1, 1, p.seq_q, p.seq_k))
    mask[0, 0, 1, 2] = -1e30
    mask[0, 0, 2, 3] = -np.inf
    mask[0, 0, 3, 4] = -0.99e30  # finite, below but above the sentinel: added, not hard
    for h in range(3):
        hard, bias = A.hard_and_bias(p, mask, 0, h)
        assert hard[1, 2] and hard[2, 3] and not hard[3, 4]
        assert bias[3, 4] == -0.99e30 and hard.sum() == 2


# ---------------------------------------------------------------- dropout

def test_philox_known_answers():
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        out = philox.philox4x32_10(v[0], v[1], v[2], v[3], v[4], v[5])
        assert [int(o) for o in out] == v[6:10]


@pytest.mark.parametrize("p_drop", [0.1, 0.5, 0.9])
def test_keep_rate(p_drop):
    n = 0
    kept = 0
    for bh in range(4):
        k = philox.keep_mask(0xABCDEF0123, bh, 500, 500, p_drop)
        n += k.size
        kept += int(k.sum())
    rate = kept / n
    sigma = math.sqrt(p_drop * (1 - p_drop) / n)
    assert abs(rate - (1 - p_drop)) < 4 * sigma


def test_dropout_edges():
    assert philox.keep_mask(1, 0, 3, 3, 0.0).all()
    assert philox.keep_threshold(0.0) == 0
    assert philox.keep_threshold(0.5) == 2 ** 31
    assert philox.keep_threshold(0.99999999999) <= 2 ** 32 - 1
    M = philox.dropout_multiplier(5, 2, 8, 8, 0.25)
    assert set(np.unique(M)) <= {0.0, 1.0 / (1.0 - np.float64(np.float32(0.25)))}
    # the word used for query i is word (i & 3) of the counter (i >> 2, j, bh, 0)
    words = philox.philox4x32_10(1, 3, 2, 0, 5, 0)
    keep = philox.keep_mask(5, 2, 8, 8, 0.25)
    T = philox.keep_threshold(0.25)
    for i in range(4, 8):
        assert keep[i, 3] == (int(words[i & 3]) >= T)


# ---------------------------------------------------------------- decode

def test_decode_finite_differences():
    rng = np.random.default_rng(0)
    N, hist, n_kv, n_heads, D = 2, 6, 2, 4, 3
    k = rng.standard_normal((N, hist, n_kv, D))
    v = rng.standard_normal((N, hist, n_kv, D))
    q = rng.standard_normal((N, n_heads, D))
    d_out = rng.standard_normal((N, n_heads, D))

    def loss(qq):
        tot = 0.0
        for n in range(N):
            for h in range(n_heads):
                kv = h // (n_heads // n_kv)
                sc = k[n, :, kv] @ qq[n, h]          # unscaled scores
                pr = Dec.softmax_rows(sc)
                tot += d_out[n, h] @ (pr @ v[n, :, kv])
        return tot

    scores = np.einsum("njkd,nhd->nhj", k, q)
    kv_of = np.arange(n_heads) // (n_heads // n_kv)
    scores = np.stack([np.stack([k[n, :, kv_of[h]] @ q[n, h] for h in range(n_heads)])
                       for n in range(N)])
    probs = Dec.softmax_rows(scores)
    d_scores, d_q = Dec.decode_backward(k, v, probs, d_out)
    h = 1e-6
    fd_q = np.zeros_like(q)
    for idx in np.ndindex(q.shape):
        qp, qm = q.copy(), q.copy()
        qp[idx] += h
        qm[idx] -= h
        fd_q[idx] = (loss(qp) - loss(qm)) / (2 * h)
    np.testing.assert_allclose(d_q, fd_q, rtol=1e-6, atol=1e-8)
    # d_scores is the gradient of the same loss w.r.t. the scores
    for n in range(N):
        for hh in range(n_heads):
            kv = kv_of[hh]
            for j in range(hist):
                sp, sm = scores[n, hh].copy(), scores[n, hh].copy()
                sp[j] += h
                sm[j] -= h
                fp = d_out[n, hh] @ (Dec.softmax_rows(sp) @ v[n, :, kv])
                fm = d_out[n, hh] @ (Dec.softmax_rows(sm) @ v[n, :, kv])
                assert abs((fp - fm) / (2 * h) - d_scores[n, hh, j]) < 1e-7


def test_decode_kv_finite_differences():
    """Pass 2 (history gradients) against central differences of the decode
    loss sum_h d_out_h . out_h w.r.t. k_hist and v_hist, with d_scores from
    pass 1."""
    rng = np.random.default_rng(3)
    N, hist, n_kv, n_heads, D = 2, 5, 2, 4, 3
    k = rng.standard_normal((N, hist, n_kv, D))
    v = rng.standard_normal((N, hist, n_kv, D))
    q = rng.standard_normal((N, n_heads, D))
    d_out = rng.standard_normal((N, n_heads, D))
    kv_of = np.arange(n_heads) // (n_heads // n_kv)

    def loss(kk, vv):
        tot = 0.0
        for n in range(N):
            for h in range(n_heads):
                pr = Dec.softmax_rows(kk[n, :, kv_of[h]] @ q[n, h])
                tot += d_out[n, h] @ (pr @ vv[n, :, kv_of[h]])
        return tot

    scores = np.stack([np.stack([k[n, :, kv_of[h]] @ q[n, h] for h in range(n_heads)])
                       for n in range(N)])
    probs = Dec.softmax_rows(scores)
    d_scores, _ = Dec.decode_backward(k, v, probs, d_out)
    d_k, d_v = Dec.decode_backward_kv(q, probs, d_out, d_scores, n_kv)
    h = 1e-6
    fd_k, fd_v = np.zeros_like(k), np.zeros_like(v)
    for idx in np.ndindex(k.shape):
        kp, km = k.copy(), k.copy()
        kp[idx] += h
        km[idx] -= h
        fd_k[idx] = (loss(kp, v) - loss(km, v)) / (2 * h)
        vp, vm = v.copy(), v.copy()
        vp[idx] += h
        vm[idx] -= h
        fd_v[idx] = (loss(k, vp) - loss(k, vm)) / (2 * h)
    np.testing.assert_allclose(d_k, fd_k, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(d_v, fd_v, rtol=1e-6, atol=1e-8)


def test_decode_kv_history_sums():
    """Summed over the history, d_k vanishes (each head's d_scores sum to 0)
    and d_v is the sum of the group's d_out (each head's probabilities sum to
    1)."""
    rng = np.random.default_rng(4)
    N, hist, n_kv, n_heads, D = 3, 9, 2, 8, 5
    k = rng.standard_normal((N, hist, n_kv, D))
    v = rng.standard_normal((N, hist, n_kv, D))
    q = rng.standard_normal((N, n_heads, D))
    d_out = rng.standard_normal((N, n_heads, D))
    probs = Dec.softmax_rows(rng.standard_normal((N, n_heads, hist)))
    d_scores, _ = Dec.decode_backward(k, v, probs, d_out)
    d_k, d_v = Dec.decode_backward_kv(q, probs, d_out, d_scores, n_kv)
    np.testing.assert_allclose(d_k.sum(axis=1), 0.0, atol=1e-12)
    G = n_heads // n_kv
    want = d_out.reshape(N, n_kv, G, D).sum(axis=2)
    np.testing.assert_allclose(d_v.sum(axis=1), want, rtol=1e-12, atol=1e-12)


def test_decode_one_hot_and_delta():
    rng = np.random.default_rng(1)
    N, hist, n_kv, n_heads, D = 1, 8, 1, 3, 5
    k = rng.standard_normal((N, hist, n_kv, D))
    v = rng.standard_normal((N, hist, n_kv, D))
    d_out = rng.standard_normal((N, n_heads, D))
    probs = np.zeros((N, n_heads, hist))
    probs[0, :, 3] = 1.0
    ds, dq = Dec.decode_backward(k, v, probs, d_out)
    assert np.max(np.abs(ds)) < 1e-14 and np.max(np.abs(dq)) < 1e-14
    probs = Dec.softmax_rows(rng.standard_normal((N, n_heads, hist)))
    ds, dq = Dec.decode_backward(k, v, probs, d_out)
    # sum_j d_scores_j = 0 and sum_pd = d_out . O with O = probs @ v (Delta)
    assert np.max(np.abs(ds.sum(axis=-1))) < 1e-14
    for h in range(n_heads):
        O = probs[0, h] @ v[0, :, 0]
        dp = v[0, :, 0] @ d_out[0, h]
        assert abs(probs[0, h] @ dp - d_out[0, h] @ O) < 1e-13


def test_decode_is_single_query_special_case():
    # page 3 == page 2 with Sq = 1, scale = 1 and probabilities given
    rng = np.random.default_rng(2)
    hist, D, n_heads = 7, 4, 2
    p = W.AttnProblem(1, n_heads, 1, 1, hist, D, scale=1.0)
    Q = rng.standard_normal((1, n_heads, 1, D))
    K = rng.standard_normal((1, 1, hist, D))
    V = rng.standard_normal((1, 1, hist, D))
    dO = rng.standard_normal((1, n_heads, 1, D))
    O, LSE = A.forward(p, Q, K, V)
    dQ, dK, dV, parts = A.backward(p, Q, K, V, O, dO, LSE, return_parts=True)
    probs = np.stack([parts[(0, h)]["P"][0] for h in range(n_heads)])[None]
    ds, dq = Dec.decode_backward(K.transpose(0, 2, 1, 3), V.transpose(0, 2, 1, 3), probs,
                                 dO[:, :, 0, :])
    np.testing.assert_allclose(dq[0], dQ[0, :, 0, :], rtol=1e-12, atol=1e-14)
    for h in range(n_heads):
        np.testing.assert_allclose(ds[0, h], parts[(0, h)]["dS"][0], rtol=1e-12, atol=1e-14)
