"""C-ABI checks that need no GPU: the library loads, exports every function
include/attn_bwd.h declares, validates arguments before touching the device,
and its host-side query-range planner covers exactly the visible pairs."""
import ctypes
import os
import re

import numpy as np
import pytest

import attention_backward_pass_gb300 as ab
from attention_backward_pass_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ab.LIB_PATH):
        ab.build()
    return ab.load_library()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(attn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 8, names
    for n in names:
        assert hasattr(lib, n), n
        assert n in ab._SIGS, n


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.attn_status_string(code)


def P(**kw):
    base = dict(batch=1, num_heads=2, num_kv_heads=2, seq_q=64, seq_k=64, head_dim=64, scale=0.125)
    base.update(kw)
    return W.AttnProblem(**base)


@pytest.mark.parametrize("bad", [dict(num_heads=3, num_kv_heads=2), dict(seq_q=0),
                                 dict(dropout_prob=1.0), dict(dropout_prob=-0.1),
                                 dict(causal_offset=-1), dict(window=-2), dict(causal=2),
                                 dict(layout=5), dict(dtype=7), dict(batch=0)])
def test_invalid_params_rejected(lib, bad):
    prm = ab.make_params(P(**bad))
    assert lib.attn_bwd_workspace_size(ctypes.byref(prm)) == 0
    st = lib.attn_bwd(ctypes.byref(prm), *([None] * 10), None, 0, None)
    assert st == -1


def test_unsupported_head_dim(lib):
    prm = ab.make_params(P(head_dim=96))
    st = lib.attn_bwd(ctypes.byref(prm), *([None] * 10), None, 0, None)
    assert st == -2


def test_null_pointers_and_mask_mismatch(lib):
    prm = ab.make_params(P())
    fake = ctypes.c_void_p(4096)
    args = [fake] * 6 + [None] + [fake] * 3
    # has_mask = 0 but a mask pointer given
    args_mask = [fake] * 7 + [fake] * 3
    assert lib.attn_bwd(ctypes.byref(prm), *args_mask, fake, 1 << 30, None) == -1
    # a null tensor (O; a null LSE is legal and means "recompute it")
    args_null = [fake] * 3 + [None] + [fake] + [fake] + [None] + [fake] * 3
    assert lib.attn_bwd(ctypes.byref(prm), *args_null, fake, 1 << 30, None) == -1
    # the LSE sweep: null Q or output, mask pointer without has_mask, misaligned
    assert lib.attn_bwd_lse(ctypes.byref(prm), None, fake, None, fake, None) == -1
    assert lib.attn_bwd_lse(ctypes.byref(prm), fake, fake, None, None, None) == -1
    assert lib.attn_bwd_lse(ctypes.byref(prm), fake, fake, fake, fake, None) == -1
    assert lib.attn_bwd_lse(ctypes.byref(prm), fake, ctypes.c_void_p(4100), None, fake, None) == -1
    # attn_bwd_prepare needs the LSE
    assert lib.attn_bwd_prepare(ctypes.byref(prm), fake, fake, fake, fake, None, fake, fake,
                                1 << 30, None) == -1
    # misaligned pointer
    args_mis = [ctypes.c_void_p(4100)] + [fake] * 5 + [None] + [fake] * 3
    assert lib.attn_bwd(ctypes.byref(prm), *args_mis, fake, 1 << 30, None) == -1
    # workspace too small / misaligned
    assert lib.attn_bwd(ctypes.byref(prm), *args, fake, 16, None) == -5
    assert lib.attn_bwd(ctypes.byref(prm), *args, ctypes.c_void_p(4096 + 16), 1 << 30, None) == -5


@pytest.mark.parametrize("which", ["dQ", "dK", "dV"])
def test_misaligned_or_null_outputs_rejected(lib, which):
    """dQ, dK and dV are written with 16-byte vector and TMA stores: a
    misaligned or null output pointer is refused before anything is enqueued,
    by attn_bwd and by the tile stage alone."""
    prm = ab.make_params(P())
    fake = ctypes.c_void_p(4096)
    ws = ctypes.c_void_p(1 << 20)
    for bad in (ctypes.c_void_p(4096 + 4), None):
        outs = {"dQ": fake, "dK": fake, "dV": fake}
        outs[which] = bad
        # attn_bwd: Q, K, V, O, dO, LSE, mask, dQ, dK, dV
        assert lib.attn_bwd(ctypes.byref(prm), fake, fake, fake, fake, fake, fake, None,
                            outs["dQ"], outs["dK"], outs["dV"], ws, 1 << 30, None) == -1
        # attn_bwd_tiles: Q, K, V, dO, mask, dQ, dK, dV
        assert lib.attn_bwd_tiles(ctypes.byref(prm), fake, fake, fake, fake, None,
                                  outs["dQ"], outs["dK"], outs["dV"], ws, 1 << 30, None) == -1


def test_forward_validation(lib):
    prm = ab.make_params(P())
    fake = ctypes.c_void_p(4096)
    ws = ctypes.c_void_p(1 << 20)
    # null or misaligned tensors, mask pointer without has_mask, small workspace
    assert lib.attn_fwd(ctypes.byref(prm), None, fake, fake, None, fake, fake, ws, 1 << 30,
                        None) == -1
    assert lib.attn_fwd(ctypes.byref(prm), fake, fake, ctypes.c_void_p(4100), None, fake, fake,
                        ws, 1 << 30, None) == -1
    assert lib.attn_fwd(ctypes.byref(prm), fake, fake, fake, fake, fake, fake, ws, 1 << 30,
                        None) == -1
    assert lib.attn_fwd(ctypes.byref(prm), fake, fake, fake, None, fake, fake, ws, 16,
                        None) == -5
    # the forward needs no scratch in either dtype (fp32 reads V MN-major)
    assert ab.fwd_workspace_size(W.causal_mha()) == 256
    assert ab.fwd_workspace_size(W.gqa_window(W.DTYPE_BF16)) == 256


def test_deterministic_workspace_and_flag(lib):
    # one fp32 dQ slice per key tile (128 keys for fp32 D=64) on top of the
    # usual workspace; any flag value other than 0 / 1 is rejected
    p = W.causal_mha()
    n0 = ab.workspace_size(p)
    p.deterministic = 1
    n1 = ab.workspace_size(p)
    n_kt = (p.seq_k + 127) // 128
    assert n1 - n0 == n_kt * p.batch * p.num_heads * p.seq_q * p.head_dim * 4
    p.deterministic = 2
    assert lib.attn_bwd_workspace_size(ctypes.byref(ab.make_params(p))) == 0
    assert ab.kernels_per_call(W.causal_mha()) == 2
    p.deterministic = 1
    assert ab.kernels_per_call(p) == 3


def test_workspace_sizes(lib):
    for p in (W.tiny(), W.causal_mha(), W.gqa_window(W.DTYPE_BF16), W.masked_dropout()):
        n = ab.workspace_size(p)
        rows = p.batch * p.num_heads * ((p.seq_q + 127) // 128 * 128)
        assert n >= 2 * rows * 4 and n % 256 == 0
    dp = W.decode()
    assert ab.decode_workspace_size(dp) > 0


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("off", [0, 3, 9])
@pytest.mark.parametrize("window", [0, 1, 4])
def test_query_range_brute_force(lib, causal, off, window):
    from oracle.attention import visible
    sq, sk = 11, 13
    p = P(seq_q=sq, seq_k=sk, causal=causal, causal_offset=off, window=window)
    vis = visible(sq, sk, causal, off, window)
    for k0 in range(sk):
        for k1 in range(k0, sk):
            qb, qe = ab.query_range(p, k0, k1)
            rows = np.nonzero(vis[:, k0:k1 + 1].any(axis=1))[0]
            if rows.size == 0:
                assert qe <= qb or not vis[qb:qe, k0:k1 + 1].any()
            else:
                # covers every query that sees a key of the tile, and the
                # range ends are tight
                assert qb <= rows.min() and qe >= rows.max() + 1
                assert qb == rows.min() and qe == rows.max() + 1


def test_decode_validation(lib):
    for bad in (W.DecodeProblem(1, 3, 2, 64, 10), W.DecodeProblem(1, 8, 1, 96, 10),
                W.DecodeProblem(0, 8, 1, 64, 10), W.DecodeProblem(1, 64, 2, 64, 10)):
        prm = ab.make_decode_params(bad)
        assert lib.attn_bwd_decode_workspace_size(ctypes.byref(prm)) == 0
