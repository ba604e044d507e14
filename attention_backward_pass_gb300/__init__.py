"""GB300 (sm_103a) attention backward pass: Python binding of the C ABI.

The compute lives in ``_lib/libattnbwd.so`` (hand-written CUDA: TMA +
tcgen05/TMEM tile kernel, Delta/LSE preprocessing, decode backward).  This
module only marshals arguments: torch tensors are used for device memory and
streams, and their pointers are handed to the library's ``extern "C"`` entry
points.  There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import workloads  # noqa: F401  (seeded synthetic inputs; no arithmetic)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libattnbwd.so")

ATTN_OK = 0
ATTN_ERR_TIMEOUT = -4
STATUS_NAMES = {0: "ok", -1: "invalid argument", -2: "unsupported configuration",
                -3: "CUDA error", -4: "device wait timed out", -5: "workspace problem",
                -6: "problem exceeds the fixed no-allocation scratch array"}
ATTN_F32, ATTN_BF16 = 0, 1
ATTN_LAYOUT_BHSD, ATTN_LAYOUT_BSHD = 0, 1


class AttnError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)} ({status})")
        self.status = status


class AttnBwdParams(ctypes.Structure):
    """Mirror of ``attn_bwd_params`` in include/attn_bwd.h."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("seq_q", ctypes.c_int32),
        ("seq_k", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("scale", ctypes.c_float), ("dropout_prob", ctypes.c_float),
        ("seed", ctypes.c_uint64),
        ("causal", ctypes.c_int32), ("causal_offset", ctypes.c_int32),
        ("window", ctypes.c_int32), ("has_mask", ctypes.c_int32),
        ("mask_stride_b", ctypes.c_int64), ("mask_stride_h", ctypes.c_int64),
        ("mask_stride_q", ctypes.c_int64), ("mask_stride_k", ctypes.c_int64),
        ("layout", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("deterministic", ctypes.c_int32),
    ]


class AttnBwdDecodeParams(ctypes.Structure):
    """Mirror of ``attn_bwd_decode_params``."""
    _fields_ = [("num_seqs", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("history_len", ctypes.c_int32)]


# exported symbols and their argument types (also used by the ABI tests)
_P = ctypes.c_void_p
_SIGS = {
    "attn_bwd_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(AttnBwdParams)]),
    "attn_bwd": (ctypes.c_int, [ctypes.POINTER(AttnBwdParams), _P, _P, _P, _P, _P, _P, _P, _P,
                                _P, _P, _P, ctypes.c_size_t, _P]),
    "attn_bwd_prepare": (ctypes.c_int, [ctypes.POINTER(AttnBwdParams), _P, _P, _P, _P, _P, _P, _P,
                                        ctypes.c_size_t, _P]),
    "attn_bwd_tiles": (ctypes.c_int, [ctypes.POINTER(AttnBwdParams), _P, _P, _P, _P, _P, _P, _P,
                                      _P, _P, ctypes.c_size_t, _P]),
    "attn_bwd_finish": (ctypes.c_int, [ctypes.POINTER(AttnBwdParams), _P, _P, ctypes.c_size_t,
                                       _P]),
    "attn_bwd_lse": (ctypes.c_int, [ctypes.POINTER(AttnBwdParams), _P, _P, _P, _P, _P]),
    "attn_fwd_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(AttnBwdParams)]),
    "attn_fwd": (ctypes.c_int, [ctypes.POINTER(AttnBwdParams), _P, _P, _P, _P, _P, _P, _P,
                                ctypes.c_size_t, _P]),
    "attn_bwd_decode_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(AttnBwdDecodeParams)]),
    "attn_bwd_decode": (ctypes.c_int, [ctypes.POINTER(AttnBwdDecodeParams), _P, _P, _P, _P, _P,
                                       _P, _P, ctypes.c_size_t, _P]),
    "attn_bwd_decode_noalloc": (ctypes.c_int, [ctypes.POINTER(AttnBwdDecodeParams), _P, _P, _P,
                                               _P, _P, _P, _P]),
    "attn_bwd_decode_kv": (ctypes.c_int, [ctypes.POINTER(AttnBwdDecodeParams), _P, _P, _P, _P,
                                          _P, _P, _P]),
    "attn_dropout_keep_mask": (ctypes.c_int, [ctypes.POINTER(AttnBwdParams), ctypes.c_int32,
                                              ctypes.c_int32, _P, _P]),
    "attn_bwd_query_range": (ctypes.c_int, [ctypes.POINTER(AttnBwdParams), ctypes.c_int32,
                                            ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                            ctypes.POINTER(ctypes.c_int32)]),
    "attn_bwd_check_device_error": (ctypes.c_int, [ctypes.c_int32]),
    "attn_selftest_wait_timeout": (ctypes.c_int, [_P]),
    "attn_selftest_mma": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, _P, _P, _P, _P, _P]),
    "attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


def load_library(path: str = LIB_PATH):
    """Load libattnbwd.so (built by ``build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run attention_backward_pass_gb300.build() first")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def build(verbose_ptxas: bool = False) -> str:
    """Compile the CUDA sources into _lib/libattnbwd.so (nvcc, sm_103a)."""
    from .build import build as _build
    return _build(verbose_ptxas=verbose_ptxas)


def _check(fn, status):
    if status != ATTN_OK:
        raise AttnError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_params(p) -> AttnBwdParams:
    """Fill the C params struct from an ``AttnProblem``-like object."""
    return AttnBwdParams(p.batch, p.num_heads, p.num_kv_heads, p.seq_q, p.seq_k, p.head_dim,
                         float(p.scale), float(p.dropout_prob), int(p.seed) & (2**64 - 1),
                         int(p.causal), int(p.causal_offset), int(p.window), int(p.has_mask),
                         int(p.mask_stride_b), int(p.mask_stride_h), int(p.mask_stride_q),
                         int(p.mask_stride_k), int(p.layout), int(p.dtype),
                         int(getattr(p, "deterministic", 0)))


def workspace_size(p) -> int:
    lib = load_library()
    n = lib.attn_bwd_workspace_size(ctypes.byref(make_params(p)))
    if n == 0:
        raise AttnError("attn_bwd_workspace_size", -1)
    return int(n)


def alloc_workspace(p, device="cuda"):
    import torch
    # torch's caching allocator hands out 512-byte aligned blocks
    return torch.empty(workspace_size(p), dtype=torch.uint8, device=device)


def attn_bwd(p, Q, K, V, O, dO, LSE, mask, dQ, dK, dV, workspace, stream=None):
    """Enqueue the backward pass; outputs dQ, dK, dV are overwritten.
    LSE=None recomputes the row log-sum-exp first (into the workspace)."""
    lib = load_library()
    prm = make_params(p)
    st = lib.attn_bwd(ctypes.byref(prm), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE),
                      _ptr(mask), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(workspace),
                      ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                      _stream_ptr(stream))
    _check("attn_bwd", st)


def _wsb(workspace):
    return ctypes.c_size_t(workspace.numel() * workspace.element_size())


def attn_bwd_prepare(p, Q, K, O, dO, LSE, dQ, workspace, stream=None):
    """Stage 1 of attn_bwd: Delta, LSE*log2(e), dQ accumulator reset."""
    st = load_library().attn_bwd_prepare(ctypes.byref(make_params(p)), _ptr(Q), _ptr(K), _ptr(O),
                                         _ptr(dO), _ptr(LSE), _ptr(dQ), _ptr(workspace),
                                         _wsb(workspace), _stream_ptr(stream))
    _check("attn_bwd_prepare", st)


def attn_bwd_tiles(p, Q, K, V, dO, mask, dQ, dK, dV, workspace, stream=None):
    """Stage 2 of attn_bwd: the fused tcgen05 tile kernel."""
    st = load_library().attn_bwd_tiles(ctypes.byref(make_params(p)), _ptr(Q), _ptr(K), _ptr(V),
                                       _ptr(dO), _ptr(mask), _ptr(dQ), _ptr(dK), _ptr(dV),
                                       _ptr(workspace), _wsb(workspace), _stream_ptr(stream))
    _check("attn_bwd_tiles", st)


def attn_bwd_finish(p, dQ, workspace, stream=None):
    """Stage 3 of attn_bwd: bf16 dQ from the fp32 accumulator (no-op for fp32)."""
    st = load_library().attn_bwd_finish(ctypes.byref(make_params(p)), _ptr(dQ), _ptr(workspace),
                                        _wsb(workspace), _stream_ptr(stream))
    _check("attn_bwd_finish", st)


def attn_bwd_lse(p, Q, K, mask, LSE, stream=None):
    """Row log-sum-exp of the scores into LSE [B, H, Sq] (fp32, 3e38 for
    rows without a visible, non-hard key)."""
    st = load_library().attn_bwd_lse(ctypes.byref(make_params(p)), _ptr(Q), _ptr(K), _ptr(mask),
                                     _ptr(LSE), _stream_ptr(stream))
    _check("attn_bwd_lse", st)


def fwd_workspace_size(p) -> int:
    lib = load_library()
    n = lib.attn_fwd_workspace_size(ctypes.byref(make_params(p)))
    if n == 0:
        raise AttnError("attn_fwd_workspace_size", -1)
    return int(n)


def attn_fwd(p, Q, K, V, mask, O, LSE, workspace, stream=None):
    """Fused forward: O (p's layout and dtype) and LSE [B, H, Sq] (fp32)."""
    st = load_library().attn_fwd(ctypes.byref(make_params(p)), _ptr(Q), _ptr(K), _ptr(V),
                                 _ptr(mask), _ptr(O), _ptr(LSE), _ptr(workspace),
                                 _wsb(workspace), _stream_ptr(stream))
    _check("attn_fwd", st)


def kernels_per_call(p, recompute_lse: bool = False) -> int:
    """Kernels one attn_bwd call launches (the LSE sweep when no LSE is
    given, prepare, tile kernel, and the finishing kernel: bf16 dQ conversion,
    or the ordered dQ reduction when deterministic)."""
    finish = 1 if (p.dtype == ATTN_BF16 or getattr(p, "deterministic", 0)) else 0
    return (1 if recompute_lse else 0) + 1 + 1 + finish


def make_decode_params(p) -> AttnBwdDecodeParams:
    return AttnBwdDecodeParams(p.num_seqs, p.n_heads, p.n_kv_heads, p.head_dim, p.history_len)


def decode_workspace_size(p) -> int:
    lib = load_library()
    n = lib.attn_bwd_decode_workspace_size(ctypes.byref(make_decode_params(p)))
    if n == 0:
        raise AttnError("attn_bwd_decode_workspace_size", -1)
    return int(n)


def alloc_decode_workspace(p, device="cuda"):
    import torch
    return torch.empty(decode_workspace_size(p), dtype=torch.uint8, device=device)


def attn_bwd_decode(p, k_hist, v_hist, probs, d_out, d_scores, d_q, workspace, stream=None):
    lib = load_library()
    prm = make_decode_params(p)
    st = lib.attn_bwd_decode(ctypes.byref(prm), _ptr(k_hist), _ptr(v_hist), _ptr(probs),
                             _ptr(d_out), _ptr(d_scores), _ptr(d_q), _ptr(workspace),
                             ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                             _stream_ptr(stream))
    _check("attn_bwd_decode", st)


def attn_bwd_decode_noalloc(p, k_hist, v_hist, probs, d_out, d_scores, d_q, stream=None):
    """Decode backward with the library's fixed scratch array instead of a
    workspace, for callers that cannot allocate device memory."""
    st = load_library().attn_bwd_decode_noalloc(ctypes.byref(make_decode_params(p)), _ptr(k_hist),
                                                _ptr(v_hist), _ptr(probs), _ptr(d_out),
                                                _ptr(d_scores), _ptr(d_q), _stream_ptr(stream))
    _check("attn_bwd_decode_noalloc", st)


def attn_bwd_decode_kv(p, q, probs, d_out, d_scores, d_k_hist, d_v_hist, stream=None):
    """Decode backward pass 2 (gradients of k_hist and v_hist) from pass 1's
    d_scores."""
    st = load_library().attn_bwd_decode_kv(ctypes.byref(make_decode_params(p)), _ptr(q),
                                           _ptr(probs), _ptr(d_out), _ptr(d_scores),
                                           _ptr(d_k_hist), _ptr(d_v_hist), _stream_ptr(stream))
    _check("attn_bwd_decode_kv", st)


def dropout_keep_mask(p, b, h, keep, stream=None):
    lib = load_library()
    st = lib.attn_dropout_keep_mask(ctypes.byref(make_params(p)), b, h, _ptr(keep),
                                    _stream_ptr(stream))
    _check("attn_dropout_keep_mask", st)


def query_range(p, k0, k1):
    """Host-side planner: queries [begin, end) that can see a key of [k0, k1]."""
    lib = load_library()
    qb, qe = ctypes.c_int32(), ctypes.c_int32()
    st = lib.attn_bwd_query_range(ctypes.byref(make_params(p)), k0, k1, ctypes.byref(qb),
                                  ctypes.byref(qe))
    _check("attn_bwd_query_range", st)
    return qb.value, qe.value


def selftest_wait_timeout(stream=None):
    """Enqueue the failure-path self test (a wait that runs out)."""
    _check("attn_selftest_wait_timeout",
           load_library().attn_selftest_wait_timeout(_stream_ptr(stream)))


def check_device_error(clear: bool = True) -> int:
    """0 if no kernel's bounded wait ran out since the last clear."""
    return int(load_library().attn_bwd_check_device_error(1 if clear else 0))


def selftest_mma(dtype, M, N, K, a_mn, b_mn, A, B, C, dump=None, stream=None, a_tmem=False):
    lib = load_library()
    st = lib.attn_selftest_mma(dtype, M, N, K, int(a_mn), int(b_mn), int(a_tmem), _ptr(A),
                               _ptr(B), _ptr(C), _ptr(dump), _stream_ptr(stream))
    _check("attn_selftest_mma", st)
