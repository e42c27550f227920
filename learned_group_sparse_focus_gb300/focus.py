"""Python binding of libfocus.so (the Focus C ABI declared in include/focus.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  PyTorch provides device memory and streams.  If the compiled
library is missing, importing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libfocus.so")

F32, BF16 = 0, 1
TILE_M = 128
TILE_N = 128

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small",
          4: "CUDA error", 5: "device wait timed out", 6: "group id outside [0, K)"}


class FocusError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({status})")
        self.status = status


class Params(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int32) for k in ("B", "H", "H_kv", "n", "d", "D", "d_g", "K", "A", "w")] + \
               [("scale", ctypes.c_float), ("dtype", ctypes.c_int32)]


class Item(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int32) for k in ("b", "a", "g", "row0", "rows", "keys", "key0", "pad")]


class Index(ctypes.Structure):
    _fields_ = [("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p), ("perm", ctypes.c_void_p),
                ("rank", ctypes.c_void_p), ("farlen_tok", ctypes.c_void_p),
                ("farlen_slot", ctypes.c_void_p), ("items", ctypes.c_void_p),
                ("order", ctypes.c_void_p), ("n_items", ctypes.c_void_p),
                ("max_items", ctypes.c_int32), ("w_eff", ctypes.c_int32)]


class IndexTopk(ctypes.Structure):
    _fields_ = [("entry", Index), ("pair", Index), ("pair_gid", ctypes.c_void_p),
                ("far_tok", ctypes.c_void_p), ("k", ctypes.c_int32), ("split", ctypes.c_int32),
                ("farlen_sub", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libfocus.so not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, P = ctypes.c_void_p, ctypes.POINTER(Params)
    sig = {
        "focus_abi_version": ([], ctypes.c_int32),
        "focus_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "focus_workspace_bytes": ([P], ctypes.c_size_t),
        "focus_workspace_init": ([vp, vp], ctypes.c_int),
        "focus_assign": ([P, vp, vp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "focus_build_index": ([P, vp, ctypes.POINTER(Index), vp, ctypes.c_size_t, vp], ctypes.c_int),
        "focus_attention_fwd": ([P, vp, vp, vp, ctypes.POINTER(Index), vp, vp, vp, ctypes.c_size_t, vp],
                                ctypes.c_int),
        "focus_attention_fwd_timed": ([P, vp, vp, vp, ctypes.POINTER(Index), vp, vp, vp, ctypes.c_size_t,
                                       vp, ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
        "focus_dense_causal_fwd": ([P, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "focus_test_attention_wait_limit": ([P, vp, vp, vp, vp, vp, ctypes.c_size_t, ctypes.c_uint64, vp],
                                            ctypes.c_int),
        "focus_sinkhorn_workspace_bytes": ([P], ctypes.c_size_t),
        "focus_assign_scores": ([P, vp, vp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "focus_sinkhorn_fwd": ([P, ctypes.c_int32, ctypes.c_float, vp, vp, vp, ctypes.c_size_t, vp],
                               ctypes.c_int),
        "focus_backward_workspace_bytes": ([P], ctypes.c_size_t),
        "focus_attention_bwd": ([P, vp, vp, vp, vp, vp, vp, ctypes.POINTER(Index), vp, vp, vp, vp,
                                 ctypes.c_size_t, vp], ctypes.c_int),
        "focus_attention_two_call_fwd": ([P, vp, vp, vp, ctypes.POINTER(Index), vp, vp, vp, ctypes.c_size_t,
                                          vp], ctypes.c_int),
        "focus_layer_fwd_host": ([P] + [vp] * 7 + [vp] * 8 + [vp, ctypes.c_size_t, vp], ctypes.c_int),
        "focus_check_errors": ([vp, vp], ctypes.c_int),
        "focus_build_index_static": ([P, vp, ctypes.POINTER(Index), vp, vp], ctypes.c_int),
        "focus_workspace_bytes_topk": ([P, ctypes.c_int32], ctypes.c_size_t),
        "focus_assign_topk": ([P, ctypes.c_int32, vp, vp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "focus_build_index_topk": ([P, ctypes.c_int32, vp, ctypes.POINTER(IndexTopk), vp, ctypes.c_size_t,
                                    vp], ctypes.c_int),
        "focus_attention_topk_fwd": ([P, vp, vp, vp, ctypes.POINTER(IndexTopk), vp, vp, vp, ctypes.c_size_t,
                                      vp], ctypes.c_int),
        "focus_attention_topk_fwd_timed": ([P, vp, vp, vp, ctypes.POINTER(IndexTopk), vp, vp, vp,
                                            ctypes.c_size_t, vp, ctypes.POINTER(ctypes.c_void_p)],
                                           ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib = _load()

EXPORTED = ("focus_abi_version", "focus_status_string", "focus_workspace_bytes",
            "focus_workspace_init", "focus_assign", "focus_build_index", "focus_attention_fwd",
            "focus_attention_fwd_timed", "focus_dense_causal_fwd", "focus_layer_fwd_host", "focus_check_errors",
            "focus_build_index_static", "focus_workspace_bytes_topk", "focus_assign_topk",
            "focus_build_index_topk", "focus_attention_topk_fwd", "focus_attention_topk_fwd_timed",
            "focus_attention_two_call_fwd", "focus_sinkhorn_workspace_bytes", "focus_assign_scores",
            "focus_sinkhorn_fwd", "focus_backward_workspace_bytes", "focus_attention_bwd",
            "focus_test_attention_wait_limit")


def lib():
    return _lib


def make_params(B, H, H_kv, n, d, D, d_g, K, A, w, scale=None, dtype=BF16) -> Params:
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    if isinstance(dtype, str):
        dtype = BF16 if dtype == "bf16" else F32
    return Params(B, H, H_kv, n, d, D, d_g, K, A, w, float(scale), int(dtype))


def params_from_workload(wl, **override) -> Params:
    f = dict(B=wl.B, H=wl.H, H_kv=wl.H_kv, n=wl.n, d=wl.d, D=wl.D, d_g=wl.d_g, K=wl.K, A=wl.A,
             w=wl.w, scale=wl.scale, dtype=wl.dtype)
    f.update(override)
    return make_params(**f)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return t.data_ptr()
    return int(t)


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn: str, st: int):
    if st != 0:
        raise FocusError(fn, st)


def focus_workspace_bytes(p: Params) -> int:
    return int(_lib.focus_workspace_bytes(ctypes.byref(p)))


def alloc_workspace(p: Params, device="cuda", stream=None) -> torch.Tensor:
    """Caller-owned workspace (a uint8 device tensor), error word cleared."""
    nbytes = focus_workspace_bytes(p)
    if nbytes == 0:
        raise FocusError("focus_workspace_bytes", 1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    focus_workspace_init(ws, stream)
    return ws


def focus_workspace_init(ws, stream=None):
    _check("focus_workspace_init", _lib.focus_workspace_init(_ptr(ws), _stream(stream)))


def focus_assign(p: Params, h, W, C, gid, ws, stream=None):
    _check("focus_assign", _lib.focus_assign(ctypes.byref(p), _ptr(h), _ptr(W), _ptr(C), _ptr(gid),
                                             _ptr(ws), ws.numel(), _stream(stream)))


def focus_build_index(p: Params, gid, ws, stream=None) -> Index:
    idx = Index()
    _check("focus_build_index", _lib.focus_build_index(ctypes.byref(p), _ptr(gid), ctypes.byref(idx),
                                                       _ptr(ws), ws.numel(), _stream(stream)))
    return idx


def focus_attention_fwd(p: Params, Q, K, V, idx: Index, O, lse, ws, stream=None):
    _check("focus_attention_fwd",
           _lib.focus_attention_fwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), ctypes.byref(idx),
                                    _ptr(O), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))


def focus_attention_fwd_timed(p: Params, Q, K, V, idx: Index, O, lse, ws, events, stream=None):
    """events: four recorded-once torch.cuda.Event objects (see include/focus.h)."""
    arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
    _check("focus_attention_fwd_timed",
           _lib.focus_attention_fwd_timed(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), ctypes.byref(idx),
                                          _ptr(O), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream), arr))


def focus_attention_two_call_fwd(p: Params, Q, K, V, idx: Index, O, lse, ws, stream=None):
    """The two-call comparator (group call, window call, separate combine)."""
    _check("focus_attention_two_call_fwd",
           _lib.focus_attention_two_call_fwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), ctypes.byref(idx),
                                             _ptr(O), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))


def focus_dense_causal_fwd(p: Params, Q, K, V, O, lse, ws, stream=None):
    _check("focus_dense_causal_fwd",
           _lib.focus_dense_causal_fwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse),
                                       _ptr(ws), ws.numel(), _stream(stream)))


def focus_test_attention_wait_limit(p: Params, Q, K, V, O, ws, wait_ns: int, stream=None):
    """Test hook: the dense kernel with its first Q tile withheld and every
    device wait limited to wait_ns; the device error word then holds the
    timeout bit (read it with focus_check_errors)."""
    _check("focus_test_attention_wait_limit",
           _lib.focus_test_attention_wait_limit(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(ws),
                                                ws.numel(), int(wait_ns), _stream(stream)))


def focus_layer_fwd_host(p: Params, host: dict, dev: dict, ws, stream=None):
    """host: pinned CPU tensors h, W, C, Q, K, V, O; dev: device tensors of the same
    names plus gid.  Enqueues H2D copies, the three steps and the D2H copy of O."""
    _check("focus_layer_fwd_host", _lib.focus_layer_fwd_host(
        ctypes.byref(p), *[_ptr(host[k]) for k in ("h", "W", "C", "Q", "K", "V", "O")],
        *[_ptr(dev[k]) for k in ("h", "W", "C", "Q", "K", "V", "O", "gid")],
        _ptr(ws), ws.numel(), _stream(stream)))


def focus_check_errors(ws, stream=None) -> int:
    """Synchronise the stream; return (and clear) the device error status."""
    return int(_lib.focus_check_errors(_ptr(ws), _stream(stream)))


def index_buffers(p: Params, device="cuda") -> dict:
    """Caller-owned output buffers for focus_build_index_static, sized as the
    index arrays of focus_build_index, plus a zeroed 256-byte error word."""
    P, n, K = p.B * p.A, p.n, p.K
    m = P * ((n + TILE_M - 1) // TILE_M + min(K, n))
    z = lambda *shape: torch.empty(shape, dtype=torch.int32, device=device)
    return dict(counts=z(p.B, p.A, K), offsets=z(p.B, p.A, K + 1), perm=z(p.B, p.A, n),
                rank=z(p.B, p.A, n), farlen_tok=z(p.B, p.A, n), farlen_slot=z(p.B, p.A, n),
                items=z(m, 8), order=z(m), n_items=z(1),
                err=torch.zeros(64, dtype=torch.int32, device=device))


def focus_build_index_static(p: Params, gid, bufs: dict, stream=None) -> Index:
    """focus_build_index into the caller-owned buffers of index_buffers(); the
    sort's scratch is the library's fixed device array (no workspace)."""
    idx = Index()
    for name in ("counts", "offsets", "perm", "rank", "farlen_tok", "farlen_slot", "items", "order",
                 "n_items"):
        setattr(idx, name, _ptr(bufs[name]))
    idx.max_items = bufs["order"].numel()
    _check("focus_build_index_static",
           _lib.focus_build_index_static(ctypes.byref(p), _ptr(gid), ctypes.byref(idx), _ptr(bufs["err"]),
                                         _stream(stream)))
    return idx


# ------------------------------------------------------- top-k membership ---

def focus_workspace_bytes_topk(p: Params, k: int) -> int:
    return int(_lib.focus_workspace_bytes_topk(ctypes.byref(p), int(k)))


def alloc_workspace_topk(p: Params, k: int, device="cuda", stream=None) -> torch.Tensor:
    """Caller-owned workspace for the top-k calls, error word cleared."""
    nbytes = focus_workspace_bytes_topk(p, k)
    if nbytes == 0:
        raise FocusError("focus_workspace_bytes_topk", 1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    focus_workspace_init(ws, stream)
    return ws


def focus_assign_topk(p: Params, k: int, h, W, C, gid, ws, stream=None):
    """gid: [B, A, n, k] int32 device tensor (best first)."""
    _check("focus_assign_topk", _lib.focus_assign_topk(ctypes.byref(p), int(k), _ptr(h), _ptr(W), _ptr(C),
                                                       _ptr(gid), _ptr(ws), ws.numel(), _stream(stream)))


def focus_build_index_topk(p: Params, k: int, gid, ws, stream=None) -> IndexTopk:
    idx = IndexTopk()
    _check("focus_build_index_topk",
           _lib.focus_build_index_topk(ctypes.byref(p), int(k), _ptr(gid), ctypes.byref(idx), _ptr(ws),
                                       ws.numel(), _stream(stream)))
    return idx


def focus_attention_topk_fwd(p: Params, Q, K, V, idx: IndexTopk, O, lse, ws, stream=None):
    _check("focus_attention_topk_fwd",
           _lib.focus_attention_topk_fwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), ctypes.byref(idx),
                                         _ptr(O), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))


def focus_attention_topk_fwd_timed(p: Params, Q, K, V, idx: IndexTopk, O, lse, ws, events, stream=None):
    """events: five torch.cuda.Event objects (see include/focus.h)."""
    arr = (ctypes.c_void_p * 5)(*[e.cuda_event for e in events])
    _check("focus_attention_topk_fwd_timed",
           _lib.focus_attention_topk_fwd_timed(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), ctypes.byref(idx),
                                               _ptr(O), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream),
                                               arr))


def run_layer_topk(p: Params, k: int, h, W, C, Q, K, V, ws, stream=None, want_lse=False):
    """assign (top-k) -> index -> attention; returns (O, gid, idx, lse)."""
    dev = Q.device
    gid = torch.empty((p.B, p.A, p.n, k), dtype=torch.int32, device=dev)
    focus_assign_topk(p, k, h, W, C, gid, ws, stream)
    idx = focus_build_index_topk(p, k, gid, ws, stream)
    O = torch.empty_like(Q)
    lse = torch.empty((p.B, p.H, p.n), dtype=torch.float32, device=dev) if want_lse else None
    focus_attention_topk_fwd(p, Q, K, V, idx, O, lse, ws, stream)
    return O, gid, idx, lse


# ---------------------------------------------------------------- backward ---

def alloc_workspace_backward(p: Params, device="cuda", stream=None) -> torch.Tensor:
    nbytes = int(_lib.focus_backward_workspace_bytes(ctypes.byref(p)))
    if nbytes == 0:
        raise FocusError("focus_backward_workspace_bytes", 1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    focus_workspace_init(ws, stream)
    return ws


def focus_attention_bwd(p: Params, Q, K, V, O, dO, lse, idx: Index, dQ, dK, dV, ws, stream=None):
    """Gradients over the kept pairs; lse from the forward call, idx from
    focus_build_index (forward workspace), ws a backward workspace."""
    _check("focus_attention_bwd",
           _lib.focus_attention_bwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(lse),
                                    ctypes.byref(idx), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(),
                                    _stream(stream)))


# ------------------------------------------------ Sinkhorn soft assignment ---

def alloc_workspace_sinkhorn(p: Params, device="cuda", stream=None) -> torch.Tensor:
    nbytes = int(_lib.focus_sinkhorn_workspace_bytes(ctypes.byref(p)))
    if nbytes == 0:
        raise FocusError("focus_sinkhorn_workspace_bytes", 1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    focus_workspace_init(ws, stream)
    return ws


def focus_assign_scores(p: Params, h, W, C, S, ws, stream=None):
    """S: [B, A, n, K] fp32 device tensor."""
    _check("focus_assign_scores", _lib.focus_assign_scores(ctypes.byref(p), _ptr(h), _ptr(W), _ptr(C), _ptr(S),
                                                           _ptr(ws), ws.numel(), _stream(stream)))


def focus_sinkhorn_fwd(p: Params, iters: int, tau: float, S, G, ws, stream=None):
    """G (may be S): [B, A, n, K] fp32 soft assignment after `iters` rounds."""
    _check("focus_sinkhorn_fwd", _lib.focus_sinkhorn_fwd(ctypes.byref(p), int(iters), float(tau), _ptr(S),
                                                         _ptr(G), _ptr(ws), ws.numel(), _stream(stream)))


# ------------------------------------------------------------ index views ---

def index_views(p: Params, idx: Index, ws: torch.Tensor, n: int | None = None,
                K: int | None = None) -> dict:
    """Torch views (no copy) of the index arrays living inside the workspace.
    n: sorted items per (b, a) (p.n; n * k for a top-k entry index); K: groups
    (p.K; K (K - 1) / 2 for a top-2 pair index)."""
    base = ws.data_ptr()
    P = p.B * p.A
    n = p.n if n is None else n
    K = p.K if K is None else K

    def view(ptr, count, dtype=torch.int32, shape=None):
        off = ptr - base
        t = ws[off:off + count * 4].view(dtype)
        return t.view(*shape) if shape else t

    out = dict(counts=view(idx.counts, P * K, shape=(p.B, p.A, K)),
               offsets=view(idx.offsets, P * (K + 1), shape=(p.B, p.A, K + 1)),
               perm=view(idx.perm, P * n, shape=(p.B, p.A, n)),
               rank=view(idx.rank, P * n, shape=(p.B, p.A, n)),
               farlen_tok=view(idx.farlen_tok, P * n, shape=(p.B, p.A, n)),
               farlen_slot=view(idx.farlen_slot, P * n, shape=(p.B, p.A, n)),
               n_items=view(idx.n_items, 1))
    m = idx.max_items
    out["items"] = view(idx.items, m * 8, shape=(m, 8))
    out["order"] = view(idx.order, m)
    return out


def run_layer(p: Params, h, W, C, Q, K, V, ws, stream=None, want_lse=False):
    """assign -> index -> attention on device tensors; returns (O, gid, idx, lse)."""
    dev = Q.device
    gid = torch.empty((p.B, p.A, p.n), dtype=torch.int32, device=dev)
    focus_assign(p, h, W, C, gid, ws, stream)
    idx = focus_build_index(p, gid, ws, stream)
    O = torch.empty_like(Q)
    lse = torch.empty((p.B, p.H, p.n), dtype=torch.float32, device=dev) if want_lse else None
    focus_attention_fwd(p, Q, K, V, idx, O, lse, ws, stream)
    return O, gid, idx, lse
