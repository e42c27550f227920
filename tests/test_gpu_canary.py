"""Output canaries: every buffer a call writes sits between guard zones of
poisoned bytes, and the guards must come back untouched.

Covers the outputs of the forward layer (group ids, the workspace holding the
index and the partials, O, LSE), the dense comparator, the index built into
caller buffers with no workspace, top-2 membership, and the backward (dQ, dK,
dV).  Sizes are ragged (n not a multiple of the 128-row tiles) so that tail
tiles run; a write past the end of any buffer, or before its start, changes a
guard byte.  This is the bounds check that the sanitizer would otherwise give.
"""
import numpy as np
import pytest

from learned_group_sparse_focus_gb300 import synth
from _helpers import to_dev, margin_filtered, margin_filtered_topk

GUARD = 4096          # bytes on each side (keeps 256-byte alignment)
POISON = 0xA5


@pytest.fixture(scope="module")
def fz():
    from learned_group_sparse_focus_gb300 import focus
    return focus


class Guarded:
    """A device buffer of `shape` x `dtype` between two poisoned guard zones."""

    def __init__(self, shape, dtype, fill=None):
        import torch
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), POISON, dtype=torch.uint8, device="cuda")
        self.n = n
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(*shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self) -> bool:
        import torch
        torch.cuda.synchronize()
        lo = self.raw[:GUARD].cpu().numpy()
        hi = self.raw[GUARD + self.n:].cpu().numpy()
        return bool((lo == POISON).all() and (hi == POISON).all())


def _guarded_ws(fz, nbytes):
    import torch
    ws = Guarded((nbytes,), torch.uint8)
    fz.focus_workspace_init(ws.t)
    return ws


@pytest.mark.gpu
@pytest.mark.parametrize("n,H,H_kv,A,K,w,d", [(1000, 4, 2, 1, 8, 64, 128), (777, 4, 4, 4, 5, 100, 64)])
def test_forward_layer_writes_stay_inside_their_buffers(fz, n, H, H_kv, A, K, w, d):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    wl = synth.Workload("t", B=2, H=H, H_kv=H_kv, n=n, d=d, D=256, d_g=64, K=K, w=w, A=A, dtype="bf16",
                        groups="uniform", seed=900 + n)
    x = margin_filtered(wl)
    p = fz.params_from_workload(wl)
    ws = _guarded_ws(fz, fz.focus_workspace_bytes(p))
    h, W, C, Q, Kt, V = (to_dev(x[k], "bf16") for k in ("h", "W", "C", "Q", "K", "V"))
    gid = Guarded((wl.B, A, n), torch.int32)
    O = Guarded(tuple(Q.shape), torch.bfloat16)
    lse = Guarded((wl.B, H, n), torch.float32)
    fz.focus_assign(p, h, W, C, gid.t, ws.t)
    idx = fz.focus_build_index(p, gid.t, ws.t)
    fz.focus_attention_fwd(p, Q, Kt, V, idx, O.t, lse.t, ws.t)
    assert fz.focus_check_errors(ws.t) == 0
    assert np.array_equal(gid.t.cpu().numpy(), x["gid_ref"])
    for name, g in (("gid", gid), ("workspace", ws), ("O", O), ("lse", lse)):
        assert g.intact(), name
    # the dense comparator and the two-call comparator into the same guarded O
    fz.focus_dense_causal_fwd(p, Q, Kt, V, O.t, lse.t, ws.t)
    fz.focus_attention_two_call_fwd(p, Q, Kt, V, idx, O.t, None, ws.t)
    assert fz.focus_check_errors(ws.t) == 0
    for name, g in (("workspace", ws), ("O", O), ("lse", lse)):
        assert g.intact(), name


@pytest.mark.gpu
def test_static_index_writes_stay_inside_caller_buffers(fz):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    n, K = 1500, 9
    p = fz.make_params(B=2, H=1, H_kv=1, n=n, d=64, D=64, d_g=32, K=K, A=1, w=40)
    ref_bufs = fz.index_buffers(p)
    bufs = {k: Guarded(tuple(v.shape), v.dtype) for k, v in ref_bufs.items()}
    bufs["err"].t.zero_()
    gid = torch.from_numpy(synth.draw_group_ids(5, 2, 1, n, K, "zipf")).cuda()
    fz.focus_build_index_static(p, gid, {k: g.t for k, g in bufs.items()})
    assert fz.focus_check_errors(bufs["err"].t) == 0
    for name, g in bufs.items():
        assert g.intact(), name


@pytest.mark.gpu
def test_top2_writes_stay_inside_their_buffers(fz):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    wl = synth.Workload("t", B=1, H=4, H_kv=2, n=900, d=128, D=128, d_g=64, K=6, w=50, A=1, dtype="bf16",
                        groups="uniform", seed=31)
    x = margin_filtered_topk(wl, 2)
    p = fz.params_from_workload(wl)
    import ctypes
    nbytes = fz.focus_workspace_bytes_topk(p, 2)
    ws = Guarded((nbytes,), torch.uint8)
    fz.focus_workspace_init(ws.t)
    h, W, C, Q, Kt, V = (to_dev(x[k], "bf16") for k in ("h", "W", "C", "Q", "K", "V"))
    gid = Guarded((1, 1, wl.n, 2), torch.int32)
    O = Guarded(tuple(Q.shape), torch.bfloat16)
    lse = Guarded((1, wl.H, wl.n), torch.float32)
    fz.focus_assign_topk(p, 2, h, W, C, gid.t, ws.t)
    idx = fz.focus_build_index_topk(p, 2, gid.t, ws.t)
    fz.focus_attention_topk_fwd(p, Q, Kt, V, idx, O.t, lse.t, ws.t)
    assert fz.focus_check_errors(ws.t) == 0
    for name, g in (("gid", gid), ("workspace", ws), ("O", O), ("lse", lse)):
        assert g.intact(), name


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_writes_stay_inside_their_buffers(fz, dtype):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    wl = synth.Workload("t", B=1, H=4, H_kv=2, n=600, d=64, D=64, d_g=32, K=5, w=40, A=1, dtype=dtype,
                        groups="uniform", seed=57)
    x = synth.draw(wl, parts=("attn",))
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace(p)
    Q, Kt, V = (to_dev(x[k], dtype) for k in ("Q", "K", "V"))
    gid = torch.from_numpy(synth.draw_group_ids(9, 1, 1, wl.n, wl.K, "uniform")).cuda()
    idx = fz.focus_build_index(p, gid, ws)
    O = torch.empty_like(Q)
    lse = torch.empty((1, wl.H, wl.n), dtype=torch.float32, device="cuda")
    fz.focus_attention_fwd(p, Q, Kt, V, idx, O, lse, ws)
    dO = to_dev(np.random.default_rng(3).standard_normal(x["Q"].shape).astype(np.float32), dtype)
    wsb = Guarded((int(fz.lib().focus_backward_workspace_bytes(__import__("ctypes").byref(p))),), torch.uint8)
    fz.focus_workspace_init(wsb.t)
    dQ = Guarded(tuple(Q.shape), Q.dtype)
    dK = Guarded(tuple(Kt.shape), Kt.dtype)
    dV = Guarded(tuple(V.shape), V.dtype)
    fz.focus_attention_bwd(p, Q, Kt, V, O, dO, lse, idx, dQ.t, dK.t, dV.t, wsb.t)
    assert fz.focus_check_errors(wsb.t) == 0
    for name, g in (("workspace", wsb), ("dQ", dQ), ("dK", dK), ("dV", dV)):
        assert g.intact(), name
