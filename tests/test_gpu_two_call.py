"""GPU parity for the two-call comparator (focus_attention_two_call_fwd): an
in-group causal call, a standalone sliding-window call and a separate
log-sum-exp combine, the way the pages run Focus.  Same operation as
focus_attention_fwd, so the same oracle and tolerances apply; it is also
compared with the fused path on the benchmark shape.
"""
import os

import numpy as np
import pytest

import oracle.focus_ref as ref
from learned_group_sparse_focus_gb300 import synth

from _helpers import assert_close, assert_lse_close, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fz():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from learned_group_sparse_focus_gb300 import _build
    if not os.path.exists(_build.LIB):
        _build.build()
    from learned_group_sparse_focus_gb300 import focus
    return focus


@pytest.mark.parametrize("dtype,B,H,H_kv,A,n,d,K,w,kind", [
    ("bf16", 1, 2, 2, 1, 300, 128, 4, 32, "uniform"),
    ("bf16", 2, 4, 2, 1, 513, 64, 8, 100, "zipf"),
    ("bf16", 1, 4, 2, 2, 1000, 128, 16, 128, "uniform"),
    ("bf16", 1, 2, 1, 1, 700, 128, 1, 40, "one"),          # every row has far keys
    ("bf16", 1, 1, 1, 1, 384, 64, 384, 1, "distinct"),     # no row has far keys
    ("bf16", 1, 2, 2, 1, 1, 128, 3, 5, "uniform"),          # one token
    ("bf16", 1, 2, 2, 1, 600, 64, 6, 1000, "uniform"),      # w > n
    ("f32", 1, 2, 2, 1, 256, 64, 4, 32, "uniform"),
    ("f32", 1, 4, 2, 2, 333, 128, 5, 20, "zipf"),
])
def test_two_call_all_rows(fz, dtype, B, H, H_kv, A, n, d, K, w, kind):
    import torch
    seed = n + w + K + 1
    rng = np.random.default_rng(seed)
    store = (lambda a: synth.round_bf16(a)) if dtype == "bf16" else (lambda a: a)
    Q = store(rng.standard_normal((B, H, n, d)).astype(np.float32))
    Kt = store(rng.standard_normal((B, H_kv, n, d)).astype(np.float32))
    V = store(rng.standard_normal((B, H_kv, n, d)).astype(np.float32))
    g = synth.draw_group_ids(seed, B, A, n, K, kind)
    p = fz.make_params(B=B, H=H, H_kv=H_kv, n=n, d=d, D=64, d_g=32, K=K, A=A, w=w, dtype=dtype)
    ws = fz.alloc_workspace(p)
    idx = fz.focus_build_index(p, torch.from_numpy(g).cuda(), ws)
    Qd, Kd, Vd = to_dev(Q, dtype), to_dev(Kt, dtype), to_dev(V, dtype)
    O = torch.full_like(Qd, float("nan"))
    lse = torch.full((B, H, n), float("nan"), dtype=torch.float32, device="cuda")
    fz.focus_attention_two_call_fwd(p, Qd, Kd, Vd, idx, O, lse, ws)
    assert fz.focus_check_errors(ws) == 0
    want_O, want_L = ref.attention(Q, Kt, V, g, w, p.scale, A)
    assert_close(to_host(O), want_O, dtype, "O")
    assert_lse_close(lse.cpu().numpy(), want_L, dtype, "lse")
    # the same call without the optional LSE output
    O2 = torch.empty_like(Qd)
    fz.focus_attention_two_call_fwd(p, Qd, Kd, Vd, idx, O2, None, ws)
    assert fz.focus_check_errors(ws) == 0
    assert torch.equal(O, O2)


def test_two_call_matches_fused_at_benchmark_size(fz):
    """The 32K GQA layer: both orders of merging agree to bf16 rounding on
    every element, and the fused result is checked against the oracle by the
    full-size workload test."""
    import torch
    wl = synth.WORKLOADS["gqa_32k"]
    x = synth.draw(wl, parts=("attn",))
    g = synth.draw_group_ids(wl.seed, wl.B, wl.A, wl.n, wl.K, "zipf")
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace(p)
    idx = fz.focus_build_index(p, torch.from_numpy(g).cuda(), ws)
    Qd, Kd, Vd = (to_dev(x[k], "bf16") for k in ("Q", "K", "V"))
    O1, O2 = torch.empty_like(Qd), torch.empty_like(Qd)
    l1 = torch.empty((wl.B, wl.H, wl.n), dtype=torch.float32, device="cuda")
    l2 = torch.empty_like(l1)
    fz.focus_attention_fwd(p, Qd, Kd, Vd, idx, O1, l1, ws)
    fz.focus_attention_two_call_fwd(p, Qd, Kd, Vd, idx, O2, l2, ws)
    assert fz.focus_check_errors(ws) == 0
    diff = (O1.float() - O2.float()).abs()
    assert diff.max().item() <= 2e-2 and diff.mean().item() <= 2e-3
    assert (l1 - l2).abs().max().item() <= 1e-3
    rows = np.array([0, 1, 511, 512, 513, 4097, wl.n - 1])
    for h in (0, 31):
        kv = ref.kv_head(h, wl.H, wl.H_kv)
        wO, wL = ref.attention_rows(x["Q"][:, h:h + 1], x["K"][:, kv:kv + 1], x["V"][:, kv:kv + 1], g, wl.w,
                                    p.scale, rows, 1)
        assert_close(to_host(O2)[:, h:h + 1][:, :, rows], wO, "bf16", f"O head {h}")
        assert_lse_close(l2.cpu().numpy()[:, h:h + 1][:, :, rows], wL, "bf16", f"lse head {h}")
