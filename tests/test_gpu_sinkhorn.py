"""GPU parity for the Sinkhorn soft assignment (focus_assign_scores,
focus_sinkhorn_fwd) against the fp64 oracle.

Tolerances, derived from fp32 arithmetic: scores sum D products and then
d_g products in fp32, so |S_gpu - S| <= 3e-5 * sum |terms| (the bound
(D + d_g) * 2^-24 relative to the magnitude sum is far looser; 3e-5 covers the
observed random-walk growth with margin).  Sinkhorn works on log-potentials in
fp32: an entry exp(x + u + v) is off by a few units of 2^-24 times
|x| + |u| + |v| (<= ~40 here) relative, so G within 1e-5 absolute
(entries are <= 1) and 1e-4 relative where G >= 1e-6.
"""
import os

import numpy as np
import pytest

import oracle.focus_ref as ref
from learned_group_sparse_focus_gb300 import synth

from _helpers import to_dev

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


def _check_g(got, want):
    diff = np.abs(got - want)
    assert diff.max() <= 1e-5, f"G max abs {diff.max():.3e}"
    big = want >= 1e-6
    rel = diff[big] / want[big]
    assert rel.max() <= 1e-4, f"G max rel {rel.max():.3e}"


@pytest.mark.parametrize("dtype,B,n,D,d_g,K,A,H_kv", [
    ("bf16", 2, 300, 256, 64, 16, 1, 2),
    ("bf16", 1, 257, 520, 128, 40, 2, 2),
    ("bf16", 1, 64, 1024, 32, 300, 1, 1),
    ("f32", 2, 300, 128, 64, 4, 1, 1),
    ("f32", 1, 77, 96, 16, 9, 2, 2),
])
def test_scores_match_oracle(fz, dtype, B, n, D, d_g, K, A, H_kv):
    import torch
    wl = synth.Workload("t", B=B, H=H_kv, H_kv=H_kv, n=n, d=64, D=D, d_g=d_g, K=K, w=4, A=A,
                        dtype=dtype, groups="uniform", seed=51 + n + K)
    x = synth.draw(wl, parts=("assign",))
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace_sinkhorn(p)
    S = torch.full((B, A, n, K), float("nan"), dtype=torch.float32, device="cuda")
    fz.focus_assign_scores(p, to_dev(x["h"], dtype), to_dev(x["W"], dtype), to_dev(x["C"], dtype), S, ws)
    assert fz.focus_check_errors(ws) == 0
    want = ref.scores(x["h"], x["W"], x["C"])
    mag = ref.scores(np.abs(x["h"]), np.abs(x["W"]), np.abs(x["C"]))
    diff = np.abs(S.cpu().numpy().astype(np.float64) - want)
    assert np.all(diff <= 3e-5 * mag + 1e-7), f"max excess {(diff - 3e-5 * mag).max():.3e}"


@pytest.mark.parametrize("B,A,n,K,T,tau", [
    (1, 1, 300, 4, 5, 1.0),
    (2, 2, 1000, 16, 10, 0.5),
    (1, 1, 4096, 64, 20, 1.0),
    (1, 1, 257, 91, 3, 2.0),
    (1, 1, 128, 1, 2, 1.0),          # K = 1: every entry 1
    (1, 1, 50, 256, 4, 1.0),         # K > n
    (1, 1, 3000, 300, 7, 1.0),       # K > 256: columns in two passes
    (1, 1, 1, 5, 3, 1.0),            # one token
    (1, 1, 300000, 8, 3, 1.0),       # more than 2048 row chunks of 128
    (1, 1, 777, 33, 6, 0.7),         # K % 4 != 0: two reads of S per round
    (1, 1, 777, 36, 6, 0.7),         # one pass per round, second float4 slot mostly empty
    (1, 2, 1000, 132, 5, 1.0),       # eight float4 slots per lane, most empty
    (1, 1, 2000, 64, 5, 0.2),        # peaked rows: X up to about 45
])
def test_sinkhorn_matches_oracle(fz, B, A, n, K, T, tau):
    import torch
    rng = np.random.default_rng(n + K + T)
    S = (rng.standard_normal((B, A, n, K)) * 3).astype(np.float32)
    p = fz.make_params(B=B, H=A, H_kv=A, n=n, d=64, D=64, d_g=32, K=K, A=A, w=1)
    ws = fz.alloc_workspace_sinkhorn(p)
    Sd = torch.from_numpy(S).cuda()
    G = torch.full_like(Sd, float("nan"))
    fz.focus_sinkhorn_fwd(p, T, tau, Sd, G, ws)
    assert fz.focus_check_errors(ws) == 0
    _check_g(G.cpu().numpy().astype(np.float64), ref.sinkhorn(S, T, tau))
    # in place gives the same values
    fz.focus_sinkhorn_fwd(p, T, tau, Sd, Sd, ws)
    torch.cuda.synchronize()
    assert torch.equal(Sd, G)


def test_sinkhorn_converges_to_the_marginals(fz):
    import torch
    rng = np.random.default_rng(7)
    n, K = 2048, 32
    S = torch.from_numpy((rng.standard_normal((1, 1, n, K)) * 2).astype(np.float32)).cuda()
    p = fz.make_params(B=1, H=1, H_kv=1, n=n, d=64, D=64, d_g=32, K=K, A=1, w=1)
    ws = fz.alloc_workspace_sinkhorn(p)
    G = torch.empty_like(S)
    fz.focus_sinkhorn_fwd(p, 300, 1.0, S, G, ws)
    g = G.double().cpu().numpy()[0, 0]
    np.testing.assert_allclose(g.sum(axis=1), 1.0, atol=1e-5)
    np.testing.assert_allclose(g.sum(axis=0), n / K, rtol=1e-4)


def test_scores_then_sinkhorn_on_a_model_shape(fz):
    """The 32K GQA layer's assignment (n = 32768, D = 4096, d_g = 64, K = 64):
    scores on the tensor cores, 10 Sinkhorn rounds, against the oracle on the
    whole matrix."""
    import torch
    wl = synth.WORKLOADS["gqa_32k"]
    x = synth.draw(wl, parts=("assign",))
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace_sinkhorn(p)
    S = torch.empty((wl.B, wl.A, wl.n, wl.K), dtype=torch.float32, device="cuda")
    fz.focus_assign_scores(p, to_dev(x["h"], "bf16"), to_dev(x["W"], "bf16"), to_dev(x["C"], "bf16"), S, ws)
    G = torch.empty_like(S)
    fz.focus_sinkhorn_fwd(p, 10, 1.0, S, G, ws)
    assert fz.focus_check_errors(ws) == 0
    S_ref = ref.scores(x["h"], x["W"], x["C"])
    # Sinkhorn of the GPU's own fp32 scores isolates the normalisation error;
    # the scores themselves are checked above
    _check_g(G.cpu().numpy().astype(np.float64), ref.sinkhorn(S.cpu().numpy(), 10, 1.0))
    assert np.abs(S.cpu().numpy() - S_ref).max() < 1e-2
