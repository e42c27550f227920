"""GPU parity for the backward pass (focus_attention_bwd: tcgen05 tensor cores
for bf16, CUDA cores for fp32) against the fp64 oracle's gradients on the same
inputs and the same upstream gradient dO.

The GPU runs the forward first (its O and LSE feed the backward, as in
training).  Tolerances, relative to M = max(largest reference gradient entry, 0.1):
fp32 max |error| <= 1e-4 M (exp2 of the recomputed scores is good to about
2^-22 times |score - LSE| <= ~20, then sums of up to n products in fp32);
bf16 max |error| <= 2e-2 M and mean <= 2e-3 M (the forward O that enters
Delta = dO . O and the stored gradients are bf16, 2^-9 relative each).
"""
import os

import numpy as np
import pytest

import oracle.focus_ref as ref
from learned_group_sparse_focus_gb300 import synth

from _helpers import to_dev, to_host

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


def _close(got, want, dtype, what):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.all(np.isfinite(got)), what
    # floor 0.1: where the exact gradient is zero (one kept key per row) the
    # GPU returns rounding noise of the scale of its O(1) terms; the floor
    # makes the fp32 bar 1e-5 absolute there, the forward's own
    M = max(np.abs(want).max(), 0.1)
    diff = np.abs(got - want)
    if dtype == "bf16":
        assert diff.max() <= 2e-2 * M, f"{what}: max {diff.max() / M:.3e} of max|ref|"
        assert diff.mean() <= 2e-3 * M, f"{what}: mean {diff.mean() / M:.3e} of max|ref|"
    else:
        assert diff.max() <= 1e-4 * M, f"{what}: max {diff.max() / M:.3e} of max|ref|"


def _run(fz, dtype, B, H, H_kv, A, n, d, K, w, kind, seed, twice=False):
    import torch
    rng = np.random.default_rng(seed)
    store = (lambda a: synth.round_bf16(a)) if dtype == "bf16" else (lambda a: a)
    Q = store(rng.standard_normal((B, H, n, d)).astype(np.float32))
    Kt = store(rng.standard_normal((B, H_kv, n, d)).astype(np.float32))
    V = store(rng.standard_normal((B, H_kv, n, d)).astype(np.float32))
    dO = store(rng.standard_normal((B, H, n, d)).astype(np.float32))
    g = synth.draw_group_ids(seed, B, A, n, K, kind)
    p = fz.make_params(B=B, H=H, H_kv=H_kv, n=n, d=d, D=64, d_g=32, K=K, A=A, w=w, dtype=dtype)
    ws = fz.alloc_workspace(p)
    wsb = fz.alloc_workspace_backward(p)
    Qd, Kd, Vd, dOd = (to_dev(x, dtype) for x in (Q, Kt, V, dO))
    idx = fz.focus_build_index(p, torch.from_numpy(g).cuda(), ws)
    O = torch.empty_like(Qd)
    lse = torch.empty((B, H, n), dtype=torch.float32, device="cuda")
    fz.focus_attention_fwd(p, Qd, Kd, Vd, idx, O, lse, ws)
    dQ = torch.full_like(Qd, float("nan"))
    dK = torch.full_like(Kd, float("nan"))
    dV = torch.full_like(Vd, float("nan"))
    fz.focus_attention_bwd(p, Qd, Kd, Vd, O, dOd, lse, idx, dQ, dK, dV, wsb)
    assert fz.focus_check_errors(ws) == 0 and fz.focus_check_errors(wsb) == 0
    out = (to_host(dQ), to_host(dK), to_host(dV))
    if twice:
        # the same call again on the same workspaces
        fz.focus_attention_bwd(p, Qd, Kd, Vd, O, dOd, lse, idx, dQ, dK, dV, wsb)
        assert fz.focus_check_errors(wsb) == 0
        return (Q, Kt, V, dO, g, p), out, (to_host(dQ), to_host(dK), to_host(dV))
    return (Q, Kt, V, dO, g, p), out


@pytest.mark.parametrize("dtype,B,H,H_kv,A,n,d,K,w,kind", [
    ("f32", 1, 2, 2, 1, 256, 64, 4, 32, "uniform"),
    ("f32", 1, 4, 2, 2, 333, 128, 5, 20, "zipf"),
    ("f32", 2, 2, 1, 1, 100, 64, 1, 7, "one"),              # K = 1: dense causal
    ("f32", 1, 2, 2, 1, 130, 128, 130, 1, "distinct"),      # self pairs only
    ("bf16", 1, 2, 2, 1, 300, 128, 4, 32, "uniform"),
    ("bf16", 1, 4, 2, 1, 513, 64, 8, 100, "zipf"),
    ("bf16", 1, 8, 2, 2, 700, 128, 6, 64, "uniform"),       # per-KV-head ids, 4 query heads per KV head
    ("bf16", 1, 2, 2, 1, 1, 128, 3, 5, "uniform"),          # one token
    ("bf16", 1, 2, 1, 1, 400, 64, 5, 1000, "uniform"),      # w > n
    ("bf16", 2, 2, 2, 1, 257, 128, 3, 0, "blocks"),         # w = 0
    ("bf16", 1, 4, 2, 1, 2048, 128, 8, 128, "zipf"),        # many key and query tiles per group
    ("bf16", 1, 2, 2, 2, 1500, 64, 1, 200, "one"),          # one group: dense-like far part, d = 64
])
def test_backward_all_rows(fz, dtype, B, H, H_kv, A, n, d, K, w, kind):
    (Q, Kt, V, dO, g, p), (dQ, dK, dV) = _run(fz, dtype, B, H, H_kv, A, n, d, K, w, kind, seed=n + K + w + 3)
    wQ, wK, wV = ref.attention_backward(Q, Kt, V, g, max(w, 1), p.scale, A, dO)
    _close(dQ, wQ, dtype, "dQ")
    _close(dK, wK, dtype, "dK")
    _close(dV, wV, dtype, "dV")


@pytest.mark.gpu
def test_backward_many_units_per_cta_all_rows_and_rerun(fz):
    """More units than the 152 persistent CTAs in every kernel (B = 2, four
    KV heads with an assignment each, n = 4096: 256 window and key-tile
    units), so CTAs cross unit boundaries (fixed-tile reload, accumulator
    reuse, the dQ epilogue's staging slot, the far dK/dV work order over
    several problems); every element against the oracle, and a second call on
    the same workspaces must give the same bits (the unit ticket starts again
    from zero and the order of units changes no result)."""
    import torch
    B, H, H_kv, A, n, d, K, w = 2, 4, 4, 4, 4096, 64, 6, 64
    (Q, Kt, V, dO, g, p), (dQ, dK, dV), (dQ2, dK2, dV2) = _run(fz, "bf16", B, H, H_kv, A, n, d, K, w, "zipf",
                                                              seed=4107, twice=True)
    wQ, wK, wV = ref.attention_backward(Q, Kt, V, g, w, p.scale, A, dO)
    _close(dQ, wQ, "bf16", "dQ")
    _close(dK, wK, "bf16", "dK")
    _close(dV, wV, "bf16", "dV")
    assert np.array_equal(dQ, dQ2) and np.array_equal(dK, dK2) and np.array_equal(dV, dV2)


def _key_rows(n, seed):
    """Sampled key rows: the first keys, both tile edges at 128 and 256, the
    last keys, and random keys in the second half (late keys are kept by few
    queries, which keeps the oracle's cost down)."""
    r = np.random.default_rng(seed).integers(n // 2, n, 8)
    return np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, n // 2, n - 129, n - 2, n - 1], r]))


def test_backward_at_a_long_length_sampled_and_invariants(fz):
    """n = 8192, 8 query / 2 KV heads, d = 128, Zipf groups: sampled dQ rows
    and sampled dK, dV rows against the oracle element by element, and
    sum_j dV_j = sum_i dO_i, sum_j dK_j = 0 per KV head (rows of P sum to 1,
    rows of dS to 0)."""
    (Q, Kt, V, dO, g, p), (dQ, dK, dV) = _run(fz, "bf16", 1, 8, 2, 1, 8192, 128, 16, 256, "zipf", seed=99)
    rows = np.unique(np.concatenate([np.arange(260), [8191], np.random.default_rng(5).integers(0, 8192, 40)]))
    want = ref.attention_backward_dq_rows(Q, Kt, V, g, 256, p.scale, 1, dO, rows)
    _close(dQ[:, :, rows], want, "bf16", "dQ rows")
    krows = _key_rows(8192, 6)
    wK, wV = ref.attention_backward_dkv_rows(Q, Kt, V, g, 256, p.scale, 1, dO, krows)
    _close(dK[:, :, krows], wK, "bf16", "dK rows")
    _close(dV[:, :, krows], wV, "bf16", "dV rows")
    for kv in range(2):
        heads = [h for h in range(8) if ref.kv_head(h, 8, 2) == kv]
        sdo = dO[0, heads].astype(np.float64).sum(axis=(0, 1))
        M = np.abs(sdo).max()
        assert np.abs(dV[0, kv].sum(axis=0) - sdo).max() <= 2e-2 * M
        assert np.abs(dK[0, kv].sum(axis=0)).max() <= 2e-2 * np.abs(dK[0, kv]).sum(axis=0).max()


def test_backward_at_the_32k_gqa_workload_sampled(fz):
    """The 32K GQA benchmark shape (32 query / 8 KV heads, n = 32768, d = 128,
    w = 512, K = 64 Zipf groups) at full size: sampled dQ rows of two query
    heads and sampled dK, dV rows of two KV heads against the oracle."""
    wl = synth.WORKLOADS["gqa_32k"]
    (Q, Kt, V, dO, g, p), (dQ, dK, dV) = _run(fz, "bf16", 1, wl.H, wl.H_kv, 1, wl.n, wl.d, wl.K, wl.w, "zipf",
                                              seed=1004)
    hpk = wl.H // wl.H_kv
    rows = np.unique(np.concatenate([[0, 1, 511, 512, 513, wl.n - 1],
                                     np.random.default_rng(8).integers(0, wl.n, 30)]))
    for h in (0, wl.H - 1):
        want = ref.attention_backward_dq_rows(Q[:, h:h + 1], Kt[:, h // hpk:h // hpk + 1],
                                              V[:, h // hpk:h // hpk + 1], g, wl.w, p.scale, 1,
                                              dO[:, h:h + 1], rows)
        _close(dQ[:, h:h + 1, rows], want, "bf16", f"dQ rows, head {h}")
    krows = np.unique(np.concatenate([[wl.n - 1, wl.n - 2, wl.n - 600],
                                      np.random.default_rng(9).integers(wl.n - 2048, wl.n, 5)]))
    for kv in (0, wl.H_kv - 1):
        hs = slice(kv * hpk, (kv + 1) * hpk)
        wK, wV = ref.attention_backward_dkv_rows(Q[:, hs], Kt[:, kv:kv + 1], V[:, kv:kv + 1], g, wl.w, p.scale,
                                                 1, dO[:, hs], krows)
        _close(dK[:, kv:kv + 1, krows], wK, "bf16", f"dK rows, KV head {kv}")
        _close(dV[:, kv:kv + 1, krows], wV, "bf16", f"dV rows, KV head {kv}")
