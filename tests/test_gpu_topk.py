"""GPU parity for top-k group membership (k = 1, 2) through the C ABI, against
the fp64 oracle on the same seeded inputs.

Top-k ids and every index array are compared bit for bit; attention outputs
within max-abs 2e-2 / mean-abs 2e-3 for bf16 and 1e-5 for fp32 (LSE within
1e-3 / 1e-5), the same bar as the top-1 path.  The pair index (tokens sorted
by their two groups) is an implementation device of the library, so it is
checked against the oracle's top-1 index builder applied to pair ids that
this file computes from the group ids.
"""
import os

import numpy as np
import pytest

import oracle.focus_ref as ref
from learned_group_sparse_focus_gb300 import synth

from _helpers import (assert_close, assert_lse_close, margin_filtered, margin_filtered_topk, to_dev,
                      to_host)

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


def _pair_ids(G, K):
    lo, hi = np.minimum(G[..., 0], G[..., 1]), np.maximum(G[..., 0], G[..., 1])
    return (lo * K - lo * (lo + 1) // 2 + (hi - lo - 1)).astype(np.int32)


def _np_index(fz, p, x, ws, n_items_len, K):
    import torch
    torch.cuda.synchronize()
    v = fz.index_views(p, x, ws, n=n_items_len, K=K)
    out = {k: t.cpu().numpy() for k, t in v.items()}
    m = int(out["n_items"][0])
    out["items"] = out["items"][:m, :7]
    out["order"] = out["order"][:m]
    return out


# ------------------------------------------------------------------ assign ---

@pytest.mark.parametrize("dtype,B,n,D,d_g,K,A,H_kv", [
    ("bf16", 2, 300, 256, 64, 16, 1, 2),
    ("bf16", 1, 1000, 768, 32, 4, 1, 1),          # the pages' K = 4
    ("bf16", 1, 257, 520, 128, 40, 2, 2),
    ("bf16", 1, 200, 64, 64, 64, 8, 8),
    ("bf16", 1, 64, 1024, 128, 91, 1, 1),         # largest K for k = 2
    ("bf16", 1, 130, 128, 64, 2, 1, 1),           # K = 2: both groups, order decided
    ("bf16", 1, 21000, 128, 32, 4, 2, 2),         # tiles of fewer than 128 tokens
    ("f32", 2, 300, 128, 64, 4, 1, 1),
    ("f32", 1, 77, 96, 16, 9, 2, 2),
])
def test_assign_top2_bit_exact(fz, dtype, B, n, D, d_g, K, A, H_kv):
    import torch
    wl = synth.Workload("t", B=B, H=H_kv, H_kv=H_kv, n=n, d=64, D=D, d_g=d_g, K=K, w=4, A=A,
                        dtype=dtype, groups="uniform", seed=21 + n + K)
    x = margin_filtered_topk(wl, 2, parts=("assign",))
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace_topk(p, 2)
    gid = torch.full((B, A, n, 2), -1, dtype=torch.int32, device="cuda")
    fz.focus_assign_topk(p, 2, to_dev(x["h"], dtype), to_dev(x["W"], dtype), to_dev(x["C"], dtype), gid, ws)
    assert fz.focus_check_errors(ws) == 0
    assert np.array_equal(gid.cpu().numpy(), x["gid_ref"])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_assign_top1_through_topk_call_equals_focus_assign(fz, dtype):
    import torch
    wl = synth.Workload("t", B=1, H=2, H_kv=2, n=700, d=64, D=256, d_g=64, K=12, w=4, A=1,
                        dtype=dtype, groups="uniform", seed=77)
    x = margin_filtered(wl, parts=("assign",))
    p = fz.params_from_workload(wl)
    h, W, C = (to_dev(x[k], dtype) for k in ("h", "W", "C"))
    g1 = torch.empty((1, 1, 700), dtype=torch.int32, device="cuda")
    fz.focus_assign(p, h, W, C, g1, fz.alloc_workspace(p))
    gk = torch.empty((1, 1, 700, 1), dtype=torch.int32, device="cuda")
    ws = fz.alloc_workspace_topk(p, 1)
    fz.focus_assign_topk(p, 1, h, W, C, gk, ws)
    assert fz.focus_check_errors(ws) == 0
    assert torch.equal(g1, gk[..., 0])
    assert np.array_equal(g1.cpu().numpy(), x["gid_ref"])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_assign_top2_ties_rank_lower_index_first(fz, dtype):
    import torch
    wl = synth.Workload("t", B=1, H=1, H_kv=1, n=512, d=64, D=128, d_g=32, K=6, w=4, A=1,
                        dtype=dtype, groups="uniform", seed=9)
    x = synth.draw(wl, parts=("assign",))
    C = x["C"].copy()
    C[0, 4] = C[0, 2]                      # centroids 2 and 4 identical
    g_ref, _ = ref.assign_topk(x["h"], x["W"], C, 2)
    _, mg = ref.assign_topk(x["h"], x["W"], C[:, [0, 1, 2, 3, 5]], 2)   # gaps between distinct centroids
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace_topk(p, 2)
    gid = torch.empty((1, 1, 512, 2), dtype=torch.int32, device="cuda")
    fz.focus_assign_topk(p, 2, to_dev(x["h"], dtype), to_dev(x["W"], dtype), to_dev(C, dtype), gid, ws)
    g = gid.cpu().numpy()
    ok = mg >= 1e-3
    both = (g_ref[..., 0] == 2) & (g_ref[..., 1] == 4)       # the tie decides the runner-up
    assert np.any(both & ok)
    assert np.array_equal(g[ok], g_ref[ok])
    assert not np.any((g[..., 0] == 4) & (g[..., 1] == 2))


# ------------------------------------------------------------------- index ---

@pytest.mark.parametrize("B,A,n,K,w,kind", [
    (1, 1, 1, 2, 1, "uniform"),
    (2, 1, 300, 4, 7, "uniform"),
    (1, 2, 1000, 16, 64, "zipf"),
    (2, 3, 2049, 64, 200, "zipf"),
    (1, 1, 777, 2, 32, "both"),                # every token in groups 0 and 1
    (1, 1, 5000, 91, 3, "uniform"),            # largest K for k = 2 (4095 pairs)
    (3, 1, 130, 4, 0, "uniform"),              # w = 0 behaves as w = 1
    (1, 1, 4100, 3, 5000, "uniform"),          # w > n: no far keys
])
def test_index_top2_bit_exact(fz, B, A, n, K, w, kind):
    import torch
    G = synth.draw_group_ids_topk(200 + n, B, A, n, K, 2, kind)
    p = fz.make_params(B=B, H=A, H_kv=A, n=n, d=64, D=64, d_g=32, K=K, A=A, w=w)
    ws = fz.alloc_workspace_topk(p, 2)
    idx = fz.focus_build_index_topk(p, 2, torch.from_numpy(G).cuda(), ws)
    assert fz.focus_check_errors(ws) == 0
    we = max(w, 1)
    if K <= 8:          # bf16 params (the make_params default): the split layout
        _check_split_index(fz, p, idx, ws, G, n, K, we)
        return
    assert idx.split == 0
    # entries
    got = _np_index(fz, p, idx.entry, ws, 2 * n, K)
    want = ref.build_index_topk(G, K, we)
    for k_got, k_want in (("counts", "counts"), ("offsets", "offsets"), ("perm", "perm"), ("rank", "rank"),
                          ("farlen_tok", "farlen_entry"), ("farlen_slot", "farlen_slot")):
        assert np.array_equal(got[k_got], want[k_want]), k_got
    items = ref.work_items(want, fz.TILE_M)
    assert np.array_equal(got["items"], items)
    assert np.array_equal(got["order"], ref.lpt_order(items, fz.TILE_N))
    # pairs
    Kp = K * (K - 1) // 2
    pg = _pair_ids(G, K)
    P = B * A
    ws_base = ws.data_ptr()         # pair_gid and far_tok point into the workspace
    got_pg = ws[idx.pair_gid - ws_base:idx.pair_gid - ws_base + P * n * 4].view(torch.int32).cpu().numpy()
    assert np.array_equal(got_pg.reshape(B, A, n), pg)
    gotp = _np_index(fz, p, idx.pair, ws, n, Kp)
    wantp = ref.build_index(pg, Kp, we)
    for key in ("counts", "offsets", "perm", "rank", "farlen_tok", "farlen_slot"):
        assert np.array_equal(gotp[key], wantp[key]), "pair " + key
    pitems = ref.work_items(wantp, fz.TILE_M)
    assert np.array_equal(gotp["items"], pitems)
    # far flag per token
    far = ws[idx.far_tok - ws_base:idx.far_tok - ws_base + P * n * 4].view(torch.int32).cpu().numpy()
    fe = want["farlen_entry"].reshape(B, A, n, 2)
    assert np.array_equal(far.reshape(B, A, n), (fe.max(axis=-1) > 0).astype(np.int32))


def _check_split_index(fz, p, idx, ws, G, n, K, we):
    """Split layout (K <= 8): entries sorted by (group, other group, position),
    far prefixes per sub-run, one work item per (row tile, sub-run)."""
    import torch
    assert idx.split == 1 and idx.farlen_sub
    got = _np_index(fz, p, idx.entry, ws, 2 * n, K * K)
    want = ref.build_index_top2_split(G, K, we)
    for k_got, k_want in (("counts", "counts"), ("offsets", "offsets"), ("perm", "perm"), ("rank", "rank"),
                          ("farlen_tok", "farlen_entry")):
        assert np.array_equal(got[k_got], want[k_want]), k_got
    P = p.B * p.A
    base = ws.data_ptr()
    off = idx.farlen_sub - base
    fs = ws[off:off + P * 2 * n * (K - 1) * 4].view(torch.int32).cpu().numpy()
    assert np.array_equal(fs.reshape(p.B, p.A, 2 * n, K - 1), want["farlen_sub"])
    v = fz.index_views(p, idx.entry, ws, n=2 * n, K=K * K)
    m = int(v["n_items"][0])
    items = v["items"][:m].cpu().numpy()
    witems = ref.work_items_top2_split(want, fz.TILE_M)
    assert np.array_equal(items, witems)
    assert np.array_equal(v["order"][:m].cpu().numpy(), ref.lpt_order(witems, fz.TILE_N))
    far = ws[idx.far_tok - base:idx.far_tok - base + P * n * 4].view(torch.int32).cpu().numpy()
    fe = want["farlen_entry"].reshape(p.B, p.A, n, 2)
    assert np.array_equal(far.reshape(p.B, p.A, n), (fe.max(axis=-1) > 0).astype(np.int32))


def test_index_top2_repeated_id_is_reported(fz):
    import torch
    G = synth.draw_group_ids_topk(3, 1, 1, 100, 4, 2, "uniform")
    G[0, 0, 17, 1] = G[0, 0, 17, 0]
    p = fz.make_params(B=1, H=1, H_kv=1, n=100, d=64, D=64, d_g=32, K=4, A=1, w=3)
    ws = fz.alloc_workspace_topk(p, 2)
    fz.focus_build_index_topk(p, 2, torch.from_numpy(G).cuda(), ws)
    assert fz.focus_check_errors(ws) == 6
    assert fz.focus_check_errors(ws) == 0


# --------------------------------------------------------------- attention ---

def _topk_case(fz, dtype, B, H, H_kv, A, n, d, K, k, w, kind, seed):
    import torch
    rng = np.random.default_rng(seed)
    store = (lambda a: synth.round_bf16(a)) if dtype == "bf16" else (lambda a: a)
    Q = store(rng.standard_normal((B, H, n, d)).astype(np.float32))
    Kt = store(rng.standard_normal((B, H_kv, n, d)).astype(np.float32))
    V = store(rng.standard_normal((B, H_kv, n, d)).astype(np.float32))
    G = synth.draw_group_ids_topk(seed, B, A, n, K, k, kind)
    p = fz.make_params(B=B, H=H, H_kv=H_kv, n=n, d=d, D=64, d_g=32, K=K, A=A, w=w, dtype=dtype)
    ws = fz.alloc_workspace_topk(p, k)
    Qd, Kd, Vd = to_dev(Q, dtype), to_dev(Kt, dtype), to_dev(V, dtype)
    O = torch.full_like(Qd, float("nan"))
    lse = torch.full((B, H, n), float("nan"), dtype=torch.float32, device="cuda")
    idx = fz.focus_build_index_topk(p, k, torch.from_numpy(G).cuda(), ws)
    fz.focus_attention_topk_fwd(p, Qd, Kd, Vd, idx, O, lse, ws)
    assert fz.focus_check_errors(ws) == 0
    want_O, want_L = ref.attention_rows_topk(Q, Kt, V, G, w, p.scale, np.arange(n), A)
    assert_close(to_host(O), want_O, dtype, "O")
    assert_lse_close(lse.cpu().numpy(), want_L, dtype, "lse")
    return O, lse, G


@pytest.mark.parametrize("dtype,B,H,H_kv,A,n,d,K,w,kind", [
    ("bf16", 1, 2, 2, 1, 300, 128, 4, 32, "uniform"),
    ("bf16", 2, 4, 2, 1, 513, 64, 8, 100, "zipf"),
    ("bf16", 1, 4, 2, 2, 1000, 128, 16, 128, "uniform"),    # one assignment per kv head
    ("bf16", 1, 2, 1, 1, 700, 128, 2, 40, "both"),         # K = k = 2: dense causal
    ("bf16", 1, 2, 2, 1, 1, 128, 3, 5, "uniform"),          # one token
    ("bf16", 1, 2, 2, 1, 257, 128, 5, 0, "uniform"),        # w = 0
    ("bf16", 1, 2, 2, 1, 600, 64, 6, 1000, "uniform"),      # w > n
    ("bf16", 1, 8, 2, 2, 1500, 128, 4, 256, "zipf"),
    ("bf16", 1, 2, 2, 1, 2000, 128, 91, 64, "uniform"),     # largest K for k = 2
    ("f32", 1, 2, 2, 1, 256, 64, 4, 32, "uniform"),
    ("f32", 1, 4, 2, 2, 333, 128, 5, 20, "zipf"),
    ("f32", 2, 2, 1, 1, 100, 64, 2, 7, "both"),
])
def test_attention_top2_all_rows(fz, dtype, B, H, H_kv, A, n, d, K, w, kind):
    _topk_case(fz, dtype, B, H, H_kv, A, n, d, K, 2, w, kind, seed=n + w + K)


@pytest.mark.parametrize("dtype,n,d,K,w", [("bf16", 900, 128, 8, 64), ("f32", 300, 64, 4, 16)])
def test_attention_top1_through_topk_call_is_the_top1_path(fz, dtype, n, d, K, w):
    """k = 1 runs the same kernels on the same arrays as focus_attention_fwd:
    bit-identical output."""
    import torch
    O, lse, G = _topk_case(fz, dtype, 1, 4, 2, 1, n, d, K, 1, w, "uniform", seed=5 + n)
    p = fz.make_params(B=1, H=4, H_kv=2, n=n, d=d, D=64, d_g=32, K=K, A=1, w=w, dtype=dtype)
    rng = np.random.default_rng(5 + n)
    store = (lambda a: synth.round_bf16(a)) if dtype == "bf16" else (lambda a: a)
    Q = store(rng.standard_normal((1, 4, n, d)).astype(np.float32))
    Kt = store(rng.standard_normal((1, 2, n, d)).astype(np.float32))
    V = store(rng.standard_normal((1, 2, n, d)).astype(np.float32))
    ws = fz.alloc_workspace(p)
    idx = fz.focus_build_index(p, torch.from_numpy(np.ascontiguousarray(G[..., 0])).cuda(), ws)
    O1 = torch.empty_like(O)
    lse1 = torch.empty_like(lse)
    fz.focus_attention_fwd(p, to_dev(Q, dtype), to_dev(Kt, dtype), to_dev(V, dtype), idx, O1, lse1, ws)
    assert fz.focus_check_errors(ws) == 0
    assert torch.equal(O, O1)
    assert torch.equal(lse, lse1)


def test_attention_top2_deterministic(fz):
    import torch
    O1, l1, _ = _topk_case(fz, "bf16", 1, 2, 1, 1, 3000, 128, 4, 2, 128, "zipf", seed=41)
    O2, l2, _ = _topk_case(fz, "bf16", 1, 2, 1, 1, 3000, 128, 4, 2, 128, "zipf", seed=41)
    assert torch.equal(O1, O2) and torch.equal(l1, l2)


def test_layer_top2_from_hidden_states(fz):
    """assign (top-2 on the tensor cores) -> index -> attention, end to end, on
    a margin-filtered draw: ids bit-exact, output within tolerance."""
    import torch
    wl = synth.workload("gpt2_small_1k", B=2, n=1024, K=4)
    x = margin_filtered_topk(wl, 2)
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace_topk(p, 2)
    dev = {k: to_dev(x[k], "bf16") for k in ("h", "W", "C", "Q", "K", "V")}
    O, gid, _, lse = fz.run_layer_topk(p, 2, dev["h"], dev["W"], dev["C"], dev["Q"], dev["K"], dev["V"], ws,
                                       want_lse=True)
    assert fz.focus_check_errors(ws) == 0
    assert np.array_equal(gid.cpu().numpy(), x["gid_ref"])
    rows = np.unique(np.concatenate([np.arange(80), np.random.default_rng(3).integers(0, wl.n, 200)]))
    want_O, want_L = ref.attention_rows_topk(x["Q"], x["K"], x["V"], x["gid_ref"], wl.w, p.scale, rows, wl.A)
    assert_close(to_host(O)[:, :, rows], want_O, "bf16", "O")
    assert_lse_close(lse.cpu().numpy()[:, :, rows], want_L, "bf16", "lse")


def test_top2_at_benchmark_size_sampled_rows(fz):
    """The top-2 benchmark layer (32K tokens, 32 query / 8 kv heads, K = 4,
    k = 2) in the benchmark's launch configuration, sampled rows against the
    oracle."""
    import torch
    wl = synth.workload("gqa_32k", K=4)
    G = synth.draw_group_ids_topk(wl.seed, wl.B, wl.A, wl.n, wl.K, 2, "uniform")
    x = synth.draw(wl, parts=("attn",))
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace_topk(p, 2)
    Qd, Kd, Vd = (to_dev(x[k], "bf16") for k in ("Q", "K", "V"))
    idx = fz.focus_build_index_topk(p, 2, torch.from_numpy(G).cuda(), ws)
    O = torch.empty_like(Qd)
    lse = torch.empty((wl.B, wl.H, wl.n), dtype=torch.float32, device="cuda")
    fz.focus_attention_topk_fwd(p, Qd, Kd, Vd, idx, O, lse, ws)
    assert fz.focus_check_errors(ws) == 0
    rng = np.random.default_rng(17)
    rows = np.unique(np.concatenate([np.arange(wl.w + 2), [wl.n - 1], rng.integers(0, wl.n, 24)]))
    heads = [0, 13, 31]
    # the oracle maps query heads to kv heads by the full head count: run it per head
    Og = to_host(O)
    Lg = lse.cpu().numpy()
    for h in heads:
        kv = ref.kv_head(h, wl.H, wl.H_kv)
        wO, wL = ref.attention_rows_topk(x["Q"][:, h:h + 1], x["K"][:, kv:kv + 1], x["V"][:, kv:kv + 1], G, wl.w,
                                         p.scale, rows, 1, row_block=64)
        assert_close(Og[:, h:h + 1][:, :, rows], wO, "bf16", f"O head {h}")
        assert_lse_close(Lg[:, h:h + 1][:, :, rows], wL, "bf16", f"lse head {h}")
