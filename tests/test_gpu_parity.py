"""GPU parity: every step of the hot path, called through the C ABI, against
the fp64 oracle on the same seeded inputs.

Group ids and every index array are compared bit for bit; attention outputs
within max-abs 2e-2 / mean-abs 2e-3 for bf16 and 1e-5 for fp32 (LSE within
1e-3 / 1e-5).  Small shapes (ragged tails, several tiles, degenerate cases)
are compared on every row; the five named workloads run at full size in the
benchmark's launch configuration and are compared on sampled rows.
"""
import os

import numpy as np
import pytest

import oracle.focus_ref as ref
from learned_group_sparse_focus_gb300 import synth

from _helpers import (assert_close, assert_lse_close, margin_filtered, sample_rows, to_dev,
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


def _ws(fz, p):
    return fz.alloc_workspace(p)


def _index_np(fz, p, idx, ws):
    import torch
    torch.cuda.synchronize()
    v = fz.index_views(p, idx, ws)
    out = {k: t.cpu().numpy() for k, t in v.items()}
    m = int(out["n_items"][0])
    out["items"] = out["items"][:m, :7]
    out["order"] = out["order"][:m]
    return out


def _check_index(got, want_idx, want_items, want_order):
    for k in ("counts", "offsets", "perm", "rank", "farlen_tok", "farlen_slot"):
        assert np.array_equal(got[k], want_idx[k]), k
    assert np.array_equal(got["items"], want_items), "items"
    assert np.array_equal(got["order"], want_order), "order"


# ------------------------------------------------------------------ assign ---

@pytest.mark.parametrize("dtype,B,n,D,d_g,K,A,H_kv", [
    ("bf16", 2, 300, 256, 64, 16, 1, 2),
    ("bf16", 1, 1000, 768, 32, 7, 1, 1),
    ("bf16", 1, 257, 520, 128, 40, 2, 2),
    ("bf16", 3, 129, 128, 64, 1, 1, 1),
    ("bf16", 1, 200, 64, 64, 64, 8, 8),      # A * d_g = 512 columns
    ("bf16", 1, 64, 1024, 32, 300, 1, 1),    # centroids in several shared-memory chunks
    # more tokens than 128 per SM: tiles shrink so every SM gets the same count
    ("bf16", 1, 20000, 256, 64, 16, 1, 1),   # 66-token tiles
    ("bf16", 2, 16500, 128, 32, 8, 2, 2),    # 109-token tiles across the batch boundary
    ("bf16", 1, 20000, 256, 64, 16, 8, 8),   # 512 columns: two passes of four assignments
    ("bf16", 1, 3000, 256, 64, 37, 1, 1),    # scores on the tensor cores, N = 48 (11 empty centroid rows)
    ("bf16", 1, 3000, 256, 64, 91, 1, 1),    # d_g = 64 with K > 64: the scores in FMAs
    ("f32", 2, 300, 128, 64, 4, 1, 1),
    ("f32", 1, 77, 96, 16, 9, 2, 2),
])
def test_assign_bit_exact(fz, dtype, B, n, D, d_g, K, A, H_kv):
    import torch
    wl = synth.Workload("t", B=B, H=H_kv, H_kv=H_kv, n=n, d=64, D=D, d_g=d_g, K=K, w=4, A=A,
                        dtype=dtype, groups="uniform", seed=11 + n + K)
    x = margin_filtered(wl, parts=("assign",))
    p = fz.params_from_workload(wl)
    ws = _ws(fz, p)
    gid = torch.full((B, A, n), -1, dtype=torch.int32, device="cuda")
    fz.focus_assign(p, to_dev(x["h"], dtype), to_dev(x["W"], dtype), to_dev(x["C"], dtype), gid, ws)
    assert fz.focus_check_errors(ws) == 0
    assert np.array_equal(gid.cpu().numpy(), x["gid_ref"])


@pytest.mark.parametrize("dtype,d_g", [("bf16", 32), ("f32", 32), ("bf16", 64)])
def test_assign_ties_go_to_lowest_index(fz, dtype, d_g):
    # d_g = 64 in bf16 takes the tensor-core scores: identical centroids must
    # still give identical scores
    import torch
    wl = synth.Workload("t", B=1, H=1, H_kv=1, n=512, d=64, D=128, d_g=d_g, K=6, w=4, A=1,
                        dtype=dtype, groups="uniform", seed=5)
    x = synth.draw(wl, parts=("assign",))
    C = x["C"].copy()
    C[0, 3] = C[0, 1]                      # centroids 1 and 3 identical
    C[0, 5] = C[0, 1]
    g_ref, _ = ref.assign(x["h"], x["W"], C)
    _, mg = ref.assign(x["h"], x["W"], C[:, [0, 1, 2, 4]])    # gaps between distinct centroids
    p = fz.params_from_workload(wl)
    ws = _ws(fz, p)
    gid = torch.empty((1, 1, 512), dtype=torch.int32, device="cuda")
    fz.focus_assign(p, to_dev(x["h"], dtype), to_dev(x["W"], dtype), to_dev(C, dtype), gid, ws)
    g = gid.cpu().numpy()
    ok = mg >= 1e-3
    assert np.any(g_ref[ok] == 1)
    assert np.array_equal(g[ok], g_ref[ok])
    assert not np.any(g == 3) and not np.any(g == 5)


# ------------------------------------------------------------------- index ---

@pytest.mark.parametrize("B,A,n,K,w,kind", [
    (1, 1, 1, 1, 1, "uniform"),
    (2, 1, 300, 5, 7, "uniform"),
    (1, 2, 1000, 16, 64, "zipf"),
    (2, 3, 2049, 64, 200, "zipf"),
    (1, 1, 777, 1, 32, "one"),
    (1, 1, 512, 512, 1, "distinct"),
    (1, 1, 300, 700, 10, "uniform"),          # K > n: empty groups
    (1, 1, 5000, 4096, 3, "uniform"),         # largest K
    (3, 1, 2000, 4096, 17, "uniform"),        # tile bases of three problems read from global memory
    (3, 1, 130, 4, 0, "blocks"),              # w = 0 behaves as w = 1
    (1, 1, 4100, 3, 5000, "uniform"),         # w > n: no far keys at all
])
def test_index_bit_exact(fz, B, A, n, K, w, kind):
    import torch
    g = synth.draw_group_ids(100 + n, B, A, n, K, kind)
    p = fz.make_params(B=B, H=A, H_kv=A, n=n, d=64, D=64, d_g=32, K=K, A=A, w=w)
    ws = _ws(fz, p)
    idx = fz.focus_build_index(p, torch.from_numpy(g).cuda(), ws)
    assert fz.focus_check_errors(ws) == 0
    got = _index_np(fz, p, idx, ws)
    want = ref.build_index(g, K, max(w, 1))
    items = ref.work_items(want, fz.TILE_M)
    _check_index(got, want, items, ref.lpt_order(items, fz.TILE_N))
    assert idx.max_items >= len(items)


def test_bad_group_id_is_reported(fz):
    import torch
    g = synth.draw_group_ids(3, 1, 1, 100, 4, "uniform")
    g[0, 0, 17] = 4
    p = fz.make_params(B=1, H=1, H_kv=1, n=100, d=64, D=64, d_g=32, K=4, A=1, w=3)
    ws = _ws(fz, p)
    fz.focus_build_index(p, torch.from_numpy(g).cuda(), ws)
    assert fz.focus_check_errors(ws) == 6
    assert fz.focus_check_errors(ws) == 0      # cleared after the report


# --------------------------------------------------------------- attention ---

def _attn_case(fz, dtype, B, H, H_kv, A, n, d, K, w, kind, seed, dense=False):
    import torch
    rng = np.random.default_rng(seed)
    store = (lambda a: synth.round_bf16(a)) if dtype == "bf16" else (lambda a: a)
    Q = store(rng.standard_normal((B, H, n, d)).astype(np.float32))
    Kt = store(rng.standard_normal((B, H_kv, n, d)).astype(np.float32))
    V = store(rng.standard_normal((B, H_kv, n, d)).astype(np.float32))
    g = synth.draw_group_ids(seed, B, A, n, K, kind)
    p = fz.make_params(B=B, H=H, H_kv=H_kv, n=n, d=d, D=64, d_g=32, K=K, A=A, w=w, dtype=dtype)
    ws = _ws(fz, p)
    Qd, Kd, Vd = to_dev(Q, dtype), to_dev(Kt, dtype), to_dev(V, dtype)
    O = torch.full_like(Qd, float("nan"))
    lse = torch.full((B, H, n), float("nan"), dtype=torch.float32, device="cuda")
    if dense:
        fz.focus_dense_causal_fwd(p, Qd, Kd, Vd, O, lse, ws)
        want_O, want_L = ref.dense_causal(Q, Kt, V, p.scale)
    else:
        idx = fz.focus_build_index(p, torch.from_numpy(g).cuda(), ws)
        fz.focus_attention_fwd(p, Qd, Kd, Vd, idx, O, lse, ws)
        want_O, want_L = ref.attention(Q, Kt, V, g, w, p.scale, A)
    assert fz.focus_check_errors(ws) == 0
    assert_close(to_host(O), want_O, dtype, "O")
    assert_lse_close(lse.cpu().numpy(), want_L, dtype, "lse")


@pytest.mark.parametrize("dtype,B,H,H_kv,A,n,d,K,w,kind", [
    ("bf16", 1, 2, 2, 1, 300, 128, 4, 32, "uniform"),
    ("bf16", 2, 4, 2, 1, 513, 64, 8, 100, "zipf"),
    ("bf16", 1, 4, 2, 2, 1000, 128, 16, 128, "uniform"),    # one assignment per kv head
    ("bf16", 1, 2, 1, 1, 700, 128, 1, 40, "one"),          # K = 1: dense causal
    ("bf16", 1, 1, 1, 1, 384, 64, 384, 1, "distinct"),     # every row attends to itself only
    ("bf16", 1, 2, 2, 1, 1, 128, 3, 5, "uniform"),          # one token
    ("bf16", 1, 2, 2, 1, 257, 128, 5, 0, "uniform"),        # w = 0
    ("bf16", 1, 2, 2, 1, 600, 64, 6, 1000, "uniform"),      # w > n
    ("bf16", 1, 3, 1, 1, 2000, 128, 3, 129, "blocks"),
    ("bf16", 1, 8, 2, 2, 1500, 128, 32, 256, "zipf"),
    ("f32", 1, 2, 2, 1, 256, 64, 4, 32, "uniform"),
    ("f32", 1, 4, 2, 2, 333, 128, 5, 20, "zipf"),
    ("f32", 2, 2, 1, 1, 100, 64, 1, 7, "one"),
])
def test_attention_all_rows(fz, dtype, B, H, H_kv, A, n, d, K, w, kind):
    _attn_case(fz, dtype, B, H, H_kv, A, n, d, K, w, kind, seed=n + w + K)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 128)])
def test_attention_long_groups_deterministic(fz, dtype, d):
    """Two big groups: group-pass items walk up to ~16 key tiles, so the tile
    pipeline cycles its barriers many times; three runs must agree bit for bit
    and match the oracle on every row."""
    import torch
    B, H, H_kv, A, n, K, w = 1, 4, 2, 1, 4096, 2, 64
    rng = np.random.default_rng(77)
    store = (lambda a: synth.round_bf16(a)) if dtype == "bf16" else (lambda a: a)
    Q = store(rng.standard_normal((B, H, n, d)).astype(np.float32))
    Kt = store(rng.standard_normal((B, H_kv, n, d)).astype(np.float32))
    V = store(rng.standard_normal((B, H_kv, n, d)).astype(np.float32))
    g = synth.draw_group_ids(77, B, A, n, K, "uniform")
    p = fz.make_params(B=B, H=H, H_kv=H_kv, n=n, d=d, D=64, d_g=32, K=K, A=A, w=w, dtype=dtype)
    ws = _ws(fz, p)
    Qd, Kd, Vd = to_dev(Q, dtype), to_dev(Kt, dtype), to_dev(V, dtype)
    idx = fz.focus_build_index(p, torch.from_numpy(g).cuda(), ws)
    outs = []
    for _ in range(3):
        O = torch.full_like(Qd, float("nan"))
        fz.focus_attention_fwd(p, Qd, Kd, Vd, idx, O, None, ws)
        outs.append(O)
    assert fz.focus_check_errors(ws) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    want_O, _ = ref.attention(Q, Kt, V, g, w, p.scale, A)
    assert_close(to_host(outs[0]), want_O, dtype, "O")


@pytest.mark.parametrize("dtype,n,d,H,H_kv", [("bf16", 700, 128, 4, 2), ("bf16", 129, 64, 2, 2),
                                              ("f32", 300, 64, 2, 1)])
def test_dense_causal_all_rows(fz, dtype, n, d, H, H_kv):
    _attn_case(fz, dtype, 1, H, H_kv, 1, n, d, 1, 1, "one", seed=n, dense=True)


# ---------------------------------------------------------- full workloads ---

_SAMPLE = {  # name -> (heads to compare, random rows per head); None = all
    "tiny_fp32": (None, None),
    "gpt2_small_1k": (None, None),
    "llama7b_8k": ([0, 9, 31], 512),
    "gqa_32k": ([0, 5, 18, 31], 256),
    "llama70b_64k": ([0, 13, 37, 63], 128),
}


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_full_size(fz, name):
    import torch
    wl = synth.WORKLOADS[name]
    x = margin_filtered(wl)
    p = fz.params_from_workload(wl)
    ws = _ws(fz, p)
    dev = {k: to_dev(x[k], wl.dtype) for k in ("h", "W", "C", "Q", "K", "V")}
    O, gid, idx, lse = fz.run_layer(p, dev["h"], dev["W"], dev["C"], dev["Q"], dev["K"], dev["V"],
                                    ws, want_lse=True)
    assert fz.focus_check_errors(ws) == 0
    O2 = torch.empty_like(O)
    fz.focus_attention_fwd(p, dev["Q"], dev["K"], dev["V"], idx, O2, None, ws)
    assert fz.focus_check_errors(ws) == 0
    assert torch.equal(O, O2), "attention is not deterministic"
    g = gid.cpu().numpy()
    assert np.array_equal(g, x["gid_ref"]), "group ids"
    got_idx = _index_np(fz, p, idx, ws)
    want_idx = ref.build_index(x["gid_ref"], wl.K, max(wl.w, 1))
    items = ref.work_items(want_idx, fz.TILE_M)
    _check_index(got_idx, want_idx, items, ref.lpt_order(items, fz.TILE_N))
    heads, nrand = _SAMPLE[name]
    if heads is None:
        want_O, want_L = ref.attention(x["Q"], x["K"], x["V"], x["gid_ref"], wl.w, wl.scale, wl.A)
        assert_close(to_host(O), want_O, wl.dtype, name)
        assert_lse_close(lse.cpu().numpy(), want_L, wl.dtype, name)
        return
    for hq in heads:
        kv = ref.kv_head(hq, wl.H, wl.H_kv)
        a = ref.assignment_of_head(hq, wl.H, wl.H_kv, wl.A)
        rows = sample_rows(want_idx, 0, a, wl.n, wl.w, seed=hq, n_random=nrand)
        Oh, Lh = ref.attention_rows(x["Q"][:, hq:hq + 1], x["K"][:, kv:kv + 1], x["V"][:, kv:kv + 1],
                                    x["gid_ref"][:, a:a + 1], wl.w, wl.scale, rows, 1, row_block=256)
        got = to_host(O[0, hq, torch.from_numpy(rows).cuda()])
        assert_close(got, Oh[0, 0], wl.dtype, f"{name} head {hq}")
        assert_lse_close(lse[0, hq, torch.from_numpy(rows).cuda()].cpu().numpy(), Lh[0, 0], wl.dtype,
                         f"{name} head {hq}")


@pytest.mark.parametrize("shape", [
    dict(n=2048, H=8, H_kv=2, D=512),           # two KV-head chunks
    dict(n=1024, H=16, H_kv=8, D=512),          # eight chunks
    dict(B=2, n=1024, H=8, H_kv=2, D=512),      # B = 2: one chunk
])
def test_layer_from_host_buffers_matches_device_path(fz, shape):
    """focus_layer_fwd_host (copies overlapped with compute in KV-head chunks
    when B = 1 and A = 1) gives the device path's O bit for bit."""
    import torch
    wl = synth.workload("gqa_32k", **shape)
    x = margin_filtered(wl)
    p = fz.params_from_workload(wl)
    ws = _ws(fz, p)
    dev = {k: to_dev(x[k], wl.dtype) for k in ("h", "W", "C", "Q", "K", "V")}
    O_dev, _, _, _ = fz.run_layer(p, dev["h"], dev["W"], dev["C"], dev["Q"], dev["K"], dev["V"], ws)
    host = {k: dev[k].cpu().pin_memory() for k in dev}
    host["O"] = torch.empty(O_dev.shape, dtype=O_dev.dtype).pin_memory()
    dbuf = {k: torch.empty_like(dev[k]) for k in dev}
    dbuf["O"] = torch.empty_like(O_dev)
    dbuf["gid"] = torch.empty((p.B, p.A, p.n), dtype=torch.int32, device="cuda")
    fz.focus_layer_fwd_host(p, host, dbuf, ws)
    assert fz.focus_check_errors(ws) == 0
    assert torch.equal(host["O"], O_dev.cpu())


def test_attention_at_the_largest_supported_length(fz):
    """n = FOCUS_MAX_N (2^20 tokens, the pages' 1M-token setting): 16 uniform
    groups of ~65K tokens give group-pass units of up to ~512 key tiles.
    Index bit-exact; O and LSE on sampled rows (window start, first far row of
    each group, the smallest groups' rows, random rows); a bitwise re-run."""
    import torch
    B, H, H_kv, A, n, d, K, w = 1, 2, 1, 1, 1 << 20, 64, 16, 1024
    rng = np.random.default_rng(2024)
    Q = synth.round_bf16(rng.standard_normal((B, H, n, d), dtype=np.float32))
    Kt = synth.round_bf16(rng.standard_normal((B, H_kv, n, d), dtype=np.float32))
    V = synth.round_bf16(rng.standard_normal((B, H_kv, n, d), dtype=np.float32))
    g = synth.draw_group_ids(2024, B, A, n, K, "uniform")
    p = fz.make_params(B=B, H=H, H_kv=H_kv, n=n, d=d, D=64, d_g=32, K=K, A=A, w=w)
    ws = _ws(fz, p)
    Qd, Kd, Vd = to_dev(Q, "bf16"), to_dev(Kt, "bf16"), to_dev(V, "bf16")
    idx = fz.focus_build_index(p, torch.from_numpy(g).cuda(), ws)
    O = torch.empty_like(Qd)
    lse = torch.empty((B, H, n), dtype=torch.float32, device="cuda")
    fz.focus_attention_fwd(p, Qd, Kd, Vd, idx, O, lse, ws)
    O2 = torch.empty_like(Qd)
    fz.focus_attention_fwd(p, Qd, Kd, Vd, idx, O2, None, ws)
    assert fz.focus_check_errors(ws) == 0
    assert torch.equal(O, O2), "attention is not deterministic"
    want_idx = ref.build_index(g, K, w)
    items = ref.work_items(want_idx, fz.TILE_M)
    _check_index(_index_np(fz, p, idx, ws), want_idx, items, ref.lpt_order(items, fz.TILE_N))
    # the oracle scores every row against all 2^20 keys: keep the sample small
    perm, offs, fs = want_idx["perm"][0, 0], want_idx["offsets"][0, 0], want_idx["farlen_slot"][0, 0]
    first_far = []
    for gi in range(K):
        seg = np.arange(offs[gi], offs[gi + 1])
        far = seg[fs[seg] > 0]
        if len(far):
            first_far.append(int(perm[far[0]]))
    rows = np.array(sorted(set(range(64)) | set(range(w - 8, w + 8)) | set(first_far) | {n - 1} |
                           set(int(v) for v in rng.integers(0, n, 32))), dtype=np.int64)
    for hq in range(H):
        Oh, Lh = ref.attention_rows(Q[:, hq:hq + 1], Kt, V, g, w, p.scale, rows, 1, row_block=64)
        sel = torch.from_numpy(rows).cuda()
        assert_close(to_host(O[0, hq, sel]), Oh[0, 0], "bf16", f"n=2^20 head {hq}")
        assert_lse_close(lse[0, hq, sel].cpu().numpy(), Lh[0, 0], "bf16", f"n=2^20 head {hq}")
