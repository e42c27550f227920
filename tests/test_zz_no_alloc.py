"""focus_build_index_static: the index built with no workspace and no
allocation, against the CPU oracle's index and against focus_build_index on
the same inputs.

Every output is integer work, so the comparison is bit for bit (tolerance 0).
The GPU cases make two calls in a row (different group ids, then the first
ones again) so that leftovers in the shared fixed scratch would show; one case
needs 99% of the fixed scratch, so its far end is written and read too.  The
size and argument checks run before anything touches the device and are
tested on the CPU.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle.focus_ref as ref
from learned_group_sparse_focus_gb300 import synth

FOCUS_ERR_INVALID_ARG = 1
FOCUS_ERR_WORKSPACE = 3
FOCUS_ERR_BAD_GROUP_ID = 6
SCRATCH_BYTES = 1 << 20


@pytest.fixture(scope="module")
def fz():
    from learned_group_sparse_focus_gb300 import _build
    if not os.path.exists(_build.LIB):
        _build.build()
    from learned_group_sparse_focus_gb300 import focus
    return focus


def _fake_index(fz, max_items):
    """An Index of aligned, never-dereferenced addresses (the calls below fail
    their checks before any device access)."""
    idx = fz.Index()
    for k, name in enumerate(("counts", "offsets", "perm", "rank", "farlen_tok", "farlen_slot",
                              "items", "order", "n_items")):
        setattr(idx, name, 0x100000 * (k + 1))
    idx.max_items = max_items
    return idx


def _call_raw(fz, p, idx, err=0x4000000, gid=0x8000000):
    return fz.lib().focus_build_index_static(ctypes.byref(p), gid, ctypes.byref(idx), err, None)


def _needed(p):
    P, n, K = p.B * p.A, p.n, p.K
    nseg = -(-n // 1024)
    m = P * (-(-n // 128) + min(K, n))
    up = lambda x: -(-x // 256) * 256
    return up(up(up(P * nseg * K * 4) + P * (K + 1) * 4) + m * 4), m


def test_static_index_rejects_oversized_problem(fz):
    p = fz.make_params(B=1, H=1, H_kv=1, n=1 << 20, d=64, D=64, d_g=32, K=4096, A=1, w=64)
    need, m = _needed(p)
    assert need > SCRATCH_BYTES
    assert _call_raw(fz, p, _fake_index(fz, m)) == FOCUS_ERR_WORKSPACE


def test_static_index_largest_accepted_size_is_the_stated_limit(fz):
    # n = 64 Ki, K = 1024: 64 segments x 1024 groups of histograms = 256 KiB,
    # inside the limit; K = 4096 needs 1 MiB of histograms plus the rest: out.
    p_in = fz.make_params(B=1, H=1, H_kv=1, n=1 << 16, d=64, D=64, d_g=32, K=1024, A=1, w=64)
    p_out = fz.make_params(B=1, H=1, H_kv=1, n=1 << 16, d=64, D=64, d_g=32, K=4096, A=1, w=64)
    assert _needed(p_in)[0] <= SCRATCH_BYTES < _needed(p_out)[0]
    assert _call_raw(fz, p_out, _fake_index(fz, _needed(p_out)[1])) == FOCUS_ERR_WORKSPACE


def test_static_index_argument_checks(fz):
    p = fz.make_params(B=1, H=1, H_kv=1, n=1000, d=64, D=64, d_g=32, K=8, A=1, w=16)
    _, m = _needed(p)
    assert _call_raw(fz, p, _fake_index(fz, m - 1)) == FOCUS_ERR_INVALID_ARG      # capacity
    assert _call_raw(fz, p, _fake_index(fz, m), err=0x4000010) == FOCUS_ERR_INVALID_ARG  # err alignment
    assert _call_raw(fz, p, _fake_index(fz, m), gid=0) == FOCUS_ERR_INVALID_ARG
    bad = _fake_index(fz, m)
    bad.perm = 0x100004
    assert _call_raw(fz, p, bad) == FOCUS_ERR_INVALID_ARG
    q = fz.make_params(B=1, H=1, H_kv=1, n=1000, d=64, D=64, d_g=32, K=0, A=1, w=16)
    assert _call_raw(fz, q, _fake_index(fz, m)) == FOCUS_ERR_INVALID_ARG


def _arrays(fz, p, idx, views):
    import torch
    n_items = int(views["n_items"].item())
    out = {k: views[k].cpu().numpy().copy()
           for k in ("counts", "offsets", "perm", "rank", "farlen_tok", "farlen_slot")}
    out["items"] = views["items"][:n_items].cpu().numpy().copy()
    out["order"] = views["order"][:n_items].cpu().numpy().copy()
    out["n_items"] = n_items
    torch.cuda.synchronize()
    return out


def _regular(fz, p, gid_dev):
    ws = fz.alloc_workspace(p)
    idx = fz.focus_build_index(p, gid_dev, ws)
    assert fz.focus_check_errors(ws) == 0
    return idx, ws, _arrays(fz, p, idx, fz.index_views(p, idx, ws))


def _static(fz, p, gid_dev, bufs):
    idx = fz.focus_build_index_static(p, gid_dev, bufs)
    assert fz.focus_check_errors(bufs["err"]) == 0
    return idx, _arrays(fz, p, idx, bufs)


def _same(a, b):
    assert a["n_items"] == b["n_items"]
    for k in ("counts", "offsets", "perm", "rank", "farlen_tok", "farlen_slot", "items", "order"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def _oracle(fz, gid, K, w):
    """The CPU oracle's index, work list and longest-first order for gid."""
    want = ref.build_index(gid, K, max(w, 1))
    items = ref.work_items(want, fz.TILE_M)
    out = {k: want[k] for k in ("counts", "offsets", "perm", "rank", "farlen_tok", "farlen_slot")}
    out["items"] = items
    out["order"] = ref.lpt_order(items, fz.TILE_N)
    out["n_items"] = len(items)
    return out


def _same_as_oracle(got, want):
    assert got["n_items"] == want["n_items"]
    for k in ("counts", "offsets", "perm", "rank", "farlen_tok", "farlen_slot"):
        np.testing.assert_array_equal(got[k].reshape(want[k].shape), want[k], err_msg=k)
    np.testing.assert_array_equal(got["items"][:, :7], want["items"], err_msg="items")
    np.testing.assert_array_equal(got["order"], want["order"], err_msg="order")


@pytest.mark.gpu
@pytest.mark.parametrize("wl_name,kind", [("llama7b_8k", "zipf"), ("llama70b_64k", "uniform"),
                                          ("gpt2_small_1k", "blocks")])
def test_static_index_matches_workspace_index_twice(fz, wl_name, kind):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    wl = synth.WORKLOADS[wl_name]
    p = fz.params_from_workload(wl)
    bufs = fz.index_buffers(p)
    g1 = torch.from_numpy(synth.draw_group_ids(wl.seed, wl.B, wl.A, wl.n, wl.K, kind)).cuda()
    g2 = torch.from_numpy(synth.draw_group_ids(wl.seed + 7, wl.B, wl.A, wl.n, wl.K, "uniform")).cuda()
    _, _, want1 = _regular(fz, p, g1)
    _, _, want2 = _regular(fz, p, g2)
    ora1 = _oracle(fz, g1.cpu().numpy(), wl.K, wl.w)
    ora2 = _oracle(fz, g2.cpu().numpy(), wl.K, wl.w)
    for gid, want, ora in ((g1, want1, ora1), (g2, want2, ora2), (g1, want1, ora1)):
        idx, got = _static(fz, p, gid, bufs)
        _same(got, want)
        _same_as_oracle(got, ora)
        assert idx.max_items == bufs["order"].numel()
        assert idx.w_eff == max(wl.w, 1)


def test_static_index_near_limit_case_fits(fz):
    # the GPU case below needs 99% of the fixed scratch; ten more groups do not fit
    p = fz.make_params(B=1, H=1, H_kv=1, n=1 << 18, d=64, D=64, d_g=32, K=1000, A=1, w=64)
    q = fz.make_params(B=1, H=1, H_kv=1, n=1 << 18, d=64, D=64, d_g=32, K=1010, A=1, w=64)
    assert 0.99 * SCRATCH_BYTES <= _needed(p)[0] <= SCRATCH_BYTES < _needed(q)[0]
    assert _call_raw(fz, q, _fake_index(fz, _needed(q)[1])) == FOCUS_ERR_WORKSPACE


@pytest.mark.gpu
def test_static_index_near_the_scratch_limit_twice(fz):
    """n = 2^18 tokens in K = 1000 groups: the histograms, tile bases and item
    costs fill 1,040,384 of the 1,048,576 scratch bytes."""
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    n, K, w = 1 << 18, 1000, 64
    p = fz.make_params(B=1, H=1, H_kv=1, n=n, d=64, D=64, d_g=32, K=K, A=1, w=w)
    assert _needed(p)[0] >= 0.99 * SCRATCH_BYTES
    bufs = fz.index_buffers(p)
    g1 = synth.draw_group_ids(41, 1, 1, n, K, "uniform")
    g2 = synth.draw_group_ids(42, 1, 1, n, K, "zipf")
    ora1, ora2 = _oracle(fz, g1, K, w), _oracle(fz, g2, K, w)
    for g, ora in ((g1, ora1), (g2, ora2), (g1, ora1)):
        _, got = _static(fz, p, torch.from_numpy(g).cuda(), bufs)
        _same_as_oracle(got, ora)


@pytest.mark.gpu
def test_static_index_feeds_attention_like_the_workspace_index(fz):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    wl = synth.workload("gqa_32k", n=3000)
    p = fz.params_from_workload(wl)
    x = synth.draw(wl, parts=("attn",))
    from _helpers import to_dev
    Q, K, V = (to_dev(x[k], "bf16") for k in ("Q", "K", "V"))
    gid = torch.from_numpy(synth.draw_group_ids(wl.seed, wl.B, wl.A, wl.n, wl.K, "zipf")).cuda()
    idx_ws, ws, _ = _regular(fz, p, gid)
    O1 = torch.empty_like(Q)
    fz.focus_attention_fwd(p, Q, K, V, idx_ws, O1, None, ws)
    bufs = fz.index_buffers(p)
    for _ in range(2):
        idx_st, _ = _static(fz, p, gid, bufs)
        O2 = torch.empty_like(Q)
        fz.focus_attention_fwd(p, Q, K, V, idx_st, O2, None, ws)
        assert fz.focus_check_errors(ws) == 0
        assert torch.equal(O1, O2)


@pytest.mark.gpu
def test_static_index_reports_bad_group_id(fz):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g = synth.draw_group_ids(3, 1, 1, 100, 4, "uniform")
    g[0, 0, 17] = 4
    p = fz.make_params(B=1, H=1, H_kv=1, n=100, d=64, D=64, d_g=32, K=4, A=1, w=3)
    bufs = fz.index_buffers(p)
    fz.focus_build_index_static(p, torch.from_numpy(g).cuda(), bufs)
    assert fz.focus_check_errors(bufs["err"]) == FOCUS_ERR_BAD_GROUP_ID
    assert fz.focus_check_errors(bufs["err"]) == 0
