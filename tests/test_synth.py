"""Seeded input generators: determinism, dtype grid, shapes."""
import pytest
import numpy as np
import torch

from learned_group_sparse_focus_gb300 import synth


def test_round_bf16_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 37.0
    x[:4] = [0.0, -0.0, 1e-30, 3.0e38]
    ours = synth.round_bf16(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, theirs)
    bits = synth.bf16_bits(ours)
    back = torch.from_numpy(bits).view(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(back, ours)


def test_draw_is_deterministic_and_shaped():
    wl = synth.workload("gpt2_small_1k", B=2, n=64)
    a = synth.draw(wl)
    b = synth.draw(wl)
    for k in ("h", "W", "C", "Q", "K", "V"):
        assert np.array_equal(a[k], b[k])
        assert np.array_equal(a[k], synth.round_bf16(a[k]))
    assert a["h"].shape == (2, 64, 768) and a["W"].shape == (1, 64, 768)
    assert a["C"].shape == (1, 16, 64) and a["Q"].shape == (2, 12, 64, 64)
    np.testing.assert_allclose(np.linalg.norm(a["C"][0].astype(np.float64), axis=1), 1.0, atol=1e-2)
    # drawing attention inputs alone gives the same tensors
    c = synth.draw(wl, parts=("attn",))
    assert np.array_equal(c["Q"], a["Q"]) and "h" not in c


def test_zipf_targets_are_skewed():
    wl = synth.workload("gqa_32k", n=8192)
    t = synth._zipf_targets(wl)
    frac = np.bincount(t.ravel(), minlength=wl.K).max() / t.size
    assert 0.18 < frac < 0.32


def test_redraw_changes_only_chosen_tokens():
    wl = synth.workload("llama7b_8k", n=128, D=256)
    x = synth.draw(wl, parts=("assign",))
    h0 = x["h"].copy()
    synth.redraw_hidden(wl, x, np.array([[0, 3], [0, 77]]), attempt=1)
    changed = np.any(x["h"] != h0, axis=2)
    assert changed[0, 3] and changed[0, 77] and changed.sum() == 2


def test_topk_group_ids_are_distinct_seeded_and_shaped():
    for kind in ("uniform", "zipf"):
        g = synth.draw_group_ids_topk(5, 2, 3, 500, 6, 2, kind)
        assert g.shape == (2, 3, 500, 2) and g.dtype == np.int32
        assert np.all(g[..., 0] != g[..., 1])
        assert g.min() >= 0 and g.max() < 6
        assert np.array_equal(g, synth.draw_group_ids_topk(5, 2, 3, 500, 6, 2, kind))
        assert not np.array_equal(g, synth.draw_group_ids_topk(6, 2, 3, 500, 6, 2, kind))
    g3 = synth.draw_group_ids_topk(1, 1, 1, 200, 5, 3, "uniform")
    assert all(len(set(r.tolist())) == 3 for r in g3[0, 0])


def test_topk_group_id_kinds():
    u = synth.draw_group_ids_topk(2, 1, 1, 60000, 4, 2, "uniform")
    counts = np.bincount(u.ravel(), minlength=4)
    assert np.all(np.abs(counts / counts.sum() - 0.25) < 0.01)          # balanced memberships
    pairs = np.bincount((np.minimum(u[..., 0], u[..., 1]) * 4 + np.maximum(u[..., 0], u[..., 1])).ravel())
    assert np.count_nonzero(pairs) == 6                                  # every pair of groups occurs
    z = synth.draw_group_ids_topk(2, 1, 1, 60000, 8, 2, "zipf")
    zc = np.bincount(z.ravel(), minlength=8)
    assert zc[0] > zc[3] > zc[7]                                         # skewed toward low ids
    b = synth.draw_group_ids_topk(3, 1, 2, 100, 5, 2, "both")
    assert np.array_equal(np.sort(b, axis=-1), np.broadcast_to([0, 1], b.shape))
    with pytest.raises(ValueError):
        synth.draw_group_ids_topk(3, 1, 1, 10, 5, 3, "both")
    with pytest.raises(ValueError):
        synth.draw_group_ids_topk(3, 1, 1, 10, 2, 3, "uniform")
