"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a hand-worked example, a closed form, a
special case that reduces to a textbook routine, brute force on tiny inputs or
an invariant the method fixes, so that a dropped term, a wrong sign or index
or a transposed operand in the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle.focus_ref as ref
from learned_group_sparse_focus_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_golden(name):
    out = {"kept": {}, "item": [], "O": {}}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split(":", 1)
            vals = val.split()
            if key.startswith("kept "):
                out["kept"][int(key.split()[1])] = [int(v) for v in vals]
            elif key == "item":
                out["item"].append([int(v) for v in vals])
            elif key.startswith("O") and key[1:].isdigit():
                out["O"][int(key[1:])] = [float(v) for v in vals]
            else:
                out[key] = [float(v) if "." in v else int(v) for v in vals]
    return out


# ------------------------------------------------------------ golden case ---

def test_golden_keep_rule_index_and_softmax():
    gd = _parse_golden("keep_rule_n8.txt")
    n, w, K = gd["n"][0], gd["w"][0], gd["K"][0]
    g = np.array(gd["groups"], np.int32)
    M = ref.keep_mask(g, w)
    for i in range(n):
        assert list(np.nonzero(M[i])[0]) == gd["kept"][i], i
    idx = ref.build_index(g[None, None, :], K, w)
    for key in ("counts", "offsets", "perm", "rank", "farlen_tok", "farlen_slot"):
        assert idx[key][0, 0].tolist() == gd[key], key
    items = ref.work_items(idx, gd["BM"][0])
    assert items.tolist() == gd["item"]
    assert ref.lpt_order(items, gd["BN"][0]).tolist() == gd["lpt"]
    kc = ref.kept_counts(idx, w)[0, 0]
    assert kc.tolist() == gd["lse_count"]
    # exact softmax with all-zero scores
    Q = np.zeros((1, 1, n, 2))
    Kt = np.random.default_rng(0).standard_normal((1, 1, n, 2))
    V = np.stack([np.arange(n, dtype=np.float64), np.ones(n)], axis=1)[None, None]
    O, L = ref.attention(Q, Kt, V, g[None, None, :], w, 0.7, 1)
    for i in range(n):
        np.testing.assert_allclose(O[0, 0, i], gd["O"][i], rtol=0, atol=1e-14)
    np.testing.assert_allclose(L[0, 0], np.log(np.array(gd["lse_count"], float)), atol=1e-14)


# ----------------------------------------------------------------- assign ---

def test_assign_closed_form_signed_basis_and_ties():
    # W = I, C = signed basis vectors: the score of centroid k is a signed
    # coordinate of h, so the group is the largest signed coordinate; the
    # duplicate of e0 (index 4) never wins over index 0.
    d = 4
    W = np.eye(d)[None]
    C = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [-1, 0, 0, 0], [0, 0, 1, 0], [1, 0, 0, 0]], float)[None]
    h = np.array([[[3, -1, 0.5, 2], [-2, 1, 0, 0], [0.1, 0.2, 0.3, 0], [-1, -1, -1, -1]]], float)
    gid, margin = ref.assign(h, W, C)
    # scores: row0 [3,-1,-3,.5,3] -> 0 (tie with 4); row1 [-2,1,2,0,-2] -> 2;
    # row2 [.1,.2,-.1,.3,.1] -> 3; row3 [-1,-1,1,-1,-1] -> 2
    assert gid[0, 0].tolist() == [0, 2, 3, 2]
    np.testing.assert_allclose(margin[0, 0], [0.0, 1.0, 0.1, 2.0], atol=1e-15)


def test_assign_bruteforce_loops():
    rng = np.random.default_rng(1)
    B, n, D, A, dg, K = 2, 9, 7, 2, 5, 6
    h = rng.standard_normal((B, n, D))
    W = rng.standard_normal((A, dg, D))
    C = rng.standard_normal((A, K, dg))
    gid, margin = ref.assign(h, W, C)
    for b in range(B):
        for a in range(A):
            for i in range(n):
                p = [math.fsum(W[a, r, c] * h[b, i, c] for c in range(D)) for r in range(dg)]
                s = [math.fsum(p[r] * C[a, k, r] for r in range(dg)) for k in range(K)]
                best = 0
                for k in range(1, K):
                    if s[k] > s[best]:
                        best = k
                assert gid[b, a, i] == best
                srt = sorted(s)
                assert abs(margin[b, a, i] - (srt[-1] - srt[-2])) < 1e-12


def test_assign_centroid_permutation_relabels():
    rng = np.random.default_rng(2)
    h = rng.standard_normal((1, 200, 16))
    W = rng.standard_normal((1, 8, 16))
    C = rng.standard_normal((1, 10, 8))
    pi = rng.permutation(10)
    g1, _ = ref.assign(h, W, C)
    g2, _ = ref.assign(h, W, C[:, pi])     # centroid k of the new set is old pi[k]
    assert np.array_equal(pi[g2], g1)


def test_assign_depends_on_projection_not_raw_h():
    # with a projection that zeroes all but one hidden coordinate, only that
    # coordinate decides: transposing W would break this.
    h = np.array([[[5.0, -3.0, 0.0], [-5.0, 3.0, 0.0]]])
    W = np.array([[[0.0, 1.0, 0.0], [0.0, 0.0, 0.0]]])        # d_g=2, D=3: p = (h1, 0)
    C = np.array([[[1.0, 0.0], [-1.0, 0.0]]])
    gid, _ = ref.assign(h, W, C)
    assert gid[0, 0].tolist() == [1, 0]


# ------------------------------------------------------------------ index ---

@pytest.mark.parametrize("kind,K,n,w", [
    ("uniform", 5, 300, 7), ("zipf", 16, 512, 33), ("one", 1, 100, 10),
    ("blocks", 8, 256, 4), ("distinct", 64, 64, 1), ("uniform", 3, 50, 0),
    ("uniform", 40, 90, 200),
])
def test_index_invariants_and_bruteforce(kind, K, n, w):
    g = synth.draw_group_ids(7, 2, 2, n, K, kind)
    idx = ref.build_index(g, K, w)
    for b in range(2):
        for a in range(2):
            gg = g[b, a]
            perm, rank = idx["perm"][b, a], idx["rank"][b, a]
            assert idx["counts"][b, a].sum() == n
            assert sorted(perm.tolist()) == list(range(n))
            assert np.array_equal(rank[perm], np.arange(n))
            assert np.all(np.diff(gg[perm]) >= 0)
            for k in range(K):
                o0, o1 = idx["offsets"][b, a, k], idx["offsets"][b, a, k + 1]
                assert o1 - o0 == np.sum(gg == k)
                assert np.all(np.diff(perm[o0:o1]) > 0)
            for i in range(n):
                bf = sum(1 for j in range(n) if gg[j] == gg[i] and j <= i - w)
                assert idx["farlen_tok"][b, a, i] == bf
                assert idx["farlen_slot"][b, a, rank[i]] == bf


@pytest.mark.parametrize("K,n,w", [(4, 200, 9), (13, 333, 1), (2, 64, 64), (30, 257, 16)])
def test_kept_count_three_ways(K, n, w):
    g = synth.draw_group_ids(11, 1, 1, n, K, "uniform")
    idx = ref.build_index(g, K, w)
    total = int(ref.kept_counts(idx, w).sum())
    pop = int(ref.keep_mask(g[0, 0], w).sum())
    # inclusion-exclusion: window pairs + same-group causal pairs - same-group window pairs
    win = sum(min(i + 1, w) for i in range(n))
    cnt = np.bincount(g[0, 0], minlength=K)
    same = int(sum(c * (c + 1) // 2 for c in cnt))
    overlap = sum(1 for i in range(n) for j in range(max(0, i - w + 1), i + 1) if g[0, 0, i] == g[0, 0, j])
    assert total == pop == win + same - overlap


def test_work_items_cover_exactly_far_rows():
    g = synth.draw_group_ids(5, 2, 3, 700, 9, "zipf")
    w, BM = 40, 32
    idx = ref.build_index(g, 9, w)
    items = ref.work_items(idx, BM)
    cover = np.zeros((2, 3, 700), int)
    prev = None
    for b, a, k, row0, rows, keys, key0 in items:
        key = (b, a, k, row0)
        assert prev is None or key > prev
        prev = key
        assert 1 <= rows <= BM and key0 == idx["offsets"][b, a, k]
        assert row0 + rows <= idx["offsets"][b, a, k + 1]
        fs = idx["farlen_slot"][b, a, row0:row0 + rows]
        assert keys == fs.max() > 0
        assert keys <= row0 + rows - key0 - 1 + 1
        cover[b, a, row0:row0 + rows] += 1
    far = idx["farlen_slot"] > 0
    assert np.all(cover[far] == 1) and cover.max() <= 1
    order = ref.lpt_order(items, 64)
    assert sorted(order.tolist()) == list(range(len(items)))
    tiles = (items[order, 5] + 63) // 64
    assert np.all(np.diff(tiles) <= 0)


# -------------------------------------------------------------- attention ---

def _sdpa_causal(Q, K, V, scale):
    H, Hkv = Q.shape[1], K.shape[1]
    Kt = torch.from_numpy(np.repeat(K, H // Hkv, axis=1))
    Vt = torch.from_numpy(np.repeat(V, H // Hkv, axis=1))
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q), Kt, Vt, is_causal=True, scale=scale).numpy()


@pytest.mark.parametrize("mode", ["K1", "wide_window"])
def test_reduces_to_dense_causal_sdpa(mode):
    rng = np.random.default_rng(3)
    B, H, Hkv, n, d = 2, 4, 2, 97, 16
    Q = rng.standard_normal((B, H, n, d))
    K = rng.standard_normal((B, Hkv, n, d))
    V = rng.standard_normal((B, Hkv, n, d))
    if mode == "K1":
        g, w = np.zeros((B, 1, n), np.int32), 5
    else:
        g, w = synth.draw_group_ids(1, B, 1, n, 7, "uniform"), n
    O, L = ref.attention(Q, K, V, g, w, 0.3, 1)
    np.testing.assert_allclose(O, _sdpa_causal(Q, K, V, 0.3), atol=1e-12)
    O2, _ = ref.dense_causal(Q, K, V, 0.3)
    np.testing.assert_allclose(O2, O, atol=1e-13)


def test_distinct_groups_window_one_is_identity_on_v():
    rng = np.random.default_rng(4)
    n, d = 64, 8
    Q, K, V = (rng.standard_normal((1, 1, n, d)) for _ in range(3))
    g = synth.draw_group_ids(2, 1, 1, n, n, "distinct")
    O, L = ref.attention(Q, K, V, g, 1, 0.5, 1)
    assert np.array_equal(O[0, 0], V[0, 0])
    np.testing.assert_allclose(L[0, 0], 0.5 * np.sum(Q[0, 0] * K[0, 0], axis=1), atol=1e-14)


def test_group_relabelling_leaves_output_unchanged():
    rng = np.random.default_rng(5)
    n, d, K = 150, 12, 6
    Q, Kt, V = (rng.standard_normal((1, 2, n, d)) for _ in range(3))
    g = synth.draw_group_ids(3, 1, 1, n, K, "uniform")
    pi = rng.permutation(K)
    O1, L1 = ref.attention(Q, Kt, V, g, 10, 0.4, 1)
    O2, L2 = ref.attention(Q, Kt, V, pi[g].astype(np.int32), 10, 0.4, 1)
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(L1, L2, atol=1e-12)


def test_weights_sum_to_one_and_vanish_off_mask():
    rng = np.random.default_rng(6)
    n, d = 120, 10
    Q, K = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    g = synth.draw_group_ids(4, 1, 1, n, 5, "uniform")[0, 0]
    M = ref.keep_mask(g, 9)
    P = ref.attention_weights_rows(Q, K, M, np.arange(n), 0.3)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(P[~M] == 0) and np.all(P[M] > 0)


@pytest.mark.parametrize("n,w,K,kind", [(64, 4, 3, "uniform"), (40, 1, 40, "distinct"),
                                        (33, 0, 5, "uniform"), (50, 64, 2, "uniform"),
                                        (64, 8, 1, "one"), (17, 3, 4, "blocks")])
def test_bruteforce_small(n, w, K, kind):
    rng = np.random.default_rng(n * 100 + w)
    d = 6
    Q, Kt, V = (rng.standard_normal((1, 1, n, d)) for _ in range(3))
    g = synth.draw_group_ids(n + w, 1, 1, n, K, kind)
    O, L = ref.attention(Q, Kt, V, g, w, 0.45, 1)
    Ob, Lb = ref.attention_bruteforce(Q[0, 0], Kt[0, 0], V[0, 0], g[0, 0], w, 0.45)
    np.testing.assert_allclose(O[0, 0], np.array(Ob), atol=1e-12)
    np.testing.assert_allclose(L[0, 0], np.array(Lb), atol=1e-12)


def test_local_plus_far_merge_equals_union():
    # The two-call decomposition: window-only and far-only (j <= i - w, same
    # group) partials merged by log-sum-exp equal one softmax over the union.
    rng = np.random.default_rng(8)
    n, d, w = 200, 8, 13
    Q, K, V = (rng.standard_normal((n, d)) for _ in range(3))
    g = synth.draw_group_ids(9, 1, 1, n, 4, "uniform")[0, 0]
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    local = (j <= i) & (i - j < w)
    far = (j <= i - w) & (g[:, None] == g[None, :])
    assert not np.any(local & far)
    rows = np.arange(n)
    O1, L1 = ref.attention_masked_rows(Q, K, V, local, rows, 0.35)
    O2, L2 = ref.attention_masked_rows(Q, K, V, far, rows, 0.35)
    Om, Lm = ref.lse_merge(O1, L1, O2, L2)
    Ou, Lu = ref.attention_masked_rows(Q, K, V, ref.keep_mask(g, w), rows, 0.35)
    np.testing.assert_allclose(Om, Ou, atol=1e-12)
    np.testing.assert_allclose(Lm, Lu, atol=1e-12)
    assert np.any(~np.isfinite(L2))     # some rows have no far keys: merge must skip them


def test_window_zero_equals_window_one():
    g = synth.draw_group_ids(12, 1, 1, 80, 6, "uniform")[0, 0]
    assert np.array_equal(ref.keep_mask(g, 0), ref.keep_mask(g, 1))


def test_gqa_head_map_and_assignment_per_kv_head():
    rng = np.random.default_rng(10)
    B, H, Hkv, n, d = 1, 6, 3, 40, 4
    Q = rng.standard_normal((B, H, n, d))
    K = rng.standard_normal((B, Hkv, n, d))
    V = rng.standard_normal((B, Hkv, n, d))
    g = synth.draw_group_ids(13, B, Hkv, n, 4, "uniform")
    O, _ = ref.attention(Q, K, V, g, 5, 0.5, Hkv)
    K2, V2 = K.copy(), V.copy()
    K2[:, 2] += 3.0
    V2[:, 2] -= 1.0
    g2 = g.copy()
    g2[:, 2] = (g2[:, 2] + 1) % 4 * 0       # change kv head 2's assignment only
    O2, _ = ref.attention(Q, K2, V2, g2, 5, 0.5, Hkv)
    np.testing.assert_array_equal(O[:, :4], O2[:, :4])           # heads 0..3 -> kv 0, 1
    assert not np.allclose(O[:, 4:], O2[:, 4:])
    # each query head equals single-head attention with its own kv head and ids
    for hq in range(H):
        kv = hq * Hkv // H
        Os, _ = ref.attention(Q[:, hq:hq + 1], K[:, kv:kv + 1], V[:, kv:kv + 1],
                              g[:, kv:kv + 1], 5, 0.5, 1)
        np.testing.assert_array_equal(Os[:, 0], O[:, hq])


def test_scale_enters_as_product_with_q():
    rng = np.random.default_rng(11)
    Q, K, V = (rng.standard_normal((1, 1, 60, 8)) for _ in range(3))
    g = synth.draw_group_ids(14, 1, 1, 60, 3, "uniform")
    O1, _ = ref.attention(Q, K, V, g, 7, 0.25, 1)
    O2, _ = ref.attention(Q * 0.25, K, V, g, 7, 1.0, 1)
    np.testing.assert_allclose(O1, O2, atol=1e-13)


def test_row_sampling_matches_full():
    rng = np.random.default_rng(12)
    B, H, n, d = 1, 2, 300, 8
    Q, K, V = (rng.standard_normal((B, H, n, d)) for _ in range(3))
    g = synth.draw_group_ids(15, B, 1, n, 5, "zipf")
    O, L = ref.attention(Q, K, V, g, 17, 0.3, 1)
    rows = np.array([0, 5, 77, 299, 150])
    Os, Ls = ref.attention_rows(Q, K, V, g, 17, 0.3, rows, 1, row_block=2)
    np.testing.assert_allclose(Os, O[:, :, rows], atol=1e-14)   # BLAS blocking only
    np.testing.assert_allclose(Ls, L[:, :, rows], atol=1e-14)


# ------------------------------------------------------------------ top-k ---

def _golden_top2():
    gd = _parse_golden("keep_rule_top2_n8.txt")
    n = gd["n"][0]
    G = np.array([gd["groups %d" % i] for i in range(n)], np.int32)
    return gd, G


def test_golden_top2_keep_rule_index_and_softmax():
    gd, G = _golden_top2()
    n, w, K = gd["n"][0], gd["w"][0], gd["K"][0]
    M = ref.keep_mask_rows_topk(G, w, np.arange(n))
    for i in range(n):
        assert list(np.nonzero(M[i])[0]) == gd["kept"][i], i
    idx = ref.build_index_topk(G[None, None], K, w)
    for key in ("counts", "offsets", "perm", "rank", "farlen_slot", "farlen_entry", "other"):
        assert idx[key][0, 0].tolist() == gd[key], key
    far_total = int(idx["farlen_slot"].sum())
    assert far_total == gd["far_total"][0]
    ii, jj = np.nonzero(M)
    assert int(np.sum(ii - jj >= w)) == gd["far_kept"][0] == far_total - gd["far_both"][0]
    Q = np.zeros((1, 1, n, 2))
    Kt = np.random.default_rng(0).standard_normal((1, 1, n, 2))
    V = np.stack([np.arange(n, dtype=np.float64), np.ones(n)], axis=1)[None, None]
    O, L = ref.attention_rows_topk(Q, Kt, V, G[None, None], w, 0.7, np.arange(n), 1)
    for i in range(n):
        np.testing.assert_allclose(O[0, 0, i], gd["O"][i], rtol=0, atol=1e-14)
    np.testing.assert_allclose(L[0, 0], np.log(np.array(gd["lse_count"], float)), atol=1e-14)


def test_assign_topk_closed_form_order_and_ties():
    # W = I, C = scaled basis / duplicates: the scores are known coordinates.
    W = np.eye(4)[None]
    C = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 1, 0], [0, 1, 0, 0], [0, 0, 0, 1]], float)[None]
    h = np.array([[[4, 3, 2, 1],       # scores [4,3,2,3,1]: top2 0, then 1 (tie 1/3 -> 1)
                   [1, 2, 3, 4],       # [1,2,3,2,4]: 4, 2
                   [0, 5, 5, 0],       # [0,5,5,5,0]: 1, 2 (three-way tie -> lowest two)
                   [-1, -2, -3, -4]]], float)  # [-1,-2,-3,-2,-4]: 0, 1
    gid, margin = ref.assign_topk(h, W, C, 2)
    assert gid[0, 0].tolist() == [[0, 1], [4, 2], [1, 2], [0, 1]]
    # smallest gap among ranks 1-2 and 2-3
    np.testing.assert_allclose(margin[0, 0], [0.0, 1.0, 0.0, 0.0], atol=1e-15)
    gid3, _ = ref.assign_topk(h, W, C, 3)
    assert gid3[0, 0].tolist() == [[0, 1, 3], [4, 2, 1], [1, 2, 3], [0, 1, 3]]


def test_assign_topk_bruteforce_and_k1_is_assign():
    rng = np.random.default_rng(21)
    B, n, D, A, dg, K = 2, 11, 6, 2, 4, 5
    h = rng.standard_normal((B, n, D))
    W = rng.standard_normal((A, dg, D))
    C = rng.standard_normal((A, K, dg))
    gid, margin = ref.assign_topk(h, W, C, 2)
    for b in range(B):
        for a in range(A):
            for i in range(n):
                p = [math.fsum(W[a, r, c] * h[b, i, c] for c in range(D)) for r in range(dg)]
                s = [math.fsum(p[r] * C[a, k, r] for r in range(dg)) for k in range(K)]
                first = max(range(K), key=lambda k: (s[k], -k))
                second = max((k for k in range(K) if k != first), key=lambda k: (s[k], -k))
                assert gid[b, a, i].tolist() == [first, second]
                srt = sorted(s, reverse=True)
                assert abs(margin[b, a, i] - min(srt[0] - srt[1], srt[1] - srt[2])) < 1e-12
    g1, m1 = ref.assign(h, W, C)
    gk, mk = ref.assign_topk(h, W, C, 1)
    assert np.array_equal(gk[..., 0], g1)
    np.testing.assert_allclose(mk, m1, atol=1e-12)


@pytest.mark.parametrize("K,n,w", [(4, 200, 9), (7, 301, 1), (2, 64, 64), (16, 257, 16)])
def test_index_topk_bruteforce_and_k1_is_index(K, n, w):
    rng = np.random.default_rng(K * 1000 + n)
    G = np.stack([rng.permutation(K)[:2] for _ in range(n)]).astype(np.int32)
    idx = ref.build_index_topk(G[None, None], K, w)
    slot = 0
    for g in range(K):
        members = [(i, c) for i in range(n) for c in range(2) if G[i, c] == g]
        assert idx["counts"][0, 0, g] == len(members)
        assert idx["offsets"][0, 0, g] == slot
        for t, (i, c) in enumerate(members):
            s = slot + t
            assert idx["perm"][0, 0, s] == 2 * i + c
            assert idx["rank"][0, 0, 2 * i + c] == s
            far = sum(1 for (j, _) in members if j <= i - w)
            assert idx["farlen_slot"][0, 0, s] == far
            assert idx["farlen_entry"][0, 0, 2 * i + c] == far
            assert idx["other"][0, 0, s] == G[i, 1 - c]
        slot += len(members)
    assert slot == 2 * n
    g1 = synth.draw_group_ids(K + n, 1, 1, n, K, "uniform")
    a = ref.build_index(g1, K, w)
    b = ref.build_index_topk(g1[..., None], K, w)
    for key, key2 in (("counts", "counts"), ("offsets", "offsets"), ("perm", "perm"), ("rank", "rank"),
                      ("farlen_tok", "farlen_entry"), ("farlen_slot", "farlen_slot")):
        assert np.array_equal(a[key], b[key2]), key
    assert np.all(b["other"] == -1)


@pytest.mark.parametrize("K,n,w", [(4, 160, 5), (6, 211, 12), (3, 90, 1)])
def test_topk_far_count_once_per_pair(K, n, w):
    # Far pairs kept by the mask = per-group far pairs (sum of farlen) minus
    # the pairs whose tokens share both groups, which every group list of the
    # two holds.  Also: keeping a shared-both pair only in the group that is
    # not larger than the slot's other group counts every far pair once.
    rng = np.random.default_rng(n + w)
    G = np.stack([rng.permutation(K)[:2] for _ in range(n)]).astype(np.int32)
    M = ref.keep_mask_rows_topk(G, w, np.arange(n))
    ii, jj = np.nonzero(M)
    far_kept = int(np.sum(ii - jj >= w))
    S = [frozenset(r.tolist()) for r in G]
    both = sum(1 for i in range(n) for j in range(max(0, i - w + 1)) if S[i] == S[j])
    idx = ref.build_index_topk(G[None, None], K, w)
    assert far_kept == int(idx["farlen_slot"].sum()) - both
    perm, other, off = idx["perm"][0, 0], idx["other"][0, 0], idx["offsets"][0, 0]
    dedup = 0
    for g in range(K):
        for s in range(off[g], off[g + 1]):
            for t in range(off[g], off[g] + idx["farlen_slot"][0, 0, s]):
                if not (other[t] == other[s] and other[s] < g):
                    dedup += 1
    assert dedup == far_kept


@pytest.mark.parametrize("K,n,w", [(2, 50, 3), (3, 120, 5), (4, 200, 7), (5, 150, 1), (4, 100, 1000)])
def test_top2_split_index_visits_every_far_pair_once(K, n, w):
    # Brute force over the work list: the (row, key) token pairs that the
    # items cover, each row taking the first farlen_sub keys of the item's
    # sub-run, are exactly the far pairs of the top-2 keep mask, once each;
    # and each token's two entries together hold its far-key count.
    rng = np.random.default_rng(K * 1000 + n + w)
    G = np.stack([rng.permutation(K)[:2] for _ in range(n)]).astype(np.int32)[None, None]
    idx = ref.build_index_top2_split(G, K, w)
    items = ref.work_items_top2_split(idx, 16)
    perm, fs = idx["perm"][0, 0], idx["farlen_sub"][0, 0]
    seen = {}
    for it in items:
        row0, rows, keys = int(it[3]), int(it[4]), int(it[5])
        segs = ref.segments_top2_split(idx, it)
        assert keys == sum(ln for _, ln, _ in segs) and keys > 0
        for start, ln, j in segs:
            for s in range(row0, row0 + rows):
                assert fs[s, j] <= ln
                for t in range(start, start + fs[s, j]):
                    pr = (int(perm[s]) // 2, int(perm[t]) // 2)
                    seen[pr] = seen.get(pr, 0) + 1
    M = ref.keep_mask_rows_topk(G[0, 0], w, np.arange(n))
    ii, jj = np.nonzero(M)
    want = {(int(i), int(j)) for i, j in zip(ii, jj) if i - j >= w}
    assert set(seen) == want
    assert all(c == 1 for c in seen.values())
    per_tok = idx["farlen_entry"][0, 0].reshape(n, 2).sum(axis=1)
    assert np.array_equal(per_tok, np.bincount(ii[ii - jj >= w], minlength=n))
    # the sort: virtual group v = g * K + o, then position
    ge = G[0, 0].reshape(-1)
    oe = G[0, 0][:, ::-1].reshape(-1)
    vs = (ge * K + oe)[perm]
    assert np.all(np.diff(vs) >= 0)
    same = np.diff(vs) == 0
    assert np.all(np.diff(perm // 2)[same] > 0)


def test_topk_reduces_to_dense_and_to_top1():
    rng = np.random.default_rng(22)
    B, H, Hkv, n, d = 1, 4, 2, 83, 8
    Q = rng.standard_normal((B, H, n, d))
    Kt = rng.standard_normal((B, Hkv, n, d))
    V = rng.standard_normal((B, Hkv, n, d))
    rows = np.arange(n)
    # K = 2, k = 2: every token is in both groups -> dense causal
    G = np.stack([rng.permutation(2) for _ in range(n)]).astype(np.int32)[None, None]
    O, L = ref.attention_rows_topk(Q, Kt, V, G, 3, 0.3, rows, 1)
    np.testing.assert_allclose(O, _sdpa_causal(Q, Kt, V, 0.3), atol=1e-12)
    # window >= n -> dense causal whatever the groups
    G = np.stack([rng.permutation(9)[:2] for _ in range(n)]).astype(np.int32)[None, None]
    O, L = ref.attention_rows_topk(Q, Kt, V, G, n, 0.3, rows, 1)
    np.testing.assert_allclose(O, _sdpa_causal(Q, Kt, V, 0.3), atol=1e-12)
    # k = 1 is the top-1 path
    g = synth.draw_group_ids(5, B, 2, n, 6, "uniform")
    O1, L1 = ref.attention_rows(Q, Kt, V, g, 7, 0.3, rows, 2)
    O2, L2 = ref.attention_rows_topk(Q, Kt, V, g[..., None], 7, 0.3, rows, 2)
    np.testing.assert_allclose(O2, O1, atol=1e-13)
    np.testing.assert_allclose(L2, L1, atol=1e-13)


@pytest.mark.parametrize("n,w,K", [(40, 3, 4), (33, 1, 6), (25, 30, 3), (48, 6, 5)])
def test_topk_bruteforce_small(n, w, K):
    rng = np.random.default_rng(n * 31 + w)
    d = 5
    Q, Kt, V = (rng.standard_normal((1, 1, n, d)) for _ in range(3))
    G = np.stack([rng.permutation(K)[:2] for _ in range(n)]).astype(np.int32)
    O, L = ref.attention_rows_topk(Q, Kt, V, G[None, None], w, 0.45, np.arange(n), 1)
    Ob, Lb = ref.attention_bruteforce_topk(Q[0, 0], Kt[0, 0], V[0, 0], G, w, 0.45)
    np.testing.assert_allclose(O[0, 0], Ob, atol=1e-12)
    np.testing.assert_allclose(L[0, 0], Lb, atol=1e-12)


def test_topk_inclusion_exclusion_merge_equals_union():
    # The far keys of token i with groups {a, b}: far members of a, of b, and
    # of the pair {a, b} (in both).  With w = exp(LSE - M):
    #   O = (w_a O_a + w_b O_b - w_ab O_ab) / (w_a + w_b - w_ab)
    # equals the softmax over the union of the far keys (the GPU merge).
    rng = np.random.default_rng(49)
    n, d, w, K = 160, 6, 5, 4
    Q, Kt, V = (rng.standard_normal((n, d)) for _ in range(3))
    G = np.stack([rng.permutation(K)[:2] for _ in range(n)]).astype(np.int32)
    rows = np.arange(n)
    i = rows[:, None]
    j = rows[None, :]
    far = j <= i - w
    in_a = (G[:, 0][:, None] == G[None, :, 0]) | (G[:, 0][:, None] == G[None, :, 1])
    in_b = (G[:, 1][:, None] == G[None, :, 0]) | (G[:, 1][:, None] == G[None, :, 1])
    Oa, La = ref.attention_masked_rows(Q, Kt, V, far & in_a, rows, 0.4)
    Ob, Lb = ref.attention_masked_rows(Q, Kt, V, far & in_b, rows, 0.4)
    Oab, Lab = ref.attention_masked_rows(Q, Kt, V, far & in_a & in_b, rows, 0.4)
    Ou, Lu = ref.attention_masked_rows(Q, Kt, V, far & (in_a | in_b), rows, 0.4)
    has = np.isfinite(Lu)
    assert has.sum() > n // 2
    M = np.maximum.reduce([La, Lb, np.where(np.isfinite(Lab), Lab, -np.inf)])
    with np.errstate(invalid="ignore", divide="ignore"):      # rows with no far key: excluded below
        wa, wb = np.exp(La - M), np.exp(Lb - M)
        wab = np.where(np.isfinite(Lab), np.exp(Lab - M), 0.0)
        den = wa + wb - wab
        Om = (wa[:, None] * np.nan_to_num(Oa) + wb[:, None] * np.nan_to_num(Ob)
              - wab[:, None] * np.nan_to_num(Oab)) / den[:, None]
    np.testing.assert_allclose(Om[has], Ou[has], atol=1e-12)
    np.testing.assert_allclose(M[has] + np.log(den[has]), Lu[has], atol=1e-12)
    # the denominator never cancels: it is at least the larger entry weight
    assert np.all(den[has] >= np.maximum(wa, wb)[has] - 1e-15)
    # and the union is the top-2 keep rule's far part
    Mk = ref.keep_mask_rows_topk(G, w, rows)
    assert np.array_equal(Mk & far, far & (in_a | in_b))


def test_topk_pins_catch_planted_mistakes():
    """Plausible slips in the top-k rule each break the hand-worked example."""
    gd, G = _golden_top2()
    n, w = gd["n"][0], gd["w"][0]
    rows = np.arange(n)

    def first_only(GG, ww, rr):            # membership read as the first choice alone
        return ref.keep_mask_rows(GG[:, 0], ww, rr)

    def both_equal(GG, ww, rr):            # sets must be equal, not just meet
        S = np.sort(GG, axis=1)
        jj = np.arange(len(GG))[None, :]
        ii = np.asarray(rr)[:, None]
        same = np.all(S[rr][:, None, :] == S[None, :, :], axis=2)
        return (jj <= ii) & (((ii - jj) < ww) | same)

    def same_rank(GG, ww, rr):             # choices compared rank by rank only
        jj = np.arange(len(GG))[None, :]
        ii = np.asarray(rr)[:, None]
        sh = np.zeros((len(rr), len(GG)), bool)
        for c in range(GG.shape[1]):
            sh |= GG[rr, c][:, None] == GG[None, :, c]
        return (jj <= ii) & (((ii - jj) < ww) | sh)

    for bad in (first_only, both_equal, same_rank):
        M = bad(G, w, rows)
        assert any(list(np.nonzero(M[i])[0]) != gd["kept"][i] for i in range(n)), bad.__name__


# --------------------------------------------------------------- sinkhorn ---

def test_scores_closed_form():
    # W picks coordinates, C are signed basis rows: S is a signed coordinate of h
    h = np.array([[[3.0, -1.0, 2.0], [0.5, 4.0, -2.0]]])
    W = np.array([[[1.0, 0.0, 0.0], [0.0, 0.0, 1.0]]])         # p = (h0, h2)
    C = np.array([[[1.0, 0.0], [0.0, -1.0], [2.0, 1.0]]])
    S = ref.scores(h, W, C)
    assert S[0, 0].tolist() == [[3.0, -2.0, 8.0], [0.5, 2.0, -1.0]]


def test_sinkhorn_marginals_converge():
    # Sinkhorn's theorem: a positive matrix scales to the prescribed marginals
    rng = np.random.default_rng(31)
    for n, K in ((64, 4), (300, 16), (33, 33)):
        S = rng.standard_normal((n, K)) * 2
        G = ref.sinkhorn(S, 200)
        np.testing.assert_allclose(G.sum(axis=1), 1.0, atol=1e-12)
        np.testing.assert_allclose(G.sum(axis=0), n / K, atol=1e-8)
        assert np.all(G > 0)


def test_sinkhorn_rank_one_is_uniform_after_one_round():
    # exp(a_i + b_k) is rank one: one column and one row step give 1/K
    rng = np.random.default_rng(32)
    a, b = rng.standard_normal(50), rng.standard_normal(7)
    G = ref.sinkhorn(a[:, None] + b[None, :], 1, tau=0.7)
    np.testing.assert_allclose(G, 1.0 / 7, atol=1e-14)


def test_sinkhorn_doubly_stochastic_input_is_a_fixed_point():
    # n = K: a convex combination of permutation matrices (Birkhoff) has unit
    # row and column sums already, so every round returns it unchanged
    rng = np.random.default_rng(33)
    n = 6
    wts = rng.dirichlet(np.ones(4))
    P = sum(wv * np.eye(n)[rng.permutation(n)] for wv in wts)
    P = 0.9 * P + 0.1 / n                       # strictly positive, still doubly stochastic
    for T in (1, 3):
        np.testing.assert_allclose(ref.sinkhorn(np.log(P), T), P, atol=1e-14)


def test_sinkhorn_column_shift_invariance_and_row_shift_at_convergence():
    rng = np.random.default_rng(34)
    S = rng.standard_normal((40, 5))
    b = rng.standard_normal(5) * 3
    a = rng.standard_normal(40) * 3
    for T in (1, 2, 5):   # the first step is a column scaling: exact for any T
        np.testing.assert_allclose(ref.sinkhorn(S + b[None, :], T), ref.sinkhorn(S, T), atol=1e-13)
    # a per-row shift changes finite rounds but not the limit
    assert not np.allclose(ref.sinkhorn(S + a[:, None], 1), ref.sinkhorn(S, 1), atol=1e-6)
    np.testing.assert_allclose(ref.sinkhorn(S + a[:, None], 400), ref.sinkhorn(S, 400), atol=1e-9)


def test_sinkhorn_equivariance_and_special_cases():
    rng = np.random.default_rng(35)
    S = rng.standard_normal((2, 30, 6))
    G = ref.sinkhorn(S, 4, tau=1.5)
    pr, pc = rng.permutation(30), rng.permutation(6)
    np.testing.assert_allclose(ref.sinkhorn(S[:, pr][:, :, pc], 4, tau=1.5), G[:, pr][:, :, pc], atol=1e-14)
    np.testing.assert_allclose(ref.sinkhorn(S[:, :, :1], 3), 1.0, atol=0)        # K = 1
    np.testing.assert_allclose(ref.sinkhorn(np.zeros((9, 3)), 2), 1.0 / 3, atol=1e-15)
    # tau scales the scores: sinkhorn(S, tau) == sinkhorn(S / tau, 1)
    np.testing.assert_allclose(ref.sinkhorn(S, 3, tau=0.25), ref.sinkhorn(S * 4, 3), atol=1e-13)


def test_sinkhorn_one_round_by_hand():
    # 2 x 2, T = 1, worked by hand: exp(S) = [[1, 2], [3, 4]]; n / K = 1.
    # columns: [[1/4, 2/6], [3/4, 4/6]]; rows: [[3/7, 4/7], [9/17, 8/17]]
    S = np.log(np.array([[1.0, 2.0], [3.0, 4.0]]))
    np.testing.assert_allclose(ref.sinkhorn(S, 1), [[3 / 7, 4 / 7], [9 / 17, 8 / 17]], atol=1e-15)


def test_sinkhorn_pins_catch_planted_mistakes():
    S = np.log(np.array([[1.0, 2.0], [3.0, 4.0]]))
    want = np.array([[3 / 7, 4 / 7], [9 / 17, 8 / 17]])

    def rows_first(SS, T):             # order of the two steps swapped
        M = np.exp(SS)
        for _ in range(T):
            M = M / M.sum(axis=-1, keepdims=True)
            M = M * ((SS.shape[-2] / SS.shape[-1]) / M.sum(axis=-2, keepdims=True))
        return M

    def softmax_only(SS, T):           # the column step dropped: a row softmax
        M = np.exp(SS)
        return M / M.sum(axis=-1, keepdims=True)

    def scores_not_exponentiated(SS, T):
        M = SS - SS.min() + 1.0
        for _ in range(T):
            M = M * ((SS.shape[-2] / SS.shape[-1]) / M.sum(axis=-2, keepdims=True))
            M = M / M.sum(axis=-1, keepdims=True)
        return M

    for bad in (rows_first, softmax_only, scores_not_exponentiated):
        assert not np.allclose(bad(S, 1), want, atol=1e-6), bad.__name__
    # (the column target's value alone is not a slip: with equal targets the
    # row step removes any common factor, so columns reach n / K at the limit)
    S3 = np.log(np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 1.0]]))
    np.testing.assert_allclose(ref.sinkhorn(S3, 300).sum(axis=0), 1.5, atol=1e-9)
    assert not np.allclose(softmax_only(S3, 300).sum(axis=0), 1.5, atol=1e-3)


# --------------------------------------------------------------- backward ---

def _loss(Q, K, V, g, w, scale, A, dO):
    O, _ = ref.attention(Q, K, V, g, w, scale, A)
    return float(np.sum(O * dO))


def test_backward_matches_central_differences():
    # L = sum(O * dO) has gradient (dQ, dK, dV) for the fixed dO
    rng = np.random.default_rng(41)
    B, H, Hkv, n, d, w = 1, 2, 1, 12, 3, 3
    Q = rng.standard_normal((B, H, n, d))
    K = rng.standard_normal((B, Hkv, n, d))
    V = rng.standard_normal((B, Hkv, n, d))
    dO = rng.standard_normal((B, H, n, d))
    g = synth.draw_group_ids(6, B, 1, n, 3, "uniform")
    dQ, dK, dV = ref.attention_backward(Q, K, V, g, w, 0.6, 1, dO)
    eps = 1e-6
    for X, dX in ((Q, dQ), (K, dK), (V, dV)):
        for idx in [(0, 0, 0, 0), (0, 0, 5, 2), (0, X.shape[1] - 1, n - 1, 1), (0, 0, 7, 0)]:
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args = lambda Z: (Z if X is Q else Q, Z if X is K else K, Z if X is V else V)
            num = (_loss(*args(Xp), g, w, 0.6, 1, dO) - _loss(*args(Xm), g, w, 0.6, 1, dO)) / (2 * eps)
            assert abs(num - dX[idx]) < 1e-7, (idx, num, dX[idx])


def test_backward_dense_case_matches_torch_autograd():
    # K = 1 keeps every causal pair: the gradients of causal SDPA (torch, fp64)
    rng = np.random.default_rng(42)
    B, H, Hkv, n, d = 2, 4, 2, 37, 8
    Q = rng.standard_normal((B, H, n, d))
    K = rng.standard_normal((B, Hkv, n, d))
    V = rng.standard_normal((B, Hkv, n, d))
    dO = rng.standard_normal((B, H, n, d))
    g = np.zeros((B, 1, n), np.int32)
    dQ, dK, dV = ref.attention_backward(Q, K, V, g, 5, 0.3, 1, dO)
    Qt = torch.from_numpy(Q).requires_grad_()
    Kt = torch.from_numpy(K).requires_grad_()
    Vt = torch.from_numpy(V).requires_grad_()
    rep = H // Hkv
    O = torch.nn.functional.scaled_dot_product_attention(
        Qt, Kt.repeat_interleave(rep, dim=1), Vt.repeat_interleave(rep, dim=1), is_causal=True, scale=0.3)
    O.backward(torch.from_numpy(dO))
    np.testing.assert_allclose(dQ, Qt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dK, Kt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dV, Vt.grad.numpy(), atol=1e-12)


def test_backward_invariants():
    # rows of P sum to 1: sum_j dV_j = sum_i dO_i; rows of dS sum to 0: a
    # common shift of all keys leaves the loss unchanged, so sum_j dK_j = 0
    rng = np.random.default_rng(43)
    B, H, Hkv, n, d = 1, 3, 1, 90, 5
    Q, dO = (rng.standard_normal((B, H, n, d)) for _ in range(2))
    K, V = (rng.standard_normal((B, Hkv, n, d)) for _ in range(2))
    g = synth.draw_group_ids(44, B, 1, n, 4, "zipf")
    dQ, dK, dV = ref.attention_backward(Q, K, V, g, 7, 0.4, 1, dO)
    np.testing.assert_allclose(dV.sum(axis=2)[0, 0], dO.sum(axis=(1, 2))[0], atol=1e-11)
    np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-11)
    # a key no query keeps gets no gradient: with one group per token and
    # w = 1 only j = i is kept, so every key feeds one query
    gd = synth.draw_group_ids(45, 1, 1, 20, 20, "distinct")
    q1, k1, v1, o1 = (rng.standard_normal((1, 1, 20, 4)) for _ in range(4))
    _, dK1, dV1 = ref.attention_backward(q1, k1, v1, gd, 1, 0.5, 1, o1)
    np.testing.assert_allclose(dV1, o1, atol=1e-14)       # P = I
    np.testing.assert_allclose(dK1, 0.0, atol=1e-14)      # softmax of one key is flat


def test_backward_dq_rows_equal_full_backward_rows():
    rng = np.random.default_rng(47)
    B, H, Hkv, n, d = 1, 4, 2, 70, 6
    Q, dO = (rng.standard_normal((B, H, n, d)) for _ in range(2))
    K, V = (rng.standard_normal((B, Hkv, n, d)) for _ in range(2))
    g = synth.draw_group_ids(48, B, 2, n, 5, "uniform")
    dQ, _, _ = ref.attention_backward(Q, K, V, g, 6, 0.35, 2, dO)
    rows = np.array([0, 3, 17, 50, 69])
    np.testing.assert_allclose(ref.attention_backward_dq_rows(Q, K, V, g, 6, 0.35, 2, dO, rows),
                               dQ[:, :, rows], atol=1e-13)


def test_backward_dkv_rows_equal_full_backward_rows():
    # key rows gathered column by column (the queries that keep each key) give
    # the full backward's dK, dV rows: GQA with per-KV-head ids and Zipf groups
    rng = np.random.default_rng(49)
    for B, H, Hkv, A, n, d, w, K, kind in ((1, 4, 2, 2, 70, 6, 6, 5, "uniform"),
                                          (2, 2, 1, 1, 64, 4, 3, 3, "zipf"),
                                          (1, 2, 2, 1, 40, 5, 50, 2, "uniform")):   # w > n: dense
        Q, dO = (rng.standard_normal((B, H, n, d)) for _ in range(2))
        Kt, V = (rng.standard_normal((B, Hkv, n, d)) for _ in range(2))
        g = synth.draw_group_ids(50 + n, B, A, n, K, kind)
        _, dK, dV = ref.attention_backward(Q, Kt, V, g, w, 0.35, A, dO)
        krows = np.array([0, 1, n // 2, n - 2, n - 1])
        gK, gV = ref.attention_backward_dkv_rows(Q, Kt, V, g, w, 0.35, A, dO, krows)
        np.testing.assert_allclose(gK, dK[:, :, krows], atol=1e-12)
        np.testing.assert_allclose(gV, dV[:, :, krows], atol=1e-12)


def test_backward_dkv_rows_match_central_differences():
    rng = np.random.default_rng(51)
    B, H, Hkv, n, d, w = 1, 2, 1, 12, 3, 3
    Q, dO = (rng.standard_normal((B, H, n, d)) for _ in range(2))
    K, V = (rng.standard_normal((B, Hkv, n, d)) for _ in range(2))
    g = synth.draw_group_ids(52, B, 1, n, 3, "uniform")
    krows = np.array([2, 7, 11])
    gK, gV = ref.attention_backward_dkv_rows(Q, K, V, g, w, 0.6, 1, dO, krows)
    eps = 1e-6
    for X, G in ((K, gK), (V, gV)):
        for r, j in enumerate(krows):
            for c in range(d):
                Xp, Xm = X.copy(), X.copy()
                Xp[0, 0, j, c] += eps
                Xm[0, 0, j, c] -= eps
                args = lambda Z: (Q, Z if X is K else K, Z if X is V else V)
                num = (_loss(*args(Xp), g, w, 0.6, 1, dO) - _loss(*args(Xm), g, w, 0.6, 1, dO)) / (2 * eps)
                assert abs(num - G[0, 0, r, c]) < 1e-7, (j, c, num, G[0, 0, r, c])


def test_backward_planted_mistake_is_caught():
    # the finite-difference pin rejects a backward that drops the D term
    # (dS = P * dP): the planted version's dQ misses the numerical gradient
    rng = np.random.default_rng(46)
    n, d, w, sc = 10, 3, 2, 0.5
    Q, K, V, dO = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    g = synth.draw_group_ids(7, 1, 1, n, 2, "uniform")
    rows = np.arange(n)
    M = ref.keep_mask_rows(g[0, 0], w, rows)
    P = ref.attention_weights_rows(Q[0, 0], K[0, 0], M, rows, sc)
    bad_dQ = sc * ((P * (dO[0, 0] @ V[0, 0].T)) @ K[0, 0])
    eps = 1e-6
    worst = 0.0
    for i in range(n):
        for c in range(d):
            Qp, Qm = Q.copy(), Q.copy()
            Qp[0, 0, i, c] += eps
            Qm[0, 0, i, c] -= eps
            num = (_loss(Qp, K, V, g, w, sc, 1, dO) - _loss(Qm, K, V, g, w, sc, 1, dO)) / (2 * eps)
            worst = max(worst, abs(num - bad_dQ[i, c]))
    assert worst > 1e-3


# ------------------------------------------------ planted oracle mistakes ---

def test_pins_catch_planted_mistakes(monkeypatch):
    """Each plausible slip in the keep rule breaks the hand-worked example."""
    gd = _parse_golden("keep_rule_n8.txt")
    g = np.array(gd["groups"], np.int32)
    good = ref.keep_mask_rows

    def off_by_one(gg, w, rows):          # window read as i - j <= w
        return good(gg, w + 1, rows)

    def no_causal(gg, w, rows):           # future same-group keys leak in
        rows = np.asarray(rows)
        jj = np.arange(len(gg))[None, :]
        ii = rows[:, None]
        return (((ii - jj) < w) & (jj <= ii)) | (gg[rows][:, None] == gg[None, :])

    def no_group(gg, w, rows):            # far term dropped
        rows = np.asarray(rows)
        jj = np.arange(len(gg))[None, :]
        ii = rows[:, None]
        return (jj <= ii) & ((ii - jj) < w)

    for bad in (off_by_one, no_causal, no_group):
        M = bad(g, gd["w"][0], np.arange(gd["n"][0]))
        assert any(list(np.nonzero(M[i])[0]) != gd["kept"][i] for i in range(gd["n"][0])), bad.__name__
