"""Plain fp64 CPU oracle for the Focus inference hot path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
the benchmark's CPU-baseline leg may import this module.  The product path
(the CUDA library and its Python binding) never imports or calls it and shares
no code with it.

Sources (page titles and sections):
  [FocusJA] "Focus: Learning Which Attention Pairs Matter" (gist.science, ja),
            section 2.1 (architecture: centroids, local + group-gated far
            attention), section 2.2 (inference: hard top-k assignment, far pairs
            of different groups skipped, pair count O(n^2/K + n*w)),
            section 3.3 (local window + in-group causal decomposition).
  [FocusKO] "Why Attend to Everything? Focus is the Key" (gist.science, ko),
            section 2.1 (exact softmax preserved), section 2.3 (hard top-k
            assignment at inference, two FlashAttention calls).

What the oracle computes (fp64 throughout, no blocking or fusion):
  assign       p = W_a h (no bias), s_k = p . c_k, g = argmax_k s_k with the
               lowest index winning ties.  The decision is taken on the scores
               rounded to fp32 (the precision the hot path fixes for the
               scores); the exact fp64 margin between the best and runner-up
               score is returned as well.
  build_index  counting sort of tokens by (group, position) per (batch,
               assignment): counts, offsets, perm, rank, farlen, and the
               group-pass work list for a tile height BM.
  keep mask    pair (i, j) kept iff j <= i and (i - j < w or g_i == g_j).
  attention    exact softmax over the kept pairs only, S = scale * Q K^T.
  top-k        the hard top-k variant ([FocusJA] 2.2, 3.3; [FocusKO] 2.3,
               whose experiment uses K=4, k=2): each token belongs to its k
               best groups, and a far pair is kept when the two tokens' group
               sets intersect.  assign_topk,
               build_index_topk (memberships sorted by (group, position)),
               keep_mask_rows_topk and attention_rows_topk are the same
               definitions written for k memberships.
  sinkhorn     the training-time soft assignment ([FocusJA] 2.1, 2.3;
               [FocusKO] 2.2): the matrix exp(S / tau) of token-to-centroid
               scores is scaled to be doubly stochastic with every token's
               row summing to 1 and every group's column to n / K (equal
               group sizes), by T rounds of Sinkhorn-Knopp scaling (columns,
               then rows).  scores() gives S = (h W_a^T) C_a^T.
  backward     gradients of the attention output over the kept pairs
               (training or fine-tuning a retrofit, [FocusKO] 2.1 and
               [FocusJA] 3.1): with P the kept-pair softmax and a fixed
               upstream dO, dV = P^T dO, dS = P * (dO V^T - rowsum(dO * O)),
               dQ = scale dS K, dK = scale dS^T Q, dK and dV summed over the
               query heads that share a key/value head.

Readings where the pages are silent (each listed in the design notes):
  similarity = dot product; no projection bias; window strictly i - j < w;
  scale = 1/sqrt(d) by default; GQA head map kv = floor(h * H_kv / H);
  each kept pair counted once (union of the local and the group rule);
  top-k: the k best fp32 scores, lower index first among equal scores, and a
  pair whose tokens share several groups is still one kept pair;
  Sinkhorn: temperature tau and round count T are parameters (the pages give
  neither), each round normalises columns first and rows last, and the
  marginals are 1 per token and n / K per group.

Parity pins: every function here is checked by tests/test_oracle_pins.py
against closed forms, brute force, special cases and invariants.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "assign", "build_index", "work_items", "lpt_order", "keep_mask_rows", "keep_mask",
    "kept_counts", "attention", "attention_rows", "attention_masked_rows",
    "dense_causal", "lse_merge", "attention_bruteforce", "attention_weights_rows",
    "kv_head", "assignment_of_head",
    "assign_topk", "build_index_topk", "build_index_top2_split", "work_items_top2_split",
    "segments_top2_split",
    "keep_mask_rows_topk", "attention_rows_topk",
    "attention_bruteforce_topk", "scores", "sinkhorn", "attention_backward",
    "attention_backward_dq_rows",
]


# ---------------------------------------------------------------- helpers ---

def kv_head(h: int, H: int, H_kv: int) -> int:
    """Key/value head used by query head h: contiguous groups of H/H_kv heads."""
    return (h * H_kv) // H


def assignment_of_head(h: int, H: int, H_kv: int, A: int) -> int:
    """Assignment index a used by query head h (A == 1: shared; A == H_kv: per kv head)."""
    return 0 if A == 1 else kv_head(h, H, H_kv)


def _f64(x):
    return np.asarray(x, dtype=np.float64)


# ----------------------------------------------------------------- assign ---

def assign(h, W, C, chunk: int = 4096):
    """Nearest-centroid group ids.  [FocusJA] 2.1 (centroids, projection,
    similarity), 2.2 and [FocusKO] 2.3 (hard assignment at inference).

    h [B, n, D], W [A, d_g, D], C [A, K, d_g]  ->  gid [B, A, n] int32,
    margin [B, A, n] fp64 (best minus runner-up score; +inf when K == 1).
    """
    h = np.asarray(h)
    W = _f64(W)
    C = _f64(C)
    B, n, D = h.shape
    A, d_g, D2 = W.shape
    K = C.shape[1]
    assert D2 == D and C.shape == (A, K, d_g)
    gid = np.empty((B, A, n), dtype=np.int32)
    margin = np.empty((B, A, n), dtype=np.float64)
    for b in range(B):
        for s in range(0, n, chunk):
            hb = _f64(h[b, s:s + chunk])                  # [m, D]
            for a in range(A):
                p = hb @ W[a].T                           # projection, [m, d_g]
                sc = p @ C[a].T                           # scores, [m, K]
                sc32 = sc.astype(np.float32)              # decision precision
                gid[b, a, s:s + chunk] = np.argmax(sc32, axis=1)   # first max wins
                if K > 1:
                    top2 = np.sort(sc, axis=1)[:, -2:]
                    margin[b, a, s:s + chunk] = top2[:, 1] - top2[:, 0]
                else:
                    margin[b, a, s:s + chunk] = np.inf
    return gid, margin


# ------------------------------------------------------------------ index ---

def build_index(gid, K: int, w: int):
    """Group-sorted token index per (batch, assignment).  [FocusJA] 2.2 (far
    pairs of different groups are skipped, so each group's tokens are gathered
    together); the sort key is (group, position).

    Returns a dict of arrays, each with leading dims [B, A]:
      counts [K], offsets [K+1] (exclusive scan), perm [n] (sorted slot ->
      position), rank [n] (position -> slot), farlen_tok [n] (per position),
      farlen_slot [n] (per slot), where farlen of token i is the number of
      tokens j of the same group with j <= i - w.
    """
    gid = np.asarray(gid)
    B, A, n = gid.shape
    counts = np.zeros((B, A, K), np.int32)
    offsets = np.zeros((B, A, K + 1), np.int32)
    perm = np.zeros((B, A, n), np.int32)
    rank = np.zeros((B, A, n), np.int32)
    far_tok = np.zeros((B, A, n), np.int32)
    far_slot = np.zeros((B, A, n), np.int32)
    for b in range(B):
        for a in range(A):
            g = gid[b, a].astype(np.int64)
            assert g.min() >= 0 and g.max() < K, "group id out of range"
            counts[b, a] = np.bincount(g, minlength=K)
            offsets[b, a, 1:] = np.cumsum(counts[b, a])
            p = np.argsort(g, kind="stable")              # by group, then position
            perm[b, a] = p
            rank[b, a, p] = np.arange(n)
            for k in range(K):
                members = p[offsets[b, a, k]:offsets[b, a, k + 1]]   # increasing positions
                if len(members) == 0:
                    continue
                # members j with j <= i - w  ==  count of members < i - w + 1
                fl = np.searchsorted(members, members - w + 1, side="left")
                far_tok[b, a, members] = fl
                far_slot[b, a, offsets[b, a, k]:offsets[b, a, k + 1]] = fl
    return dict(counts=counts, offsets=offsets, perm=perm, rank=rank,
                farlen_tok=far_tok, farlen_slot=far_slot)


def work_items(index: dict, BM: int):
    """Group-pass work list in canonical order (b, a, g, row0).

    One candidate tile per BM sorted slots of each group; a tile is emitted only
    when its last row has at least one far key (farlen is non-decreasing inside
    a group, so that row has the most).  Each item is
    (b, a, g, row0, rows, keys, key0): rows = sorted slots row0..row0+rows-1,
    keys = farlen of the tile's last row, key0 = offsets[g] (first key slot).
    """
    counts, offsets, fs = index["counts"], index["offsets"], index["farlen_slot"]
    B, A, K = counts.shape
    out = []
    for b in range(B):
        for a in range(A):
            for g in range(K):
                c = int(counts[b, a, g])
                o = int(offsets[b, a, g])
                for t in range(0, c, BM):
                    rows = min(BM, c - t)
                    keys = int(fs[b, a, o + t + rows - 1])
                    if keys > 0:
                        out.append((b, a, g, o + t, rows, keys, o))
    return np.array(out, dtype=np.int32).reshape(-1, 7)


def lpt_order(items: np.ndarray, BN: int):
    """Longest-first schedule: item indices sorted by ceil(keys/BN) descending,
    ties by canonical index ascending."""
    tiles = (items[:, 5].astype(np.int64) + BN - 1) // BN
    return np.lexsort((np.arange(len(items)), -tiles)).astype(np.int32)


# ------------------------------------------------------------------- mask ---

def keep_mask_rows(g, w: int, rows):
    """Keep rule for query rows `rows` against all keys.  [FocusJA] 2.1 and
    [FocusKO] 2.1: local window at full resolution, far pairs only inside a
    group; causal.  M[r, j] = (j <= i) and ((i - j < w) or (g_i == g_j)), i = rows[r].
    """
    g = np.asarray(g)
    rows = np.asarray(rows, dtype=np.int64)
    j = np.arange(len(g))[None, :]
    i = rows[:, None]
    return (j <= i) & (((i - j) < w) | (g[rows][:, None] == g[None, :]))


def keep_mask(g, w: int):
    return keep_mask_rows(g, w, np.arange(len(g)))


def kept_counts(index: dict, w: int):
    """Kept pairs per query token: min(i+1, w) window keys plus farlen far keys.
    [FocusJA] 2.2 (pair count O(n^2/K + n*w))."""
    n = index["perm"].shape[-1]
    win = np.minimum(np.arange(n) + 1, w)
    return win[None, None, :] + index["farlen_tok"]


# -------------------------------------------------------------- attention ---

def attention_masked_rows(Q, K, V, M, rows, scale):
    """Exact softmax attention of query rows `rows` of one head over mask M.

    Q [n, d], K/V [n, d], M [len(rows), n] bool.  Returns O [len(rows), d] and
    the natural-log LSE [len(rows)]; rows with an empty kept set give O = 0 and
    LSE = -inf.  [FocusKO] 2.1: softmax exactly as in the pretrained model,
    restricted to the kept pairs.
    """
    q = _f64(Q)[np.asarray(rows)]
    S = (q @ _f64(K).T) * float(scale)
    S = np.where(M, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    empty = ~np.isfinite(m[:, 0])
    m_safe = np.where(np.isfinite(m), m, 0.0)
    P = np.exp(S - m_safe)
    P[~M] = 0.0
    l = P.sum(axis=1, keepdims=True)
    l_safe = np.where(l > 0, l, 1.0)
    O = (P @ _f64(V)) / l_safe
    lse = (m_safe + np.log(l_safe))[:, 0]
    O[empty] = 0.0
    lse[empty] = -np.inf
    return O, lse


def attention_weights_rows(Q, K, M, rows, scale):
    """Softmax weights P [len(rows), n] of query rows over mask M (for invariants)."""
    q = _f64(Q)[np.asarray(rows)]
    S = np.where(M, (q @ _f64(K).T) * float(scale), -np.inf)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    P[~M] = 0.0
    return P / P.sum(axis=1, keepdims=True)


def attention_rows(Q, K, V, gid, w: int, scale: float, rows, A: int, row_block: int = 1024):
    """Focus attention for selected query rows of every (b, h).

    Q [B,H,n,d], K/V [B,H_kv,n,d], gid [B,A,n], rows: index array into n.
    Returns O [B,H,len(rows),d] and LSE [B,H,len(rows)] in fp64.
    """
    B, H, n, d = Q.shape
    H_kv = K.shape[1]
    rows = np.asarray(rows, dtype=np.int64)
    O = np.empty((B, H, len(rows), d))
    L = np.empty((B, H, len(rows)))
    for b in range(B):
        for hq in range(H):
            kv = kv_head(hq, H, H_kv)
            a = assignment_of_head(hq, H, H_kv, A)
            Kf, Vf = _f64(K[b, kv]), _f64(V[b, kv])
            for s in range(0, len(rows), row_block):
                r = rows[s:s + row_block]
                M = keep_mask_rows(gid[b, a], w, r)
                O[b, hq, s:s + row_block], L[b, hq, s:s + row_block] = \
                    attention_masked_rows(Q[b, hq], Kf, Vf, M, r, scale)
    return O, L


def attention(Q, K, V, gid, w: int, scale: float, A: int):
    """Focus attention over all rows: O [B,H,n,d], LSE [B,H,n] (fp64)."""
    return attention_rows(Q, K, V, gid, w, scale, np.arange(Q.shape[2]), A)


def dense_causal(Q, K, V, scale: float):
    """Ordinary causal attention (every j <= i kept) over all rows."""
    B, H, n, d = Q.shape
    gid = np.zeros((B, 1, n), np.int32)
    return attention(Q, K, V, gid, n, scale, 1)


def lse_merge(O1, L1, O2, L2):
    """Merge two softmax partials over disjoint key sets into one.

    O = (e^{L1} O1 + e^{L2} O2) / (e^{L1} + e^{L2}), with the larger LSE shifted
    out; an empty partial (LSE = -inf) contributes nothing.  [FocusKO] 2.3 and
    [FocusJA] 3.3: the pattern splits into a local-window call and an in-group
    call whose results combine into the exact softmax over the union.
    """
    O1, O2 = _f64(O1), _f64(O2)
    L1, L2 = _f64(L1), _f64(L2)
    m = np.maximum(L1, L2)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e1 = np.where(np.isfinite(L1), np.exp(L1 - m_safe), 0.0)
    e2 = np.where(np.isfinite(L2), np.exp(L2 - m_safe), 0.0)
    den = e1 + e2
    den_safe = np.where(den > 0, den, 1.0)
    O = (e1[..., None] * O1 + e2[..., None] * O2) / den_safe[..., None]
    L = np.where(den > 0, m_safe + np.log(den_safe), -np.inf)
    return O, L


# ------------------------------------------------------------ brute force ---

def attention_bruteforce(q, k, v, g, w: int, scale: float):
    """Scalar-loop reference for one head at small n (n <= 64).

    The kept set of row i is built as the union of its window list
    {max(0, i-w+1), ..., i} and the list of earlier members of its own group,
    a construction independent of the n x n mask; sums use math.fsum.
    Returns O [n][d] and LSE [n] as Python lists.
    """
    n, d = len(q), len(q[0])
    members = {}
    for j in range(n):
        members.setdefault(int(g[j]), []).append(j)
    O, L = [], []
    for i in range(n):
        kept = set(range(max(0, i - w + 1), i + 1))
        kept.update(j for j in members[int(g[i])] if j <= i)
        kept = sorted(kept)
        s = [math.fsum(float(q[i][c]) * float(k[j][c]) for c in range(d)) * scale for j in kept]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        z = math.fsum(e)
        O.append([math.fsum(e[t] * float(v[j][c]) for t, j in enumerate(kept)) / z for c in range(d)])
        L.append(mx + math.log(z))
    return O, L


# ------------------------------------------------------------------ top-k ---

def assign_topk(h, W, C, k: int, chunk: int = 4096):
    """The k nearest centroids per token, best first.  [FocusJA] 2.2, 3.3 and
    [FocusKO] 2.3 (hard top-k membership at inference).

    h [B, n, D], W [A, d_g, D], C [A, K, d_g]  ->  gid [B, A, n, k] int32 (rank
    order; among equal fp32 scores the lower index ranks first), margin
    [B, A, n] fp64: the smallest gap between consecutive ranks 1..k+1 (the
    gaps that decide the set and its order; +inf where there is none).
    """
    h = np.asarray(h)
    W = _f64(W)
    C = _f64(C)
    B, n, D = h.shape
    A, d_g, _ = W.shape
    K = C.shape[1]
    assert 1 <= k <= K
    gid = np.empty((B, A, n, k), dtype=np.int32)
    margin = np.full((B, A, n), np.inf)
    for b in range(B):
        for s in range(0, n, chunk):
            hb = _f64(h[b, s:s + chunk])
            for a in range(A):
                sc = (hb @ W[a].T) @ C[a].T                      # [m, K] scores
                sc32 = sc.astype(np.float32)
                order = np.argsort(-sc32, axis=1, kind="stable")  # best first, ties by index
                gid[b, a, s:s + chunk] = order[:, :k]
                srt = np.take_along_axis(sc, order, axis=1)
                last = min(k + 1, K)
                if last > 1:
                    margin[b, a, s:s + chunk] = np.min(srt[:, :last - 1] - srt[:, 1:last], axis=1)
    return gid, margin


def build_index_topk(gid, K: int, w: int):
    """Membership index for top-k groups per (batch, assignment).  [FocusJA]
    2.2: a token sits in each of its k groups, so each group's member list
    holds every token with that group among its k.

    gid [B, A, n, k].  Entry e = i * k + c is token i's c-th membership.
    Returns arrays with leading dims [B, A]: counts [K], offsets [K+1],
    perm [n*k] (sorted slot -> entry; slots of a group in increasing
    position), rank [n*k] (entry -> slot), farlen_entry [n*k] and farlen_slot
    [n*k] (members of the entry's group at positions j <= i - w), other [n*k]
    (k = 2: the group of the slot's token other than the slot's own; -1 for
    k = 1).  For k = 1 these are exactly build_index's arrays.
    """
    gid = np.asarray(gid)
    B, A, n, k = gid.shape
    m = n * k
    counts = np.zeros((B, A, K), np.int32)
    offsets = np.zeros((B, A, K + 1), np.int32)
    perm = np.zeros((B, A, m), np.int32)
    rank = np.zeros((B, A, m), np.int32)
    far_e = np.zeros((B, A, m), np.int32)
    far_s = np.zeros((B, A, m), np.int32)
    other = np.full((B, A, m), -1, np.int32)
    for b in range(B):
        for a in range(A):
            ge = gid[b, a].reshape(m).astype(np.int64)        # group of each entry
            assert ge.min() >= 0 and ge.max() < K, "group id out of range"
            for i in range(n):
                assert len(set(gid[b, a, i].tolist())) == k, "a token's k groups must differ"
            counts[b, a] = np.bincount(ge, minlength=K)
            offsets[b, a, 1:] = np.cumsum(counts[b, a])
            p = np.argsort(ge, kind="stable")                 # by group, then entry = (position, choice)
            perm[b, a] = p
            rank[b, a, p] = np.arange(m)
            pos = p // k
            for g in range(K):
                lo, hi = offsets[b, a, g], offsets[b, a, g + 1]
                if hi == lo:
                    continue
                members = pos[lo:hi]                          # increasing positions
                fl = np.searchsorted(members, members - w + 1, side="left")
                far_s[b, a, lo:hi] = fl
                far_e[b, a, p[lo:hi]] = fl
            if k == 2:
                other[b, a] = ge[p ^ 1]                       # the token's other membership
    return dict(counts=counts, offsets=offsets, perm=perm, rank=rank,
                farlen_entry=far_e, farlen_slot=far_s, other=other)


def build_index_top2_split(gid, K: int, w: int):
    """Membership index for top-2 groups that visits every far pair once.

    [FocusJA] 2.2, 3.3: token i sits in both of its groups, and a far pair is
    kept when the two tokens share a group; a pair whose tokens share both
    groups is still one kept pair ([FocusKO] 2.3).  Here each kept far pair is
    counted in the pass of the smaller group the two tokens share (this
    build's reading of "once").  Memberships (entry e = 2 i + c, group
    g = gid[i, c], other group o = gid[i, 1 - c]) are sorted by the virtual
    group v = g * K + o, then by position, so group g's members form K - 1
    sub-runs (g, o').  For the slot s of an entry with groups (g, o) and each
    other group o' != g (column j = o' if o' < g else o' - 1):
      farlen_sub[s, j] = members of sub-run (g, o') at positions <= i - w,
    except 0 when o' == o and o < g (those tokens share both groups with i,
    and the pair is counted in group o's pass).

    gid [B, A, n, 2].  Returns arrays with leading dims [B, A]: counts [K*K],
    offsets [K*K + 1], perm [2n] (slot -> entry), rank [2n], farlen_sub
    [2n, K - 1] (by slot), farlen_entry [2n] (far keys of each entry over all
    its sub-runs).
    """
    gid = np.asarray(gid)
    B, A, n, k = gid.shape
    assert k == 2, "two groups per token"
    m = 2 * n
    Kv = K * K
    counts = np.zeros((B, A, Kv), np.int32)
    offsets = np.zeros((B, A, Kv + 1), np.int32)
    perm = np.zeros((B, A, m), np.int32)
    rank = np.zeros((B, A, m), np.int32)
    fsub = np.zeros((B, A, m, max(K - 1, 1)), np.int32)
    fent = np.zeros((B, A, m), np.int32)
    for b in range(B):
        for a in range(A):
            G = gid[b, a].astype(np.int64)
            assert G.min() >= 0 and G.max() < K, "group id out of range"
            assert np.all(G[:, 0] != G[:, 1]), "a token's two groups must differ"
            g_e = G.reshape(m)                        # own group of entry 2i + c
            o_e = G[:, ::-1].reshape(m)               # the other group
            v_e = g_e * K + o_e
            counts[b, a] = np.bincount(v_e, minlength=Kv)
            offsets[b, a, 1:] = np.cumsum(counts[b, a])
            p = np.argsort(v_e, kind="stable")        # by (g, o), then entry = position order
            perm[b, a] = p
            rank[b, a, p] = np.arange(m)
            pos_slot = p // 2
            for s in range(m):
                e = p[s]
                g, o, i = int(g_e[e]), int(o_e[e]), int(e // 2)
                for o2 in range(K):
                    if o2 == g:
                        continue
                    j = o2 if o2 < g else o2 - 1
                    if o2 == o and o < g:
                        continue                      # counted in group o's pass
                    v2 = g * K + o2
                    lo, hi = offsets[b, a, v2], offsets[b, a, v2 + 1]
                    fsub[b, a, s, j] = int(np.searchsorted(pos_slot[lo:hi], i - w + 1, side="left"))
            fent[b, a, p] = fsub[b, a].sum(axis=1)
    return dict(counts=counts, offsets=offsets, perm=perm, rank=rank,
                farlen_sub=fsub, farlen_entry=fent)


def work_items_top2_split(index: dict, BM: int):
    """Group-pass work list over the split index, canonical order
    (b, a, v, row0): one candidate per BM slots of each virtual group
    v = g * K + o.  Its keys are the K - 1 sub-runs (g, o') in increasing o',
    each up to the far prefix of the tile's last row (farlen_sub is
    non-decreasing inside a sub-run), the rows' own sub-run left out when
    o < g; a candidate is emitted when the total is positive.  Each item is
    (b, a, v, row0, rows, keys, key0, 0): keys = the total over the sub-runs,
    key0 = the first slot of group g.  segments(index, item) gives the
    sub-runs' (first slot, length).
    """
    counts, offsets, fs = index["counts"], index["offsets"], index["farlen_sub"]
    B, A, Kv = counts.shape
    K = int(round(math.sqrt(Kv)))
    out = []
    for b in range(B):
        for a in range(A):
            for v in range(Kv):
                c = int(counts[b, a, v])
                o = int(offsets[b, a, v])
                g = v // K
                for t in range(0, c, BM):
                    rows = min(BM, c - t)
                    keys = int(fs[b, a, o + t + rows - 1].sum())
                    if keys > 0:
                        out.append((b, a, v, o + t, rows, keys, int(offsets[b, a, g * K]), 0))
    return np.array(out, dtype=np.int32).reshape(-1, 8)


def segments_top2_split(index: dict, item):
    """The key sub-runs of a split work item: [(first slot, length, column j)]
    for j = 0 .. K - 2 in order; length = the far prefix of the item's last
    row in sub-run (g, o'), o' = j + (j >= g)."""
    b, a, v, row0, rows = (int(x) for x in item[:5])
    Kv = index["counts"].shape[-1]
    K = int(round(math.sqrt(Kv)))
    g = v // K
    last = index["farlen_sub"][b, a, row0 + rows - 1]
    out = []
    for j in range(K - 1):
        o2 = j if j < g else j + 1
        out.append((int(index["offsets"][b, a, g * K + o2]), int(last[j]), j))
    return out


def keep_mask_rows_topk(G, w: int, rows):
    """Top-k keep rule for query rows `rows`: j <= i and (i - j < w or the
    group sets of i and j intersect).  G [n, k].  [FocusJA] 2.2 (a far pair
    is computed only when the tokens share a group; with top-k membership a
    token is in k groups) and 3.3; [FocusKO] 2.3."""
    G = np.asarray(G)
    rows = np.asarray(rows, dtype=np.int64)
    n, k = G.shape
    j = np.arange(n)[None, :]
    i = rows[:, None]
    shared = np.zeros((len(rows), n), dtype=bool)
    for c in range(k):
        for c2 in range(k):
            shared |= G[rows, c][:, None] == G[None, :, c2]
    return (j <= i) & (((i - j) < w) | shared)


def attention_rows_topk(Q, K, V, gid, w: int, scale: float, rows, A: int, row_block: int = 256):
    """Top-k Focus attention for selected query rows of every (b, h):
    Q [B,H,n,d], K/V [B,H_kv,n,d], gid [B,A,n,k].  O [B,H,R,d], LSE [B,H,R].
    Exact softmax over the top-k keep rule's pairs, each pair once ([FocusKO]
    2.1, 2.3; [FocusJA] 2.2)."""
    B, H, n, d = Q.shape
    H_kv = K.shape[1]
    rows = np.asarray(rows, dtype=np.int64)
    O = np.empty((B, H, len(rows), d))
    L = np.empty((B, H, len(rows)))
    for b in range(B):
        for hq in range(H):
            kv = kv_head(hq, H, H_kv)
            a = assignment_of_head(hq, H, H_kv, A)
            Kf, Vf = _f64(K[b, kv]), _f64(V[b, kv])
            for s in range(0, len(rows), row_block):
                r = rows[s:s + row_block]
                M = keep_mask_rows_topk(gid[b, a], w, r)
                O[b, hq, s:s + row_block], L[b, hq, s:s + row_block] = \
                    attention_masked_rows(Q[b, hq], Kf, Vf, M, r, scale)
    return O, L


def attention_bruteforce_topk(q, k, v, G, w: int, scale: float):
    """Scalar loops for one head: kept set per row from the window and set
    intersection, math.fsum softmax.  q, k, v [n, d], G [n, kk] -> O, LSE.
    The same rule as keep_mask_rows_topk built a different way (lists, not a
    mask), for the brute-force pin ([FocusJA] 2.2; [FocusKO] 2.1)."""
    n, d = q.shape
    O = np.zeros((n, d))
    L = np.zeros(n)
    for i in range(n):
        gi = set(int(x) for x in G[i])
        kept = [j for j in range(i + 1) if i - j < w or gi & set(int(x) for x in G[j])]
        s = [scale * math.fsum(float(q[i, t]) * float(k[j, t]) for t in range(d)) for j in kept]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        tot = math.fsum(e)
        for t in range(d):
            O[i, t] = math.fsum(e[r] * float(v[kept[r], t]) for r in range(len(kept))) / tot
        L[i] = mx + math.log(tot)
    return O, L


# --------------------------------------------------------------- sinkhorn ---

def scores(h, W, C):
    """S[b, a, i, k] = p . c_k with p = W_a h_i (fp64, no bias).  [FocusJA] 2.1."""
    h = _f64(h)
    W = _f64(W)
    C = _f64(C)
    B, n, _ = h.shape
    A = W.shape[0]
    K = C.shape[1]
    out = np.empty((B, A, n, K))
    for b in range(B):
        for a in range(A):
            out[b, a] = (h[b] @ W[a].T) @ C[a].T
    return out


def sinkhorn(S, T: int, tau: float = 1.0):
    """Sinkhorn-Knopp scaling of exp(S / tau) for every leading index.
    [FocusJA] 2.3 and [FocusKO] 2.2: the forward assignment matrix is forced
    to be doubly stochastic so that every group receives an equal share of
    the tokens.

    S [..., n, K] -> G [..., n, K] (fp64).  Each of the T >= 1 rounds scales
    the columns to sum n / K, then the rows to sum 1, in the plain probability
    domain.  exp is taken after subtracting the matrix's largest S / tau: a
    constant factor, which the first column step removes exactly.
    """
    assert T >= 1 and tau > 0
    S = _f64(S)
    n, K = S.shape[-2], S.shape[-1]
    X = S / tau
    M = np.exp(X - X.max(axis=(-2, -1), keepdims=True))
    for _ in range(T):
        M = M * ((n / K) / M.sum(axis=-2, keepdims=True))
        M = M / M.sum(axis=-1, keepdims=True)
    return M


# --------------------------------------------------------------- backward ---

def attention_backward(Q, K, V, gid, w: int, scale: float, A: int, dO):
    """Gradients of O = attention(Q, K, V) (the top-1 keep rule) for a fixed
    upstream gradient dO: the exact softmax over the kept pairs ([FocusKO]
    2.1) is what a retrofitted model is fine-tuned through ([FocusJA] 3.1).  Q, dO [B, H, n, d]; K, V [B, H_kv, n, d];
    gid [B, A, n].  Returns dQ [B, H, n, d], dK, dV [B, H_kv, n, d] (fp64).

    Per (b, h), with M the keep mask and P = softmax over kept keys of
    S = scale Q K^T (exact, zero off the mask):
      O = P V,  dV += P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,
      dS = P * (dP - D),  dQ = scale dS K,  dK += scale dS^T Q.
    (D_i equals dO_i . O_i because the rows of P sum to 1.)
    """
    B, H, n, d = Q.shape
    H_kv = K.shape[1]
    dQ = np.zeros((B, H, n, d))
    dK = np.zeros((B, H_kv, n, d))
    dV = np.zeros((B, H_kv, n, d))
    rows = np.arange(n)
    for b in range(B):
        for hq in range(H):
            kv = kv_head(hq, H, H_kv)
            a = assignment_of_head(hq, H, H_kv, A)
            q, k, v, do = _f64(Q[b, hq]), _f64(K[b, kv]), _f64(V[b, kv]), _f64(dO[b, hq])
            M = keep_mask_rows(gid[b, a], w, rows)
            P = attention_weights_rows(q, k, M, rows, scale)
            dP = do @ v.T
            Dv = np.sum(P * dP, axis=1, keepdims=True)
            dS = P * (dP - Dv)
            dQ[b, hq] = scale * (dS @ k)
            dK[b, kv] += scale * (dS.T @ q)
            dV[b, kv] += P.T @ do
    return dQ, dK, dV


def attention_backward_dkv_rows(Q, K, V, gid, w: int, scale: float, A: int, dO, krows):
    """dK and dV of attention_backward for selected key rows only.  Key j
    receives gradient from every query i that keeps it (i >= j and i - j < w,
    or g_i = g_j), through that query's full softmax row:
      dV_j = sum_h sum_i P_ij dO_i,   dK_j = scale sum_h sum_i dS_ij q_i,
    h over the query heads of j's KV head.  The query rows are gathered from
    the keep rule column by column, their softmax rows computed in full
    ([FocusKO] 2.1), and only the columns krows kept.  Returns dK, dV
    [B, H_kv, R, d] (fp64)."""
    B, H, n, d = Q.shape
    H_kv = K.shape[1]
    krows = np.asarray(krows, dtype=np.int64)
    dK = np.zeros((B, H_kv, len(krows), d))
    dV = np.zeros((B, H_kv, len(krows), d))
    for b in range(B):
        for hq in range(H):
            kv = kv_head(hq, H, H_kv)
            a = assignment_of_head(hq, H, H_kv, A)
            g = np.asarray(gid[b, a])
            # the queries that keep at least one of the selected keys
            need = np.zeros(n, dtype=bool)
            for j in krows:
                i = np.arange(j, n)
                need[i[((i - j) < w) | (g[i] == g[j])]] = True
            rows = np.nonzero(need)[0]
            q, k, v, do = _f64(Q[b, hq])[rows], _f64(K[b, kv]), _f64(V[b, kv]), _f64(dO[b, hq])[rows]
            M = keep_mask_rows(g, w, rows)
            P = attention_weights_rows(_f64(Q[b, hq]), k, M, rows, scale)
            dP = do @ v.T
            dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
            dK[b, kv] += scale * (dS[:, krows].T @ q)
            dV[b, kv] += P[:, krows].T @ do
    return dK, dV


def attention_backward_dq_rows(Q, K, V, gid, w: int, scale: float, A: int, dO, rows):
    """dQ of attention_backward for selected query rows only (each row's dQ
    needs only its own kept keys): dQ_i = scale sum_j P_ij (dO_i . v_j - D_i) k_j.
    Returns [B, H, R, d].  The same definition as attention_backward
    ([FocusKO] 2.1), restricted to rows."""
    B, H, n, d = Q.shape
    H_kv = K.shape[1]
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((B, H, len(rows), d))
    for b in range(B):
        for hq in range(H):
            kv = kv_head(hq, H, H_kv)
            a = assignment_of_head(hq, H, H_kv, A)
            k, v = _f64(K[b, kv]), _f64(V[b, kv])
            M = keep_mask_rows(gid[b, a], w, rows)
            P = attention_weights_rows(_f64(Q[b, hq]), k, M, rows, scale)
            do = _f64(dO[b, hq])[rows]
            dP = do @ v.T
            dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
            out[b, hq] = scale * (dS @ k)
    return out
