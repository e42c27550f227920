"""Shared test utilities: device upload, the argmax-margin filter, tolerances,
row sampling.  Inputs come from the seeded generators; expected values come
from the fp64 oracle only."""
from __future__ import annotations

import numpy as np

import oracle.focus_ref as ref
from learned_group_sparse_focus_gb300 import synth

MARGIN = 1e-3          # smallest best-vs-runner-up score gap allowed in inputs
TOL_BF16_MAX = 2e-2
TOL_BF16_MEAN = 2e-3
TOL_F32_MAX = 1e-5
TOL_LSE_BF16 = 1e-3    # natural-log LSE, absolute
TOL_LSE_F32 = 1e-5


def to_dev(x: np.ndarray, dtype: str, device="cuda"):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(synth.bf16_bits(x)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def to_host(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy()


def margin_filtered(wl, parts=("assign", "attn"), max_rounds=30):
    """Draw inputs and redraw hidden states until every token's best centroid
    beats the runner-up by MARGIN in every assignment (fp64 on the stored
    values); returns inputs plus the oracle's gid."""
    x = synth.draw(wl, parts)
    if "assign" not in parts:
        return x
    gid, mg = ref.assign(x["h"], x["W"], x["C"])
    for attempt in range(1, max_rounds + 1):
        bad = np.argwhere((mg < MARGIN).any(axis=1))          # (b, i) pairs
        if len(bad) == 0:
            break
        synth.redraw_hidden(wl, x, bad, attempt)
        hb = x["h"][bad[:, 0], bad[:, 1]][None]                # [1, m, D]
        g2, m2 = ref.assign(hb, x["W"], x["C"])
        gid[bad[:, 0], :, bad[:, 1]] = g2[0].T
        mg[bad[:, 0], :, bad[:, 1]] = m2[0].T
    else:
        raise RuntimeError("margin filter did not converge")
    x["gid_ref"] = gid
    x["margin"] = mg
    return x


def margin_filtered_topk(wl, k, parts=("assign", "attn"), max_rounds=40):
    """margin_filtered for top-k selection: every gap that decides a token's k
    best centroids and their order (ranks 1..k+1) is at least MARGIN."""
    x = synth.draw(wl, parts)
    gid, mg = ref.assign_topk(x["h"], x["W"], x["C"], k)
    for attempt in range(1, max_rounds + 1):
        bad = np.argwhere((mg < MARGIN).any(axis=1))
        if len(bad) == 0:
            break
        synth.redraw_hidden(wl, x, bad, attempt)
        hb = x["h"][bad[:, 0], bad[:, 1]][None]
        g2, m2 = ref.assign_topk(hb, x["W"], x["C"], k)
        gid[bad[:, 0], :, bad[:, 1]] = g2[0].transpose(1, 0, 2)
        mg[bad[:, 0], :, bad[:, 1]] = m2[0].T
    else:
        raise RuntimeError("margin filter did not converge")
    x["gid_ref"] = gid
    x["margin"] = mg
    return x


def assert_close(got, want, dtype, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = np.abs(got - want)
    if dtype == "bf16":
        assert diff.max() <= TOL_BF16_MAX, f"{what}: max abs {diff.max():.3e}"
        assert diff.mean() <= TOL_BF16_MEAN, f"{what}: mean abs {diff.mean():.3e}"
    else:
        assert diff.max() <= TOL_F32_MAX, f"{what}: max abs {diff.max():.3e}"
    return float(diff.max()), float(diff.mean())


def assert_lse_close(got, want, dtype, what=""):
    diff = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))
    tol = TOL_LSE_BF16 if dtype == "bf16" else TOL_LSE_F32
    assert diff.max() <= tol, f"{what}: LSE max abs {diff.max():.3e}"


def sample_rows(index: dict, b: int, a: int, n: int, w: int, seed: int, n_random: int):
    """Rows that exercise every code path: the first w+1 rows (window start),
    the last row, the first row with far keys in each group, all rows of the
    smallest non-empty groups, and seeded random rows."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(n, w + 1)))
    rows.add(n - 1)
    counts = index["counts"][b, a]
    offs = index["offsets"][b, a]
    perm = index["perm"][b, a]
    fs = index["farlen_slot"][b, a]
    for g in range(len(counts)):
        seg = np.arange(offs[g], offs[g + 1])
        far = seg[fs[seg] > 0]
        if len(far):
            rows.add(int(perm[far[0]]))
    nz = [g for g in np.argsort(counts, kind="stable") if counts[g] > 0][:3]
    for g in nz:
        rows.update(int(v) for v in perm[offs[g]:offs[g + 1]][:256])
    rows.update(int(v) for v in rng.integers(0, n, n_random))
    return np.array(sorted(rows), dtype=np.int64)
