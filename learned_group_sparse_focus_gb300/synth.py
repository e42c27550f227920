"""Seeded synthetic inputs for the Focus attention hot path.

This module only draws random numbers and rounds them to the storage dtype.
It computes nothing of the method itself (no projection, no scores, no
argmax, no mask, no softmax): it is the one module shared by the test oracle
side and the GPU side, so it must stay free of the method's arithmetic.

Workloads mirror the model shapes the Focus pages report results on
("Focus: Learning Which Attention Pairs Matter", section 3.1: GPT-2 124M up to
LLaMA-2 70B; section 3.3: long sequences).  The pages publish no dataset that
fits here and no trained centroids, so every tensor is synthetic:

* h, Q, K, V ~ N(0, 1); W ~ N(0, 1/D) (std 1/sqrt(hidden));
  C rows are unit-norm Gaussian directions (uniform on the sphere).
* "zipf" workloads plant skewed group sizes: token i draws a target centroid
  t_i from a truncated Zipf(s=1.1) law over the K ranks (ranks mapped to
  centroid ids by a seeded permutation) and its hidden state becomes
  h_i = z_i + 6 * W^T c_{t_i} with z_i ~ N(0, 1).  With W W^T close to the
  identity this moves the projection next to c_{t_i}, so group sizes follow
  the Zipf law (largest group about a quarter of the tokens at K=32..64).
* Values are rounded to the workload dtype (bf16 round-to-nearest-even, or
  fp32) and returned as float32 numpy arrays holding exactly representable
  values, plus helpers that give the raw bf16 bit patterns for upload.

Random streams are keyed by (seed, tensor tag), so drawing one tensor never
shifts another.  ``redraw_hidden`` replaces chosen tokens' hidden states with
fresh draws from a stream keyed by the attempt number; the caller decides which
tokens to redraw (the argmax-margin filter lives with the caller).
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "draw", "redraw_hidden",
    "round_bf16", "bf16_bits", "draw_group_ids", "draw_group_ids_topk",
]

_TAGS = {"h": 1, "W": 2, "C": 3, "Q": 4, "K": 5, "V": 6, "target": 7,
         "perm": 8, "redraw": 9, "gid": 10, "gid-topk": 11}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int          # batch
    H: int          # query heads
    H_kv: int       # key/value heads (GQA when < H)
    n: int          # tokens
    d: int          # head dim
    D: int          # hidden size
    d_g: int        # projection (centroid space) dim
    K: int          # centroids (groups)
    w: int          # local window
    A: int          # independent assignments: 1 (shared by all heads) or H_kv
    dtype: str      # "f32" or "bf16"
    groups: str     # "uniform" or "zipf"
    seed: int

    def asdict(self):
        return asdict(self)

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))


# Five workloads: a tiny fp32 case and four bf16 layers shaped like the
# GPT-2-small, 7B, 32K-context GQA and 70B prefill settings.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", B=1, H=2, H_kv=2, n=256, d=64, D=128, d_g=64,
                          K=4, w=32, A=1, dtype="f32", groups="uniform", seed=1001),
    "gpt2_small_1k": Workload("gpt2_small_1k", B=8, H=12, H_kv=12, n=1024, d=64, D=768,
                              d_g=64, K=16, w=64, A=1, dtype="bf16", groups="uniform",
                              seed=1002),
    "llama7b_8k": Workload("llama7b_8k", B=1, H=32, H_kv=32, n=8192, d=128, D=4096,
                           d_g=64, K=32, w=256, A=1, dtype="bf16", groups="zipf",
                           seed=1003),
    "gqa_32k": Workload("gqa_32k", B=1, H=32, H_kv=8, n=32768, d=128, D=4096, d_g=64,
                        K=64, w=512, A=1, dtype="bf16", groups="zipf", seed=1004),
    "llama70b_64k": Workload("llama70b_64k", B=1, H=64, H_kv=8, n=65536, d=128, D=8192,
                             d_g=64, K=64, w=1024, A=8, dtype="bf16", groups="uniform",
                             seed=1005),
}


def workload(name: str, **override) -> Workload:
    """Named workload, optionally with fields replaced (e.g. a smaller n)."""
    base = WORKLOADS[name].asdict()
    base.update(override)
    if "name" not in override:
        base["name"] = name if not override else name + "+" + ",".join(
            f"{k}={v}" for k, v in sorted(override.items()))
    return Workload(**base)


def _rng(seed: int, tag: str, extra: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _TAGS[tag], extra])))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); float32 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    r = ((u + bias) & np.uint32(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (int16 view) of float32 values already on the bf16 grid."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16).view(np.int16)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    x = x.astype(np.float32, copy=False)
    return round_bf16(x) if dtype == "bf16" else np.ascontiguousarray(x)


def _normal(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def _unit_rows(rng, rows, cols):
    c = rng.standard_normal(size=(rows, cols))
    c /= np.linalg.norm(c, axis=1, keepdims=True)
    return c


def _zipf_targets(wl: Workload) -> np.ndarray:
    """Per-token target centroid ids, truncated Zipf(s=1.1) over K ranks."""
    rng = _rng(wl.seed, "target")
    ranks = np.arange(1, wl.K + 1, dtype=np.float64)
    p = ranks ** -1.1
    p /= p.sum()
    r = rng.choice(wl.K, size=(wl.B, wl.n), p=p)
    ids = _rng(wl.seed, "perm").permutation(wl.K)
    return ids[r].astype(np.int64)


def _hidden_from_noise(wl: Workload, z: np.ndarray, W: np.ndarray, C: np.ndarray,
                       target: np.ndarray | None) -> np.ndarray:
    if target is None:
        return z
    # plant: h = z + 6 * W_0^T c_t   (A == 1 for the skewed workloads)
    shift = 6.0 * (C[0].astype(np.float64) @ W[0].astype(np.float64))   # [K, D]
    return (z.astype(np.float64) + shift[target]).astype(np.float32)


def draw(wl: Workload, parts=("assign", "attn")) -> dict:
    """Draw the workload's inputs as float32 arrays on the dtype grid.

    parts: "assign" -> h [B,n,D], W [A,d_g,D], C [A,K,d_g] (and target for zipf)
           "attn"   -> Q [B,H,n,d], K/V [B,H_kv,n,d]
    """
    out = {}
    if "assign" in parts:
        W = _store(_normal(_rng(wl.seed, "W"), (wl.A, wl.d_g, wl.D)) / np.float32(np.sqrt(wl.D)), wl.dtype)
        C = _store(np.stack([_unit_rows(_rng(wl.seed, "C", a), wl.K, wl.d_g) for a in range(wl.A)]), wl.dtype)
        z = _normal(_rng(wl.seed, "h"), (wl.B, wl.n, wl.D))
        target = _zipf_targets(wl) if wl.groups == "zipf" else None
        if target is not None and wl.A != 1:
            raise ValueError("zipf planting is defined for one shared assignment")
        out.update(h=_store(_hidden_from_noise(wl, z, W, C, target), wl.dtype), W=W, C=C)
        if target is not None:
            out["target"] = target
    if "attn" in parts:
        out["Q"] = _store(_normal(_rng(wl.seed, "Q"), (wl.B, wl.H, wl.n, wl.d)), wl.dtype)
        out["K"] = _store(_normal(_rng(wl.seed, "K"), (wl.B, wl.H_kv, wl.n, wl.d)), wl.dtype)
        out["V"] = _store(_normal(_rng(wl.seed, "V"), (wl.B, wl.H_kv, wl.n, wl.d)), wl.dtype)
    return out


def redraw_hidden(wl: Workload, inputs: dict, tokens: np.ndarray, attempt: int) -> None:
    """Replace hidden states of the given (b, i) tokens in place with fresh draws.

    tokens: int array [m, 2] of (b, i).  The fresh noise comes from a stream
    keyed by (seed, attempt), drawn for all m tokens at once in the given order.
    """
    tokens = np.asarray(tokens, dtype=np.int64).reshape(-1, 2)
    if len(tokens) == 0:
        return
    z = _normal(_rng(wl.seed, "redraw", attempt), (len(tokens), wl.D))
    tgt = inputs.get("target")
    t = tgt[tokens[:, 0], tokens[:, 1]] if tgt is not None else None
    h = _hidden_from_noise(wl, z, inputs["W"], inputs["C"], t)
    inputs["h"][tokens[:, 0], tokens[:, 1]] = _store(h, wl.dtype)


def draw_group_ids(seed: int, B: int, A: int, n: int, K: int, kind: str = "uniform") -> np.ndarray:
    """Group ids drawn directly (for tests that inject an assignment).

    kind: "uniform" (iid uniform over K), "zipf" (truncated Zipf(1.1)),
          "distinct" (a random permutation of 0..n-1; needs K >= n),
          "one" (every token in group 0), "blocks" (contiguous runs).
    """
    rng = _rng(seed, "gid")
    if kind == "uniform":
        g = rng.integers(0, K, size=(B, A, n))
    elif kind == "zipf":
        p = np.arange(1, K + 1, dtype=np.float64) ** -1.1
        g = rng.choice(K, size=(B, A, n), p=p / p.sum())
    elif kind == "distinct":
        if K < n:
            raise ValueError("distinct ids need K >= n")
        g = np.stack([np.stack([rng.permutation(K)[:n] for _ in range(A)]) for _ in range(B)])
    elif kind == "one":
        g = np.zeros((B, A, n), dtype=np.int64)
    elif kind == "blocks":
        run = max(1, n // max(1, K))
        g = np.minimum(np.arange(n) // run, K - 1)[None, None, :].repeat(B, 0).repeat(A, 1)
    else:
        raise ValueError(kind)
    return np.ascontiguousarray(g, dtype=np.int32)


def draw_group_ids_topk(seed: int, B: int, A: int, n: int, K: int, k: int,
                        kind: str = "uniform") -> np.ndarray:
    """k distinct group ids per token, [B, A, n, k] (for tests and benchmarks
    that inject a top-k assignment).

    kind: "uniform" (each ordered k-subset equally likely), "zipf" (ids drawn
          from truncated Zipf(1.1), repeats redrawn), "both" (every token in
          groups 0 and 1, in a random order; needs k = 2).
    """
    if not 1 <= k <= K:
        raise ValueError("need 1 <= k <= K")
    rng = _rng(seed, "gid-topk")
    shape = (B, A, n)
    if kind == "both":
        if k != 2:
            raise ValueError("'both' is a k = 2 pattern")
        first = rng.integers(0, 2, size=shape)
        g = np.stack([first, 1 - first], axis=-1)
    elif kind in ("uniform", "zipf"):
        p = None
        if kind == "zipf":
            p = np.arange(1, K + 1, dtype=np.float64) ** -1.1
            p /= p.sum()
        g = np.empty(shape + (k,), dtype=np.int64)
        for c in range(k):
            col = rng.choice(K, size=shape, p=p)
            while True:
                clash = np.zeros(shape, dtype=bool)
                for c2 in range(c):
                    clash |= col == g[..., c2]
                if not clash.any():
                    break
                col[clash] = rng.choice(K, size=int(clash.sum()), p=p)
            g[..., c] = col
    else:
        raise ValueError(kind)
    return np.ascontiguousarray(g, dtype=np.int32)
