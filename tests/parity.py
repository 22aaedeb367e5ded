"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI and
the oracle on the same seeded inputs and compare with the stated tolerances.

Tolerances (bf16 outputs and gradients, against the oracle's bf16 flow):
max relative error 2e-2 and mean relative error 2e-3, with
max_rel = max_i |g_i - o_i| / max(|o_i|, rms(o)) and mean_rel = sum|g-o| / sum|o|.
"""

import numpy as np
import torch

import oracle
from rank_bottleneck_online_gb300 import inputs

MAX_REL = 2e-2
MEAN_REL = 2e-3


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(name, got, want, max_rel=MAX_REL, mean_rel=MEAN_REL):
    g = to_np(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    assert g.shape == w.shape, (name, g.shape, w.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    mx, mean = oracle.rel_errors(g, w)
    assert mx <= max_rel and mean <= mean_rel, f"{name}: max_rel={mx:.3e} mean_rel={mean:.3e}"
    return mx, mean


def oracle_block(w, *, act, has_norm, S, eps=1e-5):
    x = inputs.as_f64(w["x"])
    g = inputs.as_f64(w["gamma"]) if has_norm else None
    A = inputs.as_f64(w["A"])
    Bw = inputs.as_f64(w["B"])
    dy = inputs.as_f64(w["dy"])
    y, c = oracle.block_fwd(x, g, A, Bw, act=act, has_norm=has_norm, eps=eps, S=S, flow="bf16")
    gr = oracle.block_bwd(x, g, A, Bw, dy, act=act, has_norm=has_norm, eps=eps, S=S, flow="bf16")
    return y, c, gr


def random_block_shapes(count=16, seed=2026):
    """Block shapes drawn once from a fixed seed within the library's shape rules (d, r,
    n multiples of 8; S divides d when normed; k * r <= 1024, d <= 1024, n <= 2048,
    T <= 5000, so the oracle takes seconds): any mix of ragged tails, group widths,
    group counts, row splits and split-K plans the planner picks for them. Each is
    (name, T, d, r, k, n, S, act, has_norm)."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        has_norm = bool(rng.integers(0, 4) > 0)
        d = 8 * int(rng.integers(1, 129))
        S = int(rng.choice([s for s in (1, 2, 4, 8) if d % s == 0])) if has_norm else 1
        k = int(rng.integers(1, 5))
        r = 8 * int(rng.integers(1, 1024 // (8 * k) + 1))
        n = 8 * int(rng.integers(1, 257))
        T = int(rng.integers(1, 5001))
        act = "silu" if rng.integers(0, 5) > 0 else "identity"
        out.append((f"rand{i}_T{T}_d{d}_r{r}_k{k}_n{n}", T, d, r, k, n, S, act, has_norm))
    return out


def random_mlp_shapes(count=6, seed=2027):
    """LLaMA-MLP shapes (T, d, r, ffn, S) drawn once from a fixed seed within the shape
    rules (d, r, ffn multiples of 8, S divides d; T <= 4000, d <= 1024, r <= 512,
    ffn <= 2048)."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        d = 8 * int(rng.integers(1, 129))
        S = int(rng.choice([s for s in (1, 2, 4, 8) if d % s == 0]))
        r = 8 * int(rng.integers(1, 65))
        ffn = 8 * int(rng.integers(1, 257))
        T = int(rng.integers(1, 4001))
        out.append((T, d, r, ffn, S))
    return out
