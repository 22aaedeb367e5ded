"""Seeded synthetic inputs for the bottleneck block and its composed workloads.

This module draws random tensors and nothing else: it holds none of the
block's arithmetic, so both the CUDA path and the CPU oracle may use it.

Recipe (the LLaMA-2-shaped workloads of the BOOST pages, §4 of their
technical summary, with synthetic values instead of training data):

* one ``torch.Generator`` on the CPU, seeded, drawn in a fixed order:
  x, then per block in layer order gamma (if the block is normed), A, B,
  then the upstream gradients;
* x ~ N(0, 1); gamma = 1 + 0.1 * N(0, 1); A ~ N(0, 1/fan_in) with fan_in the
  block's input width; B ~ N(0, 1/r); upstream gradients ~ N(0, 1);
* SVD-style weights: per group A_i = U_i diag(s_i), B_i = V_i^T with U_i, V_i
  the Q factors of seeded Gaussian matrices and s_i = 10^U(-2, 0);
* everything is drawn in fp32 and cast to bf16 (round to nearest even).

All tensors are returned on the CPU; callers move them where they need them.
"""

from __future__ import annotations

import math

import torch

# Workloads named by what they are and their sizes.
CONFIGS = {
    "tiny_block": dict(kind="block", T=128, d=256, r=64, k=3, n=256, S=4, act="silu"),
    "llama2_1b_attn_block": dict(kind="block", T=16384, d=2048, r=512, k=3, n=2048, S=4,
                                 act="silu"),
    "llama2_7b_mlp": dict(kind="mlp", T=16384, d=4096, r=1024, ffn=11008, S=8, act="silu"),
    "llama2_13b_layer": dict(kind="layer", T=16384, d=5120, r=1280, ffn=13824, S=8,
                             act="silu"),
    "svd_40b_pair": dict(kind="svd_pair", T=8192, d=8192, r=2048, ffn=22016, S=8,
                         act="identity"),
}


def _normal(g, shape, std=1.0, mean=0.0):
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t = t * std
    if mean != 0.0:
        t = t + mean
    return t.to(torch.bfloat16)


def _block_weights(g, d, r, k, n, has_norm):
    out = {}
    if has_norm:
        out["gamma"] = _normal(g, (d,), std=0.1, mean=1.0)
    out["A"] = _normal(g, (d, k * r), std=1.0 / math.sqrt(d))
    out["B"] = _normal(g, (k, r, n), std=1.0 / math.sqrt(r))
    return out


def make_block(T, d, r, k, n, *, has_norm=True, seed=0):
    """x [T,d], gamma [d] (normed blocks), A [d,k*r], B [k,r,n], dy [k,T,n]."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = _normal(g, (T, d))
    w = _block_weights(g, d, r, k, n, has_norm)
    dy = _normal(g, (k, T, n))
    return {"x": x, "gamma": w.get("gamma"), "A": w["A"], "B": w["B"], "dy": dy}


def make_mlp(T, d, r, ffn, *, seed=0):
    """Gate/up block (normed, k=2, d->ffn) and down block (k=1, ffn->d), plus dout."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = _normal(g, (T, d))
    w1 = _block_weights(g, d, r, 2, ffn, True)
    w2 = _block_weights(g, ffn, r, 1, d, False)
    dout = _normal(g, (T, d))
    return {"x": x, "gamma": w1["gamma"], "A1": w1["A"], "B1": w1["B"],
            "A2": w2["A"], "B2": w2["B"], "dout": dout}


def make_layer(T, d, r, ffn, *, seed=0):
    """QKV (normed, k=3), O (k=1), gate/up (normed, k=2), down (k=1); dout, dq, dk."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = _normal(g, (T, d))
    qkv = _block_weights(g, d, r, 3, d, True)
    o = _block_weights(g, d, r, 1, d, False)
    gu = _block_weights(g, d, r, 2, ffn, True)
    dn = _block_weights(g, ffn, r, 1, d, False)
    p = {"gamma1": qkv["gamma"], "A_qkv": qkv["A"], "B_qkv": qkv["B"],
         "A_o": o["A"], "B_o": o["B"],
         "gamma2": gu["gamma"], "A_gu": gu["A"], "B_gu": gu["B"],
         "A_dn": dn["A"], "B_dn": dn["B"]}
    dout = _normal(g, (T, d))
    dq = _normal(g, (T, d))
    dk = _normal(g, (T, d))
    return {"x": x, "p": p, "dout": dout, "dq": dq, "dk": dk}


def _svd_weights(g, d, r, k, n):
    A = torch.empty(d, k * r, dtype=torch.float32)
    B = torch.empty(k, r, n, dtype=torch.float32)
    svals = torch.empty(k, r, dtype=torch.float32)
    for i in range(k):
        U, _ = torch.linalg.qr(torch.randn(d, r, generator=g, dtype=torch.float32))
        V, _ = torch.linalg.qr(torch.randn(n, r, generator=g, dtype=torch.float32))
        s = torch.pow(10.0, torch.rand(r, generator=g, dtype=torch.float32) * 2.0 - 2.0)
        A[:, i * r:(i + 1) * r] = U * s[None, :]
        B[i] = V.T
        svals[i] = s
    return A.to(torch.bfloat16), B.to(torch.bfloat16), svals


def make_svd_pair(T, d, r, ffn, *, seed=0):
    """Two normed SVD-style blocks on one x: QKV (k=3, d->d) and gate/up (k=2, d->ffn)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = _normal(g, (T, d))
    gq = _normal(g, (d,), std=0.1, mean=1.0)
    Aq, Bq, sq = _svd_weights(g, d, r, 3, d)
    gg = _normal(g, (d,), std=0.1, mean=1.0)
    Ag, Bg, sg = _svd_weights(g, d, r, 2, ffn)
    dy_qkv = _normal(g, (3, T, d))
    dy_gu = _normal(g, (2, T, ffn))
    p = {"gamma_qkv": gq, "A_qkv": Aq, "B_qkv": Bq, "gamma_gu": gg, "A_gu": Ag, "B_gu": Bg}
    return {"x": x, "p": p, "dy_qkv": dy_qkv, "dy_gu": dy_gu,
            "svals_qkv": sq, "svals_gu": sg}


def make_inputs(name, *, seed=0, T=None):
    """Inputs of a named workload; ``T`` overrides the token count (for samples)."""
    c = dict(CONFIGS[name])
    if T is not None:
        c["T"] = T
    if c["kind"] == "block":
        return make_block(c["T"], c["d"], c["r"], c["k"], c["n"], seed=seed)
    if c["kind"] == "mlp":
        return make_mlp(c["T"], c["d"], c["r"], c["ffn"], seed=seed)
    if c["kind"] == "layer":
        return make_layer(c["T"], c["d"], c["r"], c["ffn"], seed=seed)
    if c["kind"] == "svd_pair":
        return make_svd_pair(c["T"], c["d"], c["r"], c["ffn"], seed=seed)
    raise KeyError(name)


def as_f64(t):
    """bf16 CPU tensor -> fp64 numpy array (exact)."""
    import numpy as np
    if t is None:
        return None
    return t.to(torch.float64).numpy().astype(np.float64, copy=False)
