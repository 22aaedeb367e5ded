"""fp64 CPU oracle of the low-rank bottleneck block (TEST INFRASTRUCTURE ONLY).

Source: "BOOST: BOttleneck-Optimized Scalable Training Framework for Low-Rank
Large Language Models" (arXiv 2512.12131), as summarised on gist.science in
Chinese and French. Section references below are to the technical summary on
those pages:

* §2.1 (Bottleneck-aware TP): a low-rank layer is a pair d x r / r x d;
  the all-reduce payload shrinks from [b,s,d] to [b,s,r].
* §2.2 "Online-RMSNorm": local (per-shard) statistics, deferred global
  normalisation, statistics exchange fused into the following all-reduce,
  mathematically equivalent to RMSNorm.
* §2.2 "Linear-layer grouping": down-projections that share an input run as
  one GEMM over concatenated weights; up-projections with distinct inputs run
  as one batched GEMM.
* §2.2 "Communication-free low-rank activation checkpointing": the re-forward
  path lies inside one block; backward recomputes it there.
* §4 (Experimental results): CoLA, SVD and LaX bottlenecks on LLaMA-2 shapes.

Notation (row-major): x [T,d], gamma [d], A [d, k*r] (group i = columns
[i*r, (i+1)*r)), B [k, r, n], y [k, T, n], s = rstd [T].

Two families of functions:

* ``*_reference``: the plain definition (direct RMSNorm, one projection pair
  per group, textbook chain rule through the full RMSNorm Jacobian). fp64,
  no rounding.
* ``block_fwd`` / ``block_bwd``: the method's own steps in the pages' order
  (sharded statistics, one combine, deferred 1/rms, grouped down-projection,
  batched up-projection, recompute in backward). With ``flow="exact"`` they
  must equal the reference to fp64 rounding; with ``flow="bf16"`` values are
  rounded to bfloat16 at the storage points the method has (inputs, the folded
  weight gamma*A, the bottleneck activation a, the scaled gradient s*dz, and
  the intermediate tensors of a composed layer). Outputs are never rounded.

Readings where the pages are silent (the pages give no formulas):
eps = 1e-5 inside the square root; the mean divides by the full d; shards
are contiguous equal slices of d; sigma = SiLU (identity for the SVD
variant); gamma is folded into the down-projection weight.

Parity status: pinned (see tests/test_oracle_*.py); no function here is
"parity unpinned".
"""

from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# bfloat16 rounding, from the IEEE-754 binary definition of the format:
# 1 sign bit, 8 exponent bits (bias 127), 7 stored fraction bits.
# ---------------------------------------------------------------------------

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
_BF16_MIN_EXP = -126          # smallest normal exponent
_BF16_FRAC_BITS = 7


def to_bf16(v):
    """Round fp64 values to the nearest bfloat16 value, ties to even.

    Directly from fp64 (no intermediate fp32 step, so no double rounding).
    The quantum of a value with leading-bit exponent e is 2^(e-7), never
    smaller than the subnormal quantum 2^(-126-7). np.rint rounds halves to
    even. A result at or beyond 2^128 overflows to infinity. Returns fp64
    arrays whose values are exactly representable in bfloat16.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.array(v, dtype=np.float64, copy=True)
    finite = np.isfinite(v) & (v != 0.0)
    if np.any(finite):
        vf = v[finite]
        _, e2 = np.frexp(vf)                 # |vf| = m * 2^e2, m in [0.5, 1)
        lead = e2 - 1                        # exponent of the leading bit
        qexp = np.maximum(lead - _BF16_FRAC_BITS, _BF16_MIN_EXP - _BF16_FRAC_BITS)
        r = np.ldexp(np.rint(np.ldexp(vf, -qexp)), qexp)
        r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, vf), r)
        out[finite] = r
    return out


def _round_fn(flow):
    if flow == "exact":
        return lambda t: np.asarray(t, dtype=np.float64)
    if flow == "bf16":
        return to_bf16
    raise ValueError(f"flow must be 'exact' or 'bf16', got {flow!r}")


# ---------------------------------------------------------------------------
# Bottleneck nonlinearity. The pages name none; the CoLA variant uses SiLU and
# the SVD variant has no inner nonlinearity (§4 lists both variants).
# ---------------------------------------------------------------------------

def silu(z):
    """SiLU(z) = z * logistic(z) = z / (1 + e^-z)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def silu_grad(z):
    """d SiLU / dz = g(z) * (1 + z * (1 - g(z))), g = logistic."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        g = 1.0 / (1.0 + np.exp(-z))
    return g * (1.0 + z * (1.0 - g))


def identity(z):
    return np.asarray(z, dtype=np.float64)


def identity_grad(z):
    return np.ones_like(np.asarray(z, dtype=np.float64))


act_fns = {"silu": (silu, silu_grad), "identity": (identity, identity_grad)}


# ---------------------------------------------------------------------------
# Bookkeeping (exact integers): where the shards and the groups sit, and the
# size of the one exchange Online-RMSNorm fuses into (§2.1, §2.2).
# ---------------------------------------------------------------------------

def shard_bounds(d, S):
    """Column offsets of S contiguous equal shards of the hidden dim d.

    Shard s covers columns [off[s], off[s+1]). Requires d % S == 0.
    """
    if S < 1 or d % S != 0:
        raise ValueError(f"d={d} is not divisible into S={S} equal shards")
    w = d // S
    return [s * w for s in range(S + 1)]


def group_bounds(k, r):
    """Column offsets of the k concatenated down-projection groups in A."""
    return [i * r for i in range(k + 1)]


def exchange_elems(T, k, r):
    """Values per exchange when the statistics ride on the bottleneck reduce.

    Under bottleneck-aware TP the all-reduce after the row-parallel
    down-projection carries [T, k*r] partial products (§2.1); Online-RMSNorm
    fuses the per-row sum-of-squares into the same exchange (§2.2), one more
    value per row.
    """
    return T * (k * r + 1)


# ---------------------------------------------------------------------------
# Online-RMSNorm statistics (§2.2): per-shard partial sums of squares, then
# one combine over the shards.
# ---------------------------------------------------------------------------

def rmsnorm_stats(x, S, eps):
    """ssq[s, t] = sum_{j in shard s} x[t, j]^2 ; rstd[t] = (sum_s ssq / d + eps)^-1/2."""
    x = np.asarray(x, dtype=np.float64)
    T, d = x.shape
    off = shard_bounds(d, S)
    ssq = np.empty((S, T), dtype=np.float64)
    for s in range(S):
        xs = x[:, off[s]:off[s + 1]]
        ssq[s] = np.sum(xs * xs, axis=1)
    total = np.zeros(T, dtype=np.float64)
    for s in range(S):                      # the single combine, in shard order
        total = total + ssq[s]
    rstd = 1.0 / np.sqrt(total / d + eps)
    return ssq, rstd


# ---------------------------------------------------------------------------
# The bottleneck-aware TP exchange (§2.1, with the statistics fused in per
# §2.2), written out for S ranks on one host: what each rank sends, and the
# reduction that replaces the all-reduce.
# ---------------------------------------------------------------------------

def btp_shard_partials(x, gamma, A, S, *, has_norm=True, flow="bf16"):
    """What each of S tensor-parallel ranks contributes to the exchange.

    Rank s holds columns [shard s] of x and rows [shard s] of the folded weight
    A' (the down-projection is row-parallel, §2.1). It forms the unscaled
    partial product x[:, shard s] @ A'[shard s, :] and, for a normed block, its
    shard's per-row sums of squares (Online-RMSNorm, §2.2).
    Returns (zpart [S, T, k*r], ssq [S, T] or None).
    """
    R = _round_fn(flow)
    x = R(x)
    A = R(A)
    T, d = x.shape
    off = shard_bounds(d, S)
    Ap = R(R(gamma)[:, None] * A) if has_norm else A
    zpart = np.empty((S, T, A.shape[1]))
    ssq = np.empty((S, T)) if has_norm else None
    for s in range(S):
        xs = x[:, off[s]:off[s + 1]]
        zpart[s] = xs @ Ap[off[s]:off[s + 1], :]
        if has_norm:
            ssq[s] = np.sum(xs * xs, axis=1)
    return zpart, ssq


def btp_reduce(zpart, ssq, d, *, act="silu", eps=1e-5, flow="bf16"):
    """The exchange's reduction and the deferred normalisation after it.

    Sums the partial products and the sums of squares over the ranks (shard
    order), forms the row scale s from the full-d mean, and applies it and the
    activation: z = s * sum_s zpart[s], a = act(z). Returns (a, s).
    """
    R = _round_fn(flow)
    f, _ = act_fns[act]
    S, T, _ = zpart.shape
    zsum = np.zeros(zpart.shape[1:])
    for s in range(S):
        zsum = zsum + zpart[s]
    if ssq is not None:
        total = np.zeros(T)
        for s in range(S):
            total = total + ssq[s]
        srow = 1.0 / np.sqrt(total / d + eps)
    else:
        srow = np.ones(T)
    return R(f(srow[:, None] * zsum)), srow


# ---------------------------------------------------------------------------
# Plain definition (no sharding, no deferral, no grouping, no rounding).
# ---------------------------------------------------------------------------

def block_fwd_reference(x, gamma, A, B, *, act="silu", has_norm=True, eps=1e-5):
    """y_i = act(RMSNorm(x) @ A_i) @ B_i, one projection pair per group."""
    f, _ = act_fns[act]
    x = np.asarray(x, np.float64)
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    T, d = x.shape
    k, r, n = B.shape
    if has_norm:
        g = np.asarray(gamma, np.float64)
        rms = np.sqrt(np.mean(x * x, axis=1) + eps)
        h = g[None, :] * x / rms[:, None]
    else:
        h = x
    y = np.empty((k, T, n))
    z = np.empty((T, k * r))
    for i in range(k):
        zi = h @ A[:, i * r:(i + 1) * r]
        z[:, i * r:(i + 1) * r] = zi
        y[i] = f(zi) @ B[i]
    return y, {"h": h, "z": z}


def block_bwd_reference(x, gamma, A, B, dy, *, act="silu", has_norm=True, eps=1e-5):
    """Textbook chain rule of block_fwd_reference.

    Returns dict with dx, dgamma (None without norm), dA, dB. The input
    gradient goes through the full RMSNorm Jacobian:
      u = x / rms, h = gamma * u, du = gamma * dh,
      dx = (du - u * mean(du * u)) / rms.
    """
    f, fp = act_fns[act]
    x = np.asarray(x, np.float64)
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    dy = np.asarray(dy, np.float64)
    T, d = x.shape
    k, r, n = B.shape
    if has_norm:
        g = np.asarray(gamma, np.float64)
        rms = np.sqrt(np.mean(x * x, axis=1) + eps)
        u = x / rms[:, None]
        h = g[None, :] * u
    else:
        h = x
    dA = np.empty_like(A)
    dB = np.empty_like(B)
    dh = np.zeros((T, d))
    for i in range(k):
        Ai = A[:, i * r:(i + 1) * r]
        zi = h @ Ai
        ai = f(zi)
        dB[i] = ai.T @ dy[i]
        dai = dy[i] @ B[i].T
        dzi = dai * fp(zi)
        dA[:, i * r:(i + 1) * r] = h.T @ dzi
        dh += dzi @ Ai.T
    if has_norm:
        dgamma = np.sum(dh * u, axis=0)
        du = g[None, :] * dh
        dx = (du - u * np.mean(du * u, axis=1, keepdims=True)) / rms[:, None]
    else:
        dgamma = None
        dx = dh
    return {"dx": dx, "dgamma": dgamma, "dA": dA, "dB": dB}


# ---------------------------------------------------------------------------
# The method's own steps (§2.2): sharded statistics, one combine, gamma folded
# into the concatenated down-projection weight, 1/rms applied to the GEMM
# result (the normalised activation is never formed), one batched
# up-projection; backward recomputes z and a from x inside the block.
# ---------------------------------------------------------------------------

def block_fwd(x, gamma, A, B, *, act="silu", has_norm=True, eps=1e-5, S=1, flow="bf16"):
    """Forward of one bottleneck block, method order.

    Returns (y, cache) with y [k, T, n] unrounded and cache holding ssq, s,
    Ap (folded weight), z and a as the method forms them.
    """
    R = _round_fn(flow)
    f, _ = act_fns[act]
    x = R(x)
    A = R(A)
    B = R(B)
    T, d = x.shape
    k, r, n = B.shape
    if has_norm:
        g = R(gamma)
        ssq, s = rmsnorm_stats(x, S, eps)
        Ap = R(g[:, None] * A)                  # fold gamma into the weight
    else:
        ssq, s = None, np.ones(T)
        Ap = A
    z = s[:, None] * (x @ Ap)                   # one GEMM over the concatenation
    a = R(f(z))                                 # bottleneck activation
    y = np.empty((k, T, n))
    for i in range(k):                          # the batched up-projection
        y[i] = a[:, i * r:(i + 1) * r] @ B[i]
    return y, {"ssq": ssq, "s": s, "Ap": Ap, "z": z, "a": a}


def block_bwd(x, gamma, A, B, dy, *, act="silu", has_norm=True, eps=1e-5, S=1, flow="bf16"):
    """Backward of one bottleneck block, method order, with recompute.

    Only x (and optionally s) is kept from the forward; z and a are
    regenerated here (§2.2, activation checkpointing inside the block).
    Writing dzs = s * dz:
      dB_i = a_i^T dy_i,  G = x^T dzs,  dA = gamma * G (rows),
      dgamma_j = sum_m A_jm G_jm,
      gs = dzs @ Ap^T (= s * gamma * dh),  dx = gs - (s^2/d) * x * rowsum(gs * x).
    Returns dict with dx, dgamma, dA, dB and the intermediates a, dzs, q.
    """
    R = _round_fn(flow)
    f, fp = act_fns[act]
    x = R(x)
    A = R(A)
    B = R(B)
    dy = R(dy)
    T, d = x.shape
    k, r, n = B.shape
    if has_norm:
        g = R(gamma)
        _, s = rmsnorm_stats(x, S, eps)
        Ap = R(g[:, None] * A)
    else:
        s = np.ones(T)
        Ap = A
    z = s[:, None] * (x @ Ap)                   # recompute
    a = R(f(z))
    da = np.empty((T, k * r))
    dB = np.empty_like(B)
    for i in range(k):
        cols = slice(i * r, (i + 1) * r)
        da[:, cols] = dy[i] @ B[i].T
        dB[i] = a[:, cols].T @ dy[i]
    dz = da * fp(z)
    dzs = R(s[:, None] * dz)
    G = x.T @ dzs
    gs = dzs @ Ap.T
    if has_norm:
        dA = g[:, None] * G
        dgamma = np.sum(A * G, axis=1)
        dx = gs - (s * s / d)[:, None] * x * np.sum(gs * x, axis=1, keepdims=True)
    else:
        dA = G
        dgamma = None
        dx = gs
    q = np.sum(dz * z, axis=1)
    return {"dx": dx, "dgamma": dgamma, "dA": dA, "dB": dB, "a": a, "dzs": dzs, "q": q}


# ---------------------------------------------------------------------------
# SwiGLU glue between the gate/up bottleneck and the down bottleneck of a
# LLaMA-2 MLP (the workload shape of §4).
# ---------------------------------------------------------------------------

def swiglu_fwd(gate, up):
    """h = SiLU(gate) * up."""
    return silu(gate) * np.asarray(up, np.float64)


def swiglu_bwd(gate, up, dh):
    """dgate = dh * up * SiLU'(gate), dup = dh * SiLU(gate)."""
    gate = np.asarray(gate, np.float64)
    up = np.asarray(up, np.float64)
    dh = np.asarray(dh, np.float64)
    return dh * up * silu_grad(gate), dh * silu(gate)


# ---------------------------------------------------------------------------
# Composed workloads. In bf16 flow every tensor that crosses from one block
# to the next is rounded, because the GPU stores it in bf16.
# ---------------------------------------------------------------------------

def mlp_fwd(x, gamma, A1, B1, A2, B2, *, eps=1e-5, S=1, flow="bf16", act="silu"):
    """LLaMA-style MLP of two bottlenecks: gate/up (normed, k=2) -> SwiGLU -> down (k=1)."""
    R = _round_fn(flow)
    y1, _ = block_fwd(x, gamma, A1, B1, act=act, has_norm=True, eps=eps, S=S, flow=flow)
    gate, up = R(y1[0]), R(y1[1])
    h = R(swiglu_fwd(gate, up))
    y2, _ = block_fwd(h, None, A2, B2, act=act, has_norm=False, eps=eps, S=S, flow=flow)
    return y2[0], {"gate": gate, "up": up, "h": h}


def mlp_bwd(x, gamma, A1, B1, A2, B2, dout, *, eps=1e-5, S=1, flow="bf16", act="silu"):
    R = _round_fn(flow)
    _, c = mlp_fwd(x, gamma, A1, B1, A2, B2, eps=eps, S=S, flow=flow, act=act)
    g2 = block_bwd(c["h"], None, A2, B2, np.asarray(dout)[None], act=act, has_norm=False,
                   eps=eps, S=S, flow=flow)
    dh = R(g2["dx"])
    dgate, dup = swiglu_bwd(c["gate"], c["up"], dh)
    dy1 = np.stack([R(dgate), R(dup)])
    g1 = block_bwd(x, gamma, A1, B1, dy1, act=act, has_norm=True, eps=eps, S=S, flow=flow)
    return {"dx": g1["dx"], "dgamma": g1["dgamma"], "dA1": g1["dA"], "dB1": g1["dB"],
            "dA2": g2["dA"], "dB2": g2["dB"]}


def layer_fwd(x, p, *, eps=1e-5, S=1, flow="bf16", act="silu"):
    """Full CoLA layer without the attention core (attention output := V).

    p holds gamma1, A_qkv [d,3r], B_qkv [3,r,d], A_o [d,r], B_o [1,r,d],
    gamma2, A_gu [d,2r], B_gu [2,r,ffn], A_dn [ffn,r], B_dn [1,r,d].
    x1 = x + O(V), out = x1 + MLP(x1).
    """
    R = _round_fn(flow)
    yq, _ = block_fwd(x, p["gamma1"], p["A_qkv"], p["B_qkv"], act=act, has_norm=True,
                      eps=eps, S=S, flow=flow)
    qkv = R(yq)
    yo, _ = block_fwd(qkv[2], None, p["A_o"], p["B_o"], act=act, has_norm=False,
                      eps=eps, S=S, flow=flow)
    x1 = R(R(x) + R(yo[0]))
    m, mc = mlp_fwd(x1, p["gamma2"], p["A_gu"], p["B_gu"], p["A_dn"], p["B_dn"],
                    eps=eps, S=S, flow=flow, act=act)
    out = x1 + R(m)
    return out, {"qkv": qkv, "x1": x1}


def layer_bwd(x, p, dout, dq, dk, *, eps=1e-5, S=1, flow="bf16", act="silu"):
    """Backward of layer_fwd; dq and dk are the (seeded) upstream gradients of Q and K."""
    R = _round_fn(flow)
    _, c = layer_fwd(x, p, eps=eps, S=S, flow=flow, act=act)
    dout = R(dout)
    gm = mlp_bwd(c["x1"], p["gamma2"], p["A_gu"], p["B_gu"], p["A_dn"], p["B_dn"], dout,
                 eps=eps, S=S, flow=flow, act=act)
    dx1 = R(dout + R(gm["dx"]))
    go = block_bwd(c["qkv"][2], None, p["A_o"], p["B_o"], dx1[None], act=act, has_norm=False,
                   eps=eps, S=S, flow=flow)
    dqkv = np.stack([R(dq), R(dk), R(go["dx"])])
    gq = block_bwd(x, p["gamma1"], p["A_qkv"], p["B_qkv"], dqkv, act=act, has_norm=True,
                   eps=eps, S=S, flow=flow)
    dx = dx1 + R(gq["dx"])
    return {"dx": dx, "dgamma1": gq["dgamma"], "dA_qkv": gq["dA"], "dB_qkv": gq["dB"],
            "dA_o": go["dA"], "dB_o": go["dB"], "dgamma2": gm["dgamma"],
            "dA_gu": gm["dA1"], "dB_gu": gm["dB1"], "dA_dn": gm["dA2"], "dB_dn": gm["dB2"]}


def svd_pair_fwd(x, p, *, eps=1e-5, S=1, flow="bf16"):
    """Two independent normed SVD bottlenecks (no inner nonlinearity) on one x.

    p holds gamma_qkv, A_qkv, B_qkv, gamma_gu, A_gu, B_gu.
    """
    yq, _ = block_fwd(x, p["gamma_qkv"], p["A_qkv"], p["B_qkv"], act="identity",
                      has_norm=True, eps=eps, S=S, flow=flow)
    yg, _ = block_fwd(x, p["gamma_gu"], p["A_gu"], p["B_gu"], act="identity",
                      has_norm=True, eps=eps, S=S, flow=flow)
    return yq, yg


def svd_pair_bwd(x, p, dy_qkv, dy_gu, *, eps=1e-5, S=1, flow="bf16"):
    R = _round_fn(flow)
    gq = block_bwd(x, p["gamma_qkv"], p["A_qkv"], p["B_qkv"], dy_qkv, act="identity",
                   has_norm=True, eps=eps, S=S, flow=flow)
    gg = block_bwd(x, p["gamma_gu"], p["A_gu"], p["B_gu"], dy_gu, act="identity",
                   has_norm=True, eps=eps, S=S, flow=flow)
    return {"dx": R(gq["dx"]) + R(gg["dx"]),
            "dgamma_qkv": gq["dgamma"], "dA_qkv": gq["dA"], "dB_qkv": gq["dB"],
            "dgamma_gu": gg["dgamma"], "dA_gu": gg["dA"], "dB_gu": gg["dB"]}


# ---------------------------------------------------------------------------
# Error measures used by every parity test.
# ---------------------------------------------------------------------------

def rel_errors(got, want):
    """(max_rel, mean_rel) of got against want, both as fp64.

    max_rel = max_i |g_i - o_i| / max(|o_i|, rms(o));
    mean_rel = sum |g - o| / sum |o|.
    """
    g = np.asarray(got, np.float64).ravel()
    o = np.asarray(want, np.float64).ravel()
    if o.size == 0:
        return 0.0, 0.0
    diff = np.abs(g - o)
    rms = np.sqrt(np.mean(o * o))
    denom = np.maximum(np.abs(o), rms)
    denom = np.where(denom == 0.0, 1.0, denom)
    max_rel = float(np.max(diff / denom))
    tot = float(np.sum(np.abs(o)))
    mean_rel = float(np.sum(diff) / tot) if tot > 0 else float(np.sum(diff))
    return max_rel, mean_rel
