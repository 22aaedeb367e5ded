"""Pins of the oracle's block, composition and backward.

* the method's steps (sharded statistics, deferred 1/rms, gamma folded into
  the concatenated weight, batched up-projection, recompute) equal the plain
  definition in fp64 (the equivalence claims of Online-RMSNorm and linear-layer
  grouping, BOOST technical summary §2.2);
* the plain definition equals a forward built from torch library routines,
  and its backward equals torch autograd and central finite differences;
* S=1, gamma=1, sigma=id, k=1 reduces to the textbook RMSNorm(x) A B;
* rank(A_i B_i) <= r for a d x r / r x d pair (§2.1) and the SVD-style
  weights have the drawn singular values;
* bf16 flow stays within the bf16 error bound of the exact flow;
* planted mistakes in a copy of the oracle are caught by these pins.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import bottleneck as ob
from rank_bottleneck_online_gb300 import inputs


def _rand_block(seed, T=6, d=16, r=4, k=2, n=8, scale_z=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    g = 1.0 + 0.1 * rng.standard_normal(d)
    A = rng.standard_normal((d, k * r)) * scale_z / np.sqrt(d)
    B = rng.standard_normal((k, r, n)) / np.sqrt(r)
    dy = rng.standard_normal((k, T, n))
    return x, g, A, B, dy


def _torch_block(x, g, A, B, act, has_norm, eps):
    """Forward from torch library routines (used only to get autograd gradients)."""
    k, r, n = B.shape
    h = F.rms_norm(x, (x.shape[1],), g, eps=eps) if has_norm else x
    ys = []
    for i in range(k):
        z = h @ A[:, i * r:(i + 1) * r]
        a = F.silu(z) if act == "silu" else z
        ys.append(a @ B[i])
    return torch.stack(ys)


@pytest.mark.parametrize("act", ["silu", "identity"])
@pytest.mark.parametrize("has_norm", [True, False])
def test_reference_matches_torch_autograd(act, has_norm):
    x, g, A, B, dy = _rand_block(3)
    eps = 1e-5
    tx, tg, tA, tB = (torch.tensor(v, dtype=torch.float64, requires_grad=True)
                      for v in (x, g, A, B))
    ty = _torch_block(tx, tg, tA, tB, act, has_norm, eps)
    (ty * torch.from_numpy(dy)).sum().backward()
    y, _ = oracle.block_fwd_reference(x, g, A, B, act=act, has_norm=has_norm, eps=eps)
    gr = oracle.block_bwd_reference(x, g, A, B, dy, act=act, has_norm=has_norm, eps=eps)
    assert np.allclose(y, ty.detach().numpy(), rtol=1e-12, atol=1e-13)
    assert np.allclose(gr["dx"], tx.grad.numpy(), rtol=1e-11, atol=1e-12)
    assert np.allclose(gr["dA"], tA.grad.numpy(), rtol=1e-11, atol=1e-12)
    assert np.allclose(gr["dB"], tB.grad.numpy(), rtol=1e-11, atol=1e-12)
    if has_norm:
        assert np.allclose(gr["dgamma"], tg.grad.numpy(), rtol=1e-11, atol=1e-12)


def _fd_check(fwd, params, dy, grads, step=1e-6, tol=1e-6):
    """Central differences of L = <fwd(params), dy> against analytic grads."""
    for name, g_an in grads.items():
        p = params[name]
        flat = p.reshape(-1)
        g_fd = np.empty(flat.size)
        for idx in range(flat.size):
            old = flat[idx]
            flat[idx] = old + step
            lp = np.sum(fwd() * dy)
            flat[idx] = old - step
            lm = np.sum(fwd() * dy)
            flat[idx] = old
            g_fd[idx] = (lp - lm) / (2 * step)
        err = np.max(np.abs(g_fd - g_an.reshape(-1))) / max(np.max(np.abs(g_fd)), 1e-30)
        assert err <= tol, (name, err)


@pytest.mark.parametrize("act", ["silu", "identity"])
def test_method_backward_finite_differences(act):
    # tiny shape from the block's own recipe: T=4, d=16, r=4, k=2, n=8, S=4
    x, g, A, B, dy = _rand_block(11, T=4, d=16, r=4, k=2, n=8)
    P = {"x": x, "gamma": g, "A": A, "B": B}

    def fwd():
        return oracle.block_fwd(P["x"], P["gamma"], P["A"], P["B"], act=act, S=4,
                                flow="exact")[0]

    gr = oracle.block_bwd(x, g, A, B, dy, act=act, S=4, flow="exact")
    _fd_check(fwd, P, dy, {"x": gr["dx"], "gamma": gr["dgamma"], "A": gr["dA"],
                           "B": gr["dB"]})


@pytest.mark.parametrize("act", ["silu", "identity"])
@pytest.mark.parametrize("has_norm", [True, False])
@pytest.mark.parametrize("S", [1, 4])
def test_method_steps_equal_plain_definition(act, has_norm, S):
    # Online-RMSNorm (sharded stats + deferred scale + folded gamma) and the
    # grouped/batched projections reproduce the plain block in fp64.
    x, g, A, B, dy = _rand_block(5, T=10, d=32, r=8, k=3, n=12)
    gam = g if has_norm else None
    y_ref, c_ref = oracle.block_fwd_reference(x, gam, A, B, act=act, has_norm=has_norm)
    y, c = oracle.block_fwd(x, gam, A, B, act=act, has_norm=has_norm, S=S, flow="exact")
    assert np.allclose(y, y_ref, rtol=1e-13, atol=1e-14)
    assert np.allclose(c["z"], c_ref["z"], rtol=1e-13, atol=1e-14)      # deferral
    b_ref = oracle.block_bwd_reference(x, gam, A, B, dy, act=act, has_norm=has_norm)
    b = oracle.block_bwd(x, gam, A, B, dy, act=act, has_norm=has_norm, S=S, flow="exact")
    for key in ("dx", "dA", "dB") + (("dgamma",) if has_norm else ()):
        assert np.allclose(b[key], b_ref[key], rtol=1e-12, atol=1e-13), key
    # the recomputed activation is the forward one
    assert np.array_equal(b["a"], c["a"])


def test_rmsnorm_backward_row_dot_identity():
    # sum_j (s*gamma*dh)_j x_j = sum_m dz_m z_m per row: the RMSNorm backward
    # row reduction can be taken in the r-wide space.
    x, g, A, B, dy = _rand_block(8, T=7, d=24, r=6, k=2, n=10)
    b = oracle.block_bwd(x, g, A, B, dy, S=2, flow="exact")
    gs = b["dzs"] @ (g[:, None] * A).T
    assert np.allclose(np.sum(gs * x, axis=1), b["q"], rtol=1e-12, atol=1e-13)


def test_textbook_special_case():
    # S=1, gamma=1, sigma=id, k=1: y = rms_norm(x) @ A @ B (torch library)
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 12))
    A = rng.standard_normal((12, 3))
    B = rng.standard_normal((1, 3, 7))
    y, _ = oracle.block_fwd(x, np.ones(12), A, B, act="identity", S=1, flow="exact")
    h = F.rms_norm(torch.from_numpy(x), (12,), eps=1e-5)
    want = (h @ torch.from_numpy(A) @ torch.from_numpy(B[0])).numpy()
    assert np.allclose(y[0], want, rtol=1e-13, atol=1e-14)


def test_grouping_concatenated_equals_separate():
    x, g, A, B, dy = _rand_block(9, T=8, d=20, r=5, k=3, n=6)
    _, c = oracle.block_fwd(x, g, A, B, S=1, flow="exact")
    _, s = oracle.rmsnorm_stats(x, 1, 1e-5)
    Ap = g[:, None] * A
    for i in range(3):
        zi = s[:, None] * (x @ Ap[:, i * 5:(i + 1) * 5])
        assert np.allclose(c["z"][:, i * 5:(i + 1) * 5], zi, rtol=1e-14, atol=1e-15)


def test_rank_of_factorised_layer():
    # a d x r / r x d pair has rank <= r
    x, g, A, B, dy = _rand_block(4, T=4, d=32, r=4, k=2, n=24)
    for i in range(2):
        W = A[:, i * 4:(i + 1) * 4] @ B[i]
        sv = np.linalg.svd(W, compute_uv=False)
        assert sv[4] / sv[0] < 1e-12


def test_svd_weights_have_drawn_singular_values():
    # A_i = U_i diag(s_i), B_i = V_i^T  =>  singular values of A_i B_i are s_i
    # (up to the bf16 cast of the stored weights).
    w = inputs.make_svd_pair(T=4, d=64, r=8, ffn=48, seed=0)
    A = inputs.as_f64(w["p"]["A_qkv"])
    B = inputs.as_f64(w["p"]["B_qkv"])
    for i in range(3):
        sv = np.linalg.svd(A[:, i * 8:(i + 1) * 8] @ B[i], compute_uv=False)[:8]
        want = np.sort(w["svals_qkv"][i].double().numpy())[::-1]
        assert np.allclose(sv, want, rtol=0, atol=2e-2 * want[0])


@pytest.mark.parametrize("act", ["silu", "identity"])
def test_bf16_flow_within_bf16_error_of_exact(act):
    w = inputs.make_block(T=64, d=128, r=32, k=3, n=96, seed=1)
    x, g, A, B, dy = (inputs.as_f64(w[k]) for k in ("x", "gamma", "A", "B", "dy"))
    y_e, _ = oracle.block_fwd(x, g, A, B, act=act, S=4, flow="exact")
    y_b, c_b = oracle.block_fwd(x, g, A, B, act=act, S=4, flow="bf16")
    mx, mean = oracle.rel_errors(y_b, y_e)
    assert mean < 6e-3 and mx < 6e-2
    assert np.array_equal(oracle.to_bf16(c_b["a"]), c_b["a"])       # stored in bf16
    assert np.array_equal(oracle.to_bf16(c_b["Ap"]), c_b["Ap"])
    b_e = oracle.block_bwd(x, g, A, B, dy, act=act, S=4, flow="exact")
    b_b = oracle.block_bwd(x, g, A, B, dy, act=act, S=4, flow="bf16")
    for key in ("dx", "dgamma", "dA", "dB"):
        mx, mean = oracle.rel_errors(b_b[key], b_e[key])
        assert mean < 8e-3 and mx < 8e-2, key
    assert np.array_equal(oracle.to_bf16(b_b["dzs"]), b_b["dzs"])


def test_bf16_flow_is_deterministic_and_bf16_inputs_unchanged():
    w = inputs.make_block(T=16, d=32, r=8, k=2, n=16, seed=3)
    x = inputs.as_f64(w["x"])
    assert np.array_equal(oracle.to_bf16(x), x)       # R1 is a no-op on bf16 inputs
    a = oracle.block_fwd(x, inputs.as_f64(w["gamma"]), inputs.as_f64(w["A"]),
                         inputs.as_f64(w["B"]), S=4)[0]
    b = oracle.block_fwd(x, inputs.as_f64(w["gamma"]), inputs.as_f64(w["A"]),
                         inputs.as_f64(w["B"]), S=4)[0]
    assert np.array_equal(a, b)


# ------------------------------------------------------------ compositions

def test_swiglu_matches_torch_autograd():
    rng = np.random.default_rng(0)
    gt = torch.tensor(rng.standard_normal((5, 9)) * 3, requires_grad=True)
    ut = torch.tensor(rng.standard_normal((5, 9)), requires_grad=True)
    dh = rng.standard_normal((5, 9))
    h = F.silu(gt) * ut
    (h * torch.from_numpy(dh)).sum().backward()
    assert np.allclose(oracle.swiglu_fwd(gt.detach().numpy(), ut.detach().numpy()),
                       h.detach().numpy(), rtol=1e-14, atol=1e-15)
    dg, du = oracle.swiglu_bwd(gt.detach().numpy(), ut.detach().numpy(), dh)
    assert np.allclose(dg, gt.grad.numpy(), rtol=1e-13, atol=1e-14)
    assert np.allclose(du, ut.grad.numpy(), rtol=1e-13, atol=1e-14)


def _mlp_torch(x, g, A1, B1, A2, B2, eps=1e-5):
    y1 = _torch_block(x, g, A1, B1, "silu", True, eps)
    h = F.silu(y1[0]) * y1[1]
    return _torch_block(h, None, A2, B2, "silu", False, eps)[0]


def test_mlp_matches_torch_autograd():
    w = inputs.make_mlp(T=6, d=16, r=4, ffn=24, seed=2)
    names = ("x", "gamma", "A1", "B1", "A2", "B2")
    vals = {k: inputs.as_f64(w[k]) for k in names}
    dout = inputs.as_f64(w["dout"])
    tv = {k: torch.tensor(v, requires_grad=True) for k, v in vals.items()}
    out = _mlp_torch(*(tv[k] for k in names))
    (out * torch.from_numpy(dout)).sum().backward()
    o, _ = oracle.mlp_fwd(*(vals[k] for k in names), S=4, flow="exact")
    assert np.allclose(o, out.detach().numpy(), rtol=1e-12, atol=1e-13)
    g = oracle.mlp_bwd(*(vals[k] for k in names), dout, S=4, flow="exact")
    pairs = {"dx": "x", "dgamma": "gamma", "dA1": "A1", "dB1": "B1", "dA2": "A2", "dB2": "B2"}
    for gk, pk in pairs.items():
        assert np.allclose(g[gk], tv[pk].grad.numpy(), rtol=1e-10, atol=1e-12), gk


def test_layer_matches_torch_autograd():
    w = inputs.make_layer(T=5, d=16, r=4, ffn=24, seed=4)
    p = {k: inputs.as_f64(v) for k, v in w["p"].items()}
    x = inputs.as_f64(w["x"])
    dout, dq, dk = (inputs.as_f64(w[k]) for k in ("dout", "dq", "dk"))
    tp = {k: torch.tensor(v, requires_grad=True) for k, v in p.items()}
    tx = torch.tensor(x, requires_grad=True)
    qkv = _torch_block(tx, tp["gamma1"], tp["A_qkv"], tp["B_qkv"], "silu", True, 1e-5)
    o = _torch_block(qkv[2], None, tp["A_o"], tp["B_o"], "silu", False, 1e-5)[0]
    x1 = tx + o
    out = x1 + _mlp_torch(x1, tp["gamma2"], tp["A_gu"], tp["B_gu"], tp["A_dn"], tp["B_dn"])
    L = (out * torch.from_numpy(dout)).sum() + (qkv[0] * torch.from_numpy(dq)).sum() \
        + (qkv[1] * torch.from_numpy(dk)).sum()
    L.backward()
    o_or, _ = oracle.layer_fwd(x, p, S=4, flow="exact")
    assert np.allclose(o_or, out.detach().numpy(), rtol=1e-12, atol=1e-12)
    g = oracle.layer_bwd(x, p, dout, dq, dk, S=4, flow="exact")
    assert np.allclose(g["dx"], tx.grad.numpy(), rtol=1e-10, atol=1e-11)
    for gk, pk in (("dgamma1", "gamma1"), ("dA_qkv", "A_qkv"), ("dB_qkv", "B_qkv"),
                   ("dA_o", "A_o"), ("dB_o", "B_o"), ("dgamma2", "gamma2"),
                   ("dA_gu", "A_gu"), ("dB_gu", "B_gu"), ("dA_dn", "A_dn"),
                   ("dB_dn", "B_dn")):
        assert np.allclose(g[gk], tp[pk].grad.numpy(), rtol=1e-10, atol=1e-11), gk


def test_svd_pair_matches_torch_autograd():
    w = inputs.make_svd_pair(T=5, d=16, r=4, ffn=12, seed=5)
    p = {k: inputs.as_f64(v) for k, v in w["p"].items()}
    x = inputs.as_f64(w["x"])
    dq, dg = inputs.as_f64(w["dy_qkv"]), inputs.as_f64(w["dy_gu"])
    tp = {k: torch.tensor(v, requires_grad=True) for k, v in p.items()}
    tx = torch.tensor(x, requires_grad=True)
    yq = _torch_block(tx, tp["gamma_qkv"], tp["A_qkv"], tp["B_qkv"], "identity", True, 1e-5)
    yg = _torch_block(tx, tp["gamma_gu"], tp["A_gu"], tp["B_gu"], "identity", True, 1e-5)
    ((yq * torch.from_numpy(dq)).sum() + (yg * torch.from_numpy(dg)).sum()).backward()
    oq, og = oracle.svd_pair_fwd(x, p, S=4, flow="exact")
    assert np.allclose(oq, yq.detach().numpy(), rtol=1e-12, atol=1e-13)
    assert np.allclose(og, yg.detach().numpy(), rtol=1e-12, atol=1e-13)
    g = oracle.svd_pair_bwd(x, p, dq, dg, S=4, flow="exact")
    assert np.allclose(g["dx"], tx.grad.numpy(), rtol=1e-10, atol=1e-11)
    for gk, pk in (("dgamma_qkv", "gamma_qkv"), ("dA_qkv", "A_qkv"), ("dB_qkv", "B_qkv"),
                   ("dgamma_gu", "gamma_gu"), ("dA_gu", "A_gu"), ("dB_gu", "B_gu")):
        assert np.allclose(g[gk], tp[pk].grad.numpy(), rtol=1e-10, atol=1e-11), gk


# ------------------------------------------------------- planted mistakes

def _pins_pass():
    """Run the decisive pins; True if all hold."""
    try:
        for act in ("silu", "identity"):
            test_reference_matches_torch_autograd(act, True)
            test_method_steps_equal_plain_definition(act, True, 4)
            test_method_backward_finite_differences(act)
        test_rmsnorm_backward_row_dot_identity()
        test_textbook_special_case()
    except AssertionError:
        return False
    return True


def _bad_silu_grad(z):                        # dropped the (1 + z(1-g)) factor
    g = 1.0 / (1.0 + np.exp(-np.asarray(z, np.float64)))
    return g


def _bad_stats(x, S, eps):                    # divides by the shard width, not d
    x = np.asarray(x, np.float64)
    T, d = x.shape
    off = ob.shard_bounds(d, S)
    ssq = np.stack([np.sum(x[:, off[s]:off[s + 1]] ** 2, axis=1) for s in range(S)])
    return ssq, 1.0 / np.sqrt(ssq.sum(0) / (d // S) + eps)


def _bad_identity_grad(z):                    # wrong sign
    return -np.ones_like(np.asarray(z, np.float64))


def test_pins_hold_on_unmodified_oracle():
    assert _pins_pass()


@pytest.mark.parametrize("target,bad", [
    ("silu_grad", _bad_silu_grad),
    ("identity_grad", _bad_identity_grad),
])
def test_planted_activation_mistakes_are_caught(monkeypatch, target, bad):
    monkeypatch.setattr(ob, target, bad)
    acts = dict(ob.act_fns)
    acts["silu"] = (ob.silu, ob.silu_grad)
    acts["identity"] = (ob.identity, ob.identity_grad)
    monkeypatch.setattr(ob, "act_fns", acts)
    assert not _pins_pass()


def test_planted_stats_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(ob, "rmsnorm_stats", _bad_stats)
    assert not _pins_pass()


def test_planted_transpose_in_backward_is_caught(monkeypatch):
    real = ob.block_bwd

    def bad(x, gamma, A, B, dy, **kw):         # dB transposed within each group
        out = real(x, gamma, A, B, dy, **kw)
        out["dB"] = np.ascontiguousarray(out["dB"][:, ::-1, :])
        return out
    monkeypatch.setattr(ob, "block_bwd", bad)
    monkeypatch.setattr(oracle, "block_bwd", bad)
    assert not _pins_pass()


def test_planted_missing_norm_term_is_caught(monkeypatch):
    real = ob.block_bwd

    def bad(x, gamma, A, B, dy, **kw):         # dx without the RMSNorm row term
        out = real(x, gamma, A, B, dy, **kw)
        Ap = np.asarray(gamma)[:, None] * np.asarray(A) if gamma is not None else A
        out["dx"] = out["dzs"] @ np.asarray(Ap).T
        return out
    monkeypatch.setattr(ob, "block_bwd", bad)
    monkeypatch.setattr(oracle, "block_bwd", bad)
    assert not _pins_pass()
