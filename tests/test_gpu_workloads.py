"""GPU parity of the composed workloads against the oracle: the LLaMA MLP (gate/up
bottleneck -> SwiGLU -> down bottleneck), the full layer without its attention
core, the SVD-style pair, and the full-size LLaMA-2-1B attention-projection
block.
"""

import numpy as np
import pytest
import torch

import oracle
from rank_bottleneck_online_gb300 import binding as B
from rank_bottleneck_online_gb300 import build as build_mod
from rank_bottleneck_online_gb300 import inputs
from rank_bottleneck_online_gb300.block import MLP, Block, Layer, SVDPair

from parity import assert_close, oracle_block

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    B.lib()


def f64(w, keys):
    return [inputs.as_f64(w[k]) for k in keys]


@pytest.mark.parametrize("T,d,r,ffn,S", [(512, 256, 128, 384, 4), (300, 128, 64, 200, 2)])
def test_mlp_parity(T, d, r, ffn, S):
    w = inputs.make_mlp(T, d, r, ffn, seed=1)
    mlp = MLP(T, d, r, ffn, S=S, weights=w)
    x, dout = w["x"].cuda(), w["dout"].cuda()
    out = mlp.forward(x)
    mlp.backward(x, dout)
    B.check(mlp.gu.ws)
    args = f64(w, ("x", "gamma", "A1", "B1", "A2", "B2"))
    o, _ = oracle.mlp_fwd(*args, S=S)
    g = oracle.mlp_bwd(*args, inputs.as_f64(w["dout"]), S=S)
    assert_close("out", out, o)
    for k, v in mlp.grads().items():
        assert_close(k, v, g[k])


@pytest.mark.parametrize("T,d,r,ffn", [(512, 256, 128, 512), (600, 128, 64, 520)])
def test_fused_swiglu_backward_matches_separate_passes(T, d, r, ffn):
    # the down block's dgrad epilogue computing dgate/dup equals dx + a SwiGLU pass
    w = inputs.make_mlp(T, d, r, ffn, seed=6)
    x, dout = w["x"].cuda(), w["dout"].cuda()
    res = []
    for fused in (True, False):
        mlp = MLP(T, d, r, ffn, S=2, weights=w, fused_glu=fused)
        mlp.forward(x)
        mlp.backward(x, dout)
        B.check(mlp.gu.ws)
        res.append((mlp.dy1.clone(), {k: v.clone() for k, v in mlp.grads().items()}))
    (dy_f, g_f), (dy_s, g_s) = res
    assert_close("dgate/dup", dy_f, dy_s.double().cpu().numpy(), 1e-2, 1e-3)
    for k in g_f:
        assert_close(k, g_f[k], g_s[k].double().cpu().numpy(), 1e-2, 1e-3)


def test_layer_parity():
    T, d, r, ffn, S = 256, 256, 64, 384, 4
    w = inputs.make_layer(T, d, r, ffn, seed=2)
    layer = Layer(T, d, r, ffn, S=S, weights=w["p"])
    x = w["x"].cuda()
    out = layer.forward(x)
    layer.backward(x, w["dout"].cuda(), w["dq"].cuda(), w["dk"].cuda())
    B.check(layer.qkv.ws)
    p = {k: inputs.as_f64(v) for k, v in w["p"].items()}
    xo = inputs.as_f64(w["x"])
    o, _ = oracle.layer_fwd(xo, p, S=S)
    g = oracle.layer_bwd(xo, p, *f64(w, ("dout", "dq", "dk")), S=S)
    assert_close("out", out, o)
    assert_close("dx", layer.dx, g["dx"])
    pairs = {"dgamma1": layer.qkv.dgamma, "dA_qkv": layer.qkv.dA, "dB_qkv": layer.qkv.dB,
             "dA_o": layer.o.dA, "dB_o": layer.o.dB, "dgamma2": layer.mlp.gu.dgamma,
             "dA_gu": layer.mlp.gu.dA, "dB_gu": layer.mlp.gu.dB, "dA_dn": layer.mlp.dn.dA,
             "dB_dn": layer.mlp.dn.dB}
    for k, v in pairs.items():
        assert_close(k, v, g[k])


def test_svd_pair_parity():
    T, d, r, ffn, S = 256, 256, 64, 320, 4
    w = inputs.make_svd_pair(T, d, r, ffn, seed=3)
    pair = SVDPair(T, d, r, ffn, S=S, weights=w["p"])
    x = w["x"].cuda()
    yq, yg = pair.forward(x)
    pair.backward(x, w["dy_qkv"].cuda(), w["dy_gu"].cuda())
    B.check(pair.qkv.ws)
    p = {k: inputs.as_f64(v) for k, v in w["p"].items()}
    xo = inputs.as_f64(w["x"])
    oq, og = oracle.svd_pair_fwd(xo, p, S=S)
    g = oracle.svd_pair_bwd(xo, p, *f64(w, ("dy_qkv", "dy_gu")), S=S)
    assert_close("y_qkv", yq, oq)
    assert_close("y_gu", yg, og)
    assert_close("dx", pair.dx, g["dx"])
    for k, v in {"dgamma_qkv": pair.qkv.dgamma, "dA_qkv": pair.qkv.dA, "dB_qkv": pair.qkv.dB,
                 "dgamma_gu": pair.gu.dgamma, "dA_gu": pair.gu.dA, "dB_gu": pair.gu.dB}.items():
        assert_close(k, v, g[k])


@pytest.mark.slow
def test_llama2_1b_attention_block_full_size():
    c = inputs.CONFIGS["llama2_1b_attn_block"]
    T, d, r, k, n, S = c["T"], c["d"], c["r"], c["k"], c["n"], c["S"]
    w = inputs.make_block(T, d, r, k, n, seed=0)
    blk = Block(T, d, r, k, n, S=S, weights=w)
    x, dy = w["x"].cuda(), w["dy"].cuda()
    blk.forward(x)
    blk.backward(x, dy)
    B.check(blk.ws)
    y, _, g = oracle_block(w, act="silu", has_norm=True, S=S)
    assert_close("y", blk.y, y)
    for key, got in (("dx", blk.dx), ("dA", blk.dA), ("dB", blk.dB), ("dgamma", blk.dgamma)):
        assert_close(key, got, g[key])


# ------------------------------------------------ full-size configurations

@pytest.mark.slow
def test_llama2_7b_mlp_full_size():
    """The benchmarked workload at full size, every output against the full oracle."""
    c = inputs.CONFIGS["llama2_7b_mlp"]
    T, d, r, ffn, S = c["T"], c["d"], c["r"], c["ffn"], c["S"]
    w = inputs.make_mlp(T, d, r, ffn, seed=0)
    mlp = MLP(T, d, r, ffn, S=S, weights=w)
    x, dout = w["x"].cuda(), w["dout"].cuda()
    out = mlp.forward(x).clone()
    mlp.backward(x, dout)
    B.check(mlp.gu.ws)
    got = {k: v.cpu() for k, v in mlp.grads().items()}
    out = out.cpu()
    del mlp
    torch.cuda.empty_cache()
    args = f64(w, ("x", "gamma", "A1", "B1", "A2", "B2"))
    o, _ = oracle.mlp_fwd(*args, S=S)
    assert_close("out", out, o)
    del o
    g = oracle.mlp_bwd(*args, inputs.as_f64(w["dout"]), S=S)
    for k, v in got.items():
        assert_close(k, v, g[k])


def _sample_rows(T, n=192, seed=0):
    # spread over every 256-row tile pair, plus the first and last rows
    rng = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([[0, T - 1], rng.choice(T, n, replace=False)]))
    return np.sort(idx)


@pytest.mark.slow
def test_llama2_13b_layer_full_size_sampled_rows():
    """Full-size layer on the GPU; output and dx rows checked against the oracle run
    on those rows alone (every step of the layer is row-wise)."""
    c = inputs.CONFIGS["llama2_13b_layer"]
    T, d, r, ffn, S = c["T"], c["d"], c["r"], c["ffn"], c["S"]
    w = inputs.make_layer(T, d, r, ffn, seed=0)
    layer = Layer(T, d, r, ffn, S=S, weights=w["p"])
    x = w["x"].cuda()
    out = layer.forward(x).clone()
    layer.backward(x, w["dout"].cuda(), w["dq"].cuda(), w["dk"].cuda())
    B.check(layer.qkv.ws)
    idx = _sample_rows(T)
    out_s, dx_s = out.cpu()[idx], layer.dx.cpu()[idx]
    del layer
    torch.cuda.empty_cache()
    p = {k: inputs.as_f64(v) for k, v in w["p"].items()}
    xs = inputs.as_f64(w["x"])[idx]
    o, _ = oracle.layer_fwd(xs, p, S=S)
    assert_close("out rows", out_s, o)
    g = oracle.layer_bwd(xs, p, *(inputs.as_f64(w[k])[idx] for k in ("dout", "dq", "dk")), S=S)
    assert_close("dx rows", dx_s, g["dx"])


@pytest.mark.slow
def test_svd_40b_pair_full_size_sampled_rows():
    c = inputs.CONFIGS["svd_40b_pair"]
    T, d, r, ffn, S = c["T"], c["d"], c["r"], c["ffn"], c["S"]
    w = inputs.make_svd_pair(T, d, r, ffn, seed=0)
    pair = SVDPair(T, d, r, ffn, S=S, weights=w["p"])
    x = w["x"].cuda()
    yq, yg = pair.forward(x)
    yq, yg = yq.clone(), yg.clone()
    pair.backward(x, w["dy_qkv"].cuda(), w["dy_gu"].cuda())
    B.check(pair.qkv.ws)
    idx = _sample_rows(T)
    yq_s, yg_s, dx_s = yq.cpu()[:, idx], yg.cpu()[:, idx], pair.dx.cpu()[idx]
    del pair
    torch.cuda.empty_cache()
    p = {k: inputs.as_f64(v) for k, v in w["p"].items()}
    xs = inputs.as_f64(w["x"])[idx]
    oq, og = oracle.svd_pair_fwd(xs, p, S=S)
    assert_close("y_qkv rows", yq_s, oq)
    assert_close("y_gu rows", yg_s, og)
    g = oracle.svd_pair_bwd(xs, p, inputs.as_f64(w["dy_qkv"])[:, idx],
                            inputs.as_f64(w["dy_gu"])[:, idx], S=S)
    assert_close("dx rows", dx_s, g["dx"])
