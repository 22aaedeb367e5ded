"""The full-rank comparison leg of bench.py (the dense LLaMA MLP in plain torch with
cuBLAS bf16 GEMMs) on the GPU, against the textbook MLP in fp64 on the same bf16
inputs. It is context for the low-rank step, not a library path: this checks that
the timed dense step computes the MLP it is compared as.

Tolerance. The dense leg rounds to bf16 after every torch operation (the RMSNorm
output, both projections, SiLU, their product and the output; in backward every
gradient operation), five or more rounding points on each path against the
low-rank block's three; at about 1.4e-3 mean relative error per bf16 rounding
point that is 3-5e-3 end to end (the same leg run in bf16 on the CPU measures
4.6e-3 mean, 2.5e-2 max against fp64). The bar is 1e-2 mean and 5e-2 max relative
error per tensor; a dropped term or a transposed operand gives errors of order one.
"""

import numpy as np
import pytest
import torch

import bench
import oracle

pytestmark = pytest.mark.gpu

MAX_REL, MEAN_REL = 5e-2, 1e-2


def _textbook(x, g, Wg, Wu, Wd, dout, eps=1e-5):
    """out = (silu(n Wg) * (n Wu)) Wd, n = x / rms(x) * gamma, and every gradient."""
    rs = 1.0 / np.sqrt((x * x).mean(axis=1, keepdims=True) + eps)
    n = x * rs * g
    a, b = n @ Wg, n @ Wu
    sg = 1.0 / (1.0 + np.exp(-a))
    h = a * sg * b
    dh = dout @ Wd.T
    da = dh * b * sg * (1 + a * (1 - sg))
    db = dh * a * sg
    dn = da @ Wg.T + db @ Wu.T
    xh = x * rs
    dxh = dn * g
    dx = rs * (dxh - xh * (dxh * xh).mean(axis=1, keepdims=True))
    return {"out": h @ Wd, "x": dx, "gamma": (dn * xh).sum(axis=0), "Wg": n.T @ da,
            "Wu": n.T @ db, "Wd": h.T @ dout}


@pytest.mark.parametrize("T,d,ffn", [(512, 256, 704), (1000, 512, 1376)])
def test_dense_fullrank_leg_in_bf16_on_the_gpu(T, d, ffn):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    step, t = bench.dense_mlp(T, d, ffn, "cuda", seed=5)
    out = step()
    torch.cuda.synchronize()
    f = {k: t[k].detach().double().cpu().numpy() for k in ("x", "gamma", "Wg", "Wu", "Wd",
                                                           "dout")}
    want = _textbook(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], f["dout"])
    got = {"out": out.detach(), **{k: t[k].grad for k in ("x", "gamma", "Wg", "Wu", "Wd")}}
    for k, w in want.items():
        g = got[k].double().cpu().numpy()
        assert g.shape == w.shape, k
        mx, mean = oracle.rel_errors(g, w)
        assert mx <= MAX_REL and mean <= MEAN_REL, f"{k}: max_rel={mx:.3e} mean_rel={mean:.3e}"
