"""GPU parity of the emulated bottleneck-aware TP exchange ("BOOST" technical summary
§2.1-§2.2) through boost_block_fwd_btp: each shard's partial product and sums of
squares (the payload S ranks would exchange) against the oracle's, element by
element; the block output after the reduction against the oracle block forward; the
row scale bitwise equal to the fused path's.
"""

import numpy as np
import pytest
import torch

import oracle
from rank_bottleneck_online_gb300 import binding as B
from rank_bottleneck_online_gb300 import build as build_mod
from rank_bottleneck_online_gb300 import inputs
from rank_bottleneck_online_gb300.block import Block

from parity import assert_close, oracle_block, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    B.lib()


CASES = [
    # name, T, d, r, k, n, S, has_norm
    ("tiny", 128, 256, 64, 3, 256, 4, True),
    ("ragged_T_three_shards", 200, 192, 64, 2, 200, 3, True),
    ("rank_not_tile_multiple", 72, 128, 40, 3, 72, 2, True),
    ("no_norm", 130, 128, 64, 1, 64, 2, False),
    ("one_shard", 96, 128, 64, 2, 128, 1, True),
    ("co_scheduled_rows", 4352, 512, 512, 2, 1024, 4, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_exchange_payload_and_output_parity(case):
    name, T, d, r, k, n, S, norm = case
    w = inputs.make_block(T, d, r, k, n, has_norm=norm, seed=21)
    blk = Block(T, d, r, k, n, S=S, has_norm=norm, weights=w)
    x = w["x"].cuda()
    y_fused = blk.forward(x).clone()
    rstd_fused = blk.rstd.clone() if norm else None
    rstd = torch.full((T,), float("nan"), device="cuda") if norm else None
    y, zpart, ssq = B.block_fwd_btp(blk.desc, x, blk.gamma, blk.A, blk.B, blk.ws, rstd=rstd)
    B.check(blk.ws)
    f = {key: inputs.as_f64(v) for key, v in w.items() if v is not None}
    o_z, o_ssq = oracle.btp_shard_partials(f["x"], f.get("gamma"), f["A"], S, has_norm=norm)
    # fp32 partial sums over d/S products of bf16 values: tight tolerance per shard
    for s in range(S):
        assert_close(f"zpart[{s}]", zpart[s], o_z[s], 1e-4, 1e-5)
    if norm:
        np.testing.assert_allclose(to_np(ssq), o_ssq, rtol=2e-5, atol=1e-6)
        assert torch.equal(rstd, rstd_fused)         # same sums, same combine order
    # the block output after the reduction: same bar as the fused forward
    o_y = oracle_block(w, act="silu", has_norm=norm, S=S)[0]
    assert_close("y", y, o_y)
    assert_close("y vs fused", y, to_np(y_fused).astype(np.float64), 2e-2, 2e-3)


def test_payload_size_is_exact():
    desc = B.make_desc(128, 256, 64, 3, 256, S=4)
    assert B.btp_payload_elems(desc) == 4 * oracle.exchange_elems(128, 3, 64)
    nonorm = B.make_desc(128, 256, 64, 3, 256, S=4, has_norm=False)
    assert B.btp_payload_elems(nonorm) == 4 * 128 * 3 * 64


@pytest.mark.slow
def test_exchange_at_the_7b_gate_up_block_size_sampled_rows():
    """The benchmarked gate/up block (T=16384, d=4096, r=1024, k=2, n=11008, S=8):
    every shard's partials and sums of squares and the block output on sampled rows
    (rows are independent in the forward) against the oracle on those rows."""
    c = inputs.CONFIGS["llama2_7b_mlp"]
    T, d, r, ffn, S = c["T"], c["d"], c["r"], c["ffn"], c["S"]
    w = inputs.make_block(T, d, r, 2, ffn, seed=23)
    blk = Block(T, d, r, 2, ffn, S=S, weights=w)
    x = w["x"].cuda()
    y, zpart, ssq = B.block_fwd_btp(blk.desc, x, blk.gamma, blk.A, blk.B, blk.ws)
    B.check(blk.ws)
    rows = np.sort(np.random.default_rng(0).choice(T, 96, replace=False))
    rows = np.concatenate([[0], rows, [T - 1]])
    idx = torch.as_tensor(rows, device="cuda")
    zs = zpart.index_select(1, idx).cpu()
    qs = ssq.index_select(1, idx).cpu()
    ys = y.index_select(1, idx).cpu()
    del y, zpart, ssq, blk
    torch.cuda.empty_cache()
    X = inputs.as_f64(w["x"])[rows]
    G, A, Bw = (inputs.as_f64(w[k]) for k in ("gamma", "A", "B"))
    o_z, o_q = oracle.btp_shard_partials(X, G, A, S)
    for s in range(S):
        assert_close(f"zpart[{s}]", zs[s], o_z[s], 1e-4, 1e-5)
    np.testing.assert_allclose(qs.double().numpy(), o_q, rtol=2e-5, atol=1e-6)
    o_y, _ = oracle.block_fwd(X, G, A, Bw, S=S)
    assert_close("y", ys, o_y)
