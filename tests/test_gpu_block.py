"""GPU parity of one bottleneck block through the C ABI against the oracle.

Covers the steps of the block: Online-RMSNorm statistics (exact shard
bookkeeping, ssq and rstd), the gamma fold, the grouped down-projection with
deferred 1/rms and the activation, the batched up-projection, the dual-
accumulator recompute/dgrad, both weight gradients (split-K and not) and dx
with the RMSNorm backward, on shapes that span several tiles and ragged tails.
"""

import os

import numpy as np
import pytest
import torch

import oracle
from rank_bottleneck_online_gb300 import binding as B
from rank_bottleneck_online_gb300 import build as build_mod
from rank_bottleneck_online_gb300 import inputs
from rank_bottleneck_online_gb300.block import Block

from parity import assert_close, oracle_block, random_block_shapes, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    B.lib()


# --------------------------------------------------------------- statistics

@pytest.mark.parametrize("T,d,S", [(128, 256, 4), (100, 264, 3), (77, 40, 5), (5, 48, 16),
                                   (16384, 4096, 8), (1, 8, 1)])
def test_rmsnorm_stats_parity(T, d, S):
    g = torch.Generator().manual_seed(T + d)
    x = (torch.randn(T, d, generator=g) * 2).to(torch.bfloat16)
    desc = B.make_desc(T, d, 8, 1, 8, S=S, eps=1e-5)
    ssq, rstd = B.rmsnorm_stats(desc, x.cuda())
    torch.cuda.synchronize()
    o_ssq, o_rstd = oracle.rmsnorm_stats(inputs.as_f64(x), S, 1e-5)
    assert ssq.shape == (S, T)
    np.testing.assert_allclose(to_np(ssq), o_ssq, rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(to_np(rstd), o_rstd, rtol=2e-6, atol=0)


# ---------------------------------------------------------------- edge rows
#
# Rows the statistics and the RMSNorm-backward epilogue must survive: an all-zero row
# (rstd = eps^-1/2), constant rows (closed form (c^2 + eps)^-1/2), rows scaled to
# |x| ~ 1e3 and a row with a single non-zero value, planted among ordinary rows.

EDGE_C = (3.0, -0.5)        # constants, exact in bf16; c^2 * (d / S) is exact in fp32


def _edge_x(T, d, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g)
    x[0] = 0.0
    x[1] = EDGE_C[0]
    x[2] = EDGE_C[1]
    x[3:6] *= 1000.0
    x[6] = 0.0
    x[6, d // 2] = 7.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("T,d,S", [(64, 256, 4), (40, 48, 16), (300, 4096, 8)])
def test_rmsnorm_stats_edge_rows(T, d, S):
    x = _edge_x(T, d, seed=T)
    eps = 1e-5
    desc = B.make_desc(T, d, 8, 1, 8, S=S, eps=eps)
    ssq, rstd = B.rmsnorm_stats(desc, x.cuda())
    torch.cuda.synchronize()
    ssq, rstd = to_np(ssq), to_np(rstd)
    # closed forms: exact sums of squares, rstd to fp32 precision
    assert np.all(ssq[:, 0] == 0.0)
    assert rstd[0] == pytest.approx(eps ** -0.5, rel=1e-6)
    for row, c in ((1, EDGE_C[0]), (2, EDGE_C[1])):
        assert np.all(ssq[:, row] == c * c * (d // S))
        assert rstd[row] == pytest.approx((c * c + eps) ** -0.5, rel=1e-6)
    assert ssq[:, 6].sum() == 49.0 and rstd[6] == pytest.approx((49.0 / d + eps) ** -0.5,
                                                                 rel=1e-6)
    # and everything against the oracle
    o_ssq, o_rstd = oracle.rmsnorm_stats(inputs.as_f64(x), S, eps)
    np.testing.assert_allclose(ssq, o_ssq, rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(rstd, o_rstd, rtol=2e-6, atol=0)


@pytest.mark.parametrize("T,d,r,k,n,S", [(300, 256, 64, 3, 256, 4), (4352, 512, 512, 2, 1024, 4)])
def test_block_with_edge_rows(T, d, r, k, n, S):
    # the second shape takes the benchmarked launch shapes (2 x 2 clusters, co-scheduled
    # rows): the planted rows sit in the cluster launch's first tile
    w = inputs.make_block(T, d, r, k, n, seed=21)
    w["x"] = _edge_x(T, d, seed=22)
    blk = Block(T, d, r, k, n, S=S, weights=w)
    x, dy = w["x"].cuda(), w["dy"].cuda()
    blk.forward(x)
    blk.backward(x, dy)
    B.check(blk.ws)
    y, c, gr = oracle_block(w, act="silu", has_norm=True, S=S)
    assert torch.count_nonzero(blk.y[:, 0]) == 0          # silu(0) = 0 through B: zero
    np.testing.assert_allclose(to_np(blk.rstd), c["s"], rtol=2e-6)
    assert_close("y", blk.y, y)
    assert_close("dx", blk.dx, gr["dx"])
    assert_close("dA", blk.dA, gr["dA"])
    assert_close("dB", blk.dB, gr["dB"])
    assert_close("dgamma", blk.dgamma, gr["dgamma"])
    # the edge rows on their own (a row's dx is that row's business alone)
    rows = slice(0, 7)
    assert_close("y edge rows", blk.y[:, rows], y[:, rows])
    assert_close("dx edge rows", blk.dx[rows], gr["dx"][rows])


# ------------------------------------------------------------------- blocks

CASES = [
    # name, T, d, r, k, n, S, act, has_norm
    ("tiny_block", 128, 256, 64, 3, 256, 4, "silu", True),
    ("ragged_T_n", 200, 192, 64, 2, 200, 4, "silu", True),
    ("rank_not_tile_multiple", 72, 128, 40, 3, 72, 2, "silu", True),
    ("no_norm", 130, 96, 64, 1, 64, 1, "silu", False),
    ("identity_act", 256, 320, 128, 3, 384, 8, "identity", True),
    ("many_tiles", 1000, 512, 128, 2, 1000, 4, "silu", True),
    ("single_row", 1, 64, 64, 1, 64, 2, "silu", True),
    # >= 8 row super-tiles of 2 x 2 clusters: the row GEMMs split their last rows
    # into a concurrent CTA-pair launch; T is not a multiple of either launch's tile
    ("co_scheduled_rows", 4352, 512, 512, 2, 1024, 4, "silu", True),
    # dB's 16 column super-tiles split between the cluster launch and a pair launch
    ("co_scheduled_cols", 1024, 256, 512, 2, 8192, 4, "silu", True),
    # the down-projection and the dual kernel take the planned row split
    ("planned_row_split", 9216, 1024, 512, 1, 2048, 4, "silu", True),
]


def _run_block(name, T, d, r, k, n, S, act, has_norm, seed=0):
    w = inputs.make_block(T, d, r, k, n, has_norm=has_norm, seed=seed)
    blk = Block(T, d, r, k, n, S=S, act=act, has_norm=has_norm, weights=w)
    x = w["x"].cuda()
    dy = w["dy"].cuda()
    blk.forward(x)
    lay = B.ws_layout(blk.desc)
    a_fwd = B.ws_view(blk.ws, lay["a"], (T, k * r), torch.bfloat16).clone()
    blk.backward(x, dy)
    a_bwd = B.ws_view(blk.ws, lay["a"], (T, k * r), torch.bfloat16).clone()
    B.check(blk.ws)
    return w, blk, a_fwd, a_bwd


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_block_forward_backward_parity(case):
    name, T, d, r, k, n, S, act, has_norm = case
    w, blk, a_fwd, a_bwd = _run_block(*case)
    y, c, gr = oracle_block(w, act=act, has_norm=has_norm, S=S)
    assert_close("y", blk.y, y)
    assert_close("a", a_fwd, c["a"])
    if has_norm:
        np.testing.assert_allclose(to_np(blk.rstd), c["s"], rtol=2e-6)
    assert_close("dx", blk.dx, gr["dx"])
    assert_close("dA", blk.dA, gr["dA"])
    assert_close("dB", blk.dB, gr["dB"])
    if has_norm:
        assert_close("dgamma", blk.dgamma, gr["dgamma"])


@pytest.mark.parametrize("case", CASES[:4], ids=[c[0] for c in CASES[:4]])
def test_recompute_is_bitwise_equal_to_forward(case):
    # the backward regenerates a from x inside the block; it must be the forward's a
    _, _, a_fwd, a_bwd = _run_block(*case)
    assert torch.equal(a_fwd, a_bwd)


@pytest.mark.skipif(os.environ.get("BOOST_COSCHED", "") == "0",
                    reason="co-scheduling turned off in the environment")
def test_co_scheduled_gemms_count_two_kernels():
    # T = 8448 rows (16.5 rows of 512-row super-tiles) take the split launch shape for
    # every GEMM over the token rows, whether the split is planned from the launches' wave
    # counts or fixed per 1000 rows; the profiler counts one timed operation and two
    # kernels for each of them
    T, d, r, k, n, S = 8448, 512, 512, 2, 1024, 4
    w = inputs.make_block(T, d, r, k, n, seed=6)
    blk = Block(T, d, r, k, n, S=S, weights=w)
    x, dy = w["x"].cuda(), w["dy"].cuda()
    B.profile_enable(True)
    try:
        blk.forward(x)
        blk.backward(x, dy)
        torch.cuda.synchronize()
        ops = B.profile_read()
        kernels = B.profile_kernels()
    finally:
        B.profile_enable(False)
    for name in ("gemm_down_act", "gemm_up", "gemm_dual", "gemm_dx"):
        assert ops[name][0] == 1, name
        assert kernels[name] == 2, name
    # (the statistics and the gamma fold run as one launch on the caller's stream)
    stats = "rmsnorm_stats_fold" if "rmsnorm_stats_fold" in ops else "rmsnorm_stats"
    for name in ("gemm_wgrad_A", "gemm_wgrad_B", stats):
        assert kernels[name] == ops[name][0], name


def test_profiling_one_kernel_alone():
    # boost_profile_only restricts the timed operations to one kernel; the others run
    # untimed, and every operation is timed again once the restriction is lifted
    T, d, r, k, n, S = 512, 256, 128, 2, 512, 4
    w = inputs.make_block(T, d, r, k, n, seed=14)
    blk = Block(T, d, r, k, n, S=S, weights=w)
    x, dy = w["x"].cuda(), w["dy"].cuda()
    try:
        B.profile_only("gemm_dual")
        B.profile_enable(True)
        blk.forward(x)
        blk.backward(x, dy)
        torch.cuda.synchronize()
        ops = B.profile_read()
        assert set(ops) == {"gemm_dual"} and ops["gemm_dual"][0] == 1
        B.profile_only(None)
        B.profile_enable(True)
        blk.forward(x)
        blk.backward(x, dy)
        torch.cuda.synchronize()
        ops = B.profile_read()
        assert {"gemm_dual", "gemm_down_act", "gemm_up", "gemm_dx"} <= set(ops)
    finally:
        B.profile_only(None)
        B.profile_enable(False)
    with pytest.raises(KeyError):
        B.profile_only("no_such_kernel")


@pytest.mark.skipif(os.environ.get("BOOST_COSCHED_COLS", "") == "0",
                    reason="column co-scheduling turned off in the environment")
def test_weight_gradient_columns_are_co_scheduled():
    # dB = a^T dy has M = r = 512 rows (one super-tile row) and 16 column super-tiles:
    # its last columns run as a CTA-pair launch beside the cluster launch
    T, d, r, k, n, S = 1024, 256, 512, 2, 8192, 4
    w = inputs.make_block(T, d, r, k, n, seed=9)
    blk = Block(T, d, r, k, n, S=S, weights=w)
    x, dy = w["x"].cuda(), w["dy"].cuda()
    B.profile_enable(True)
    try:
        blk.forward(x)
        blk.backward(x, dy)
        torch.cuda.synchronize()
        ops = B.profile_read()
        kernels = B.profile_kernels()
    finally:
        B.profile_enable(False)
    assert ops["gemm_wgrad_B"][0] == 1 and kernels["gemm_wgrad_B"] == 2


def test_backward_with_and_without_saved_rstd_agree():
    T, d, r, k, n, S = 256, 256, 64, 3, 256, 4
    w = inputs.make_block(T, d, r, k, n, seed=3)
    blk = Block(T, d, r, k, n, S=S, weights=w)
    x, dy = w["x"].cuda(), w["dy"].cuda()
    blk.forward(x)
    g1 = [t.clone() for t in blk.backward(x, dy, reuse_rstd=True)]
    g2 = [t.clone() for t in blk.backward(x, dy, reuse_rstd=False)]
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_results_are_deterministic():
    T, d, r, k, n, S = 300, 256, 64, 2, 136, 4
    w = inputs.make_block(T, d, r, k, n, seed=4)
    blk = Block(T, d, r, k, n, S=S, weights=w)
    x, dy = w["x"].cuda(), w["dy"].cuda()
    outs = []
    for _ in range(2):
        y = blk.forward(x).clone()
        g = [t.clone() for t in blk.backward(x, dy)]
        outs.append([y] + g)
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_empty_token_batch():
    T, d, r, k, n = 0, 64, 64, 2, 64
    w = inputs.make_block(1, d, r, k, n, seed=5)
    desc = B.make_desc(T, d, r, k, n, S=2)
    ws = B.Workspace(B.workspace_bytes(desc))
    x = torch.empty(0, d, dtype=torch.bfloat16, device="cuda")
    dy = torch.empty(k, 0, n, dtype=torch.bfloat16, device="cuda")
    gam, A, Bw = (w[key].cuda() for key in ("gamma", "A", "B"))
    y = B.block_fwd(desc, x, gam, A, Bw, ws)
    assert y.shape == (k, 0, n)
    dA = torch.full((d, k * r), 7.0, dtype=torch.bfloat16, device="cuda")
    dx, dg, dA, dB = B.block_bwd(desc, x, gam, A, Bw, dy, ws, dA=dA)
    B.check(ws)
    assert dx.shape == (0, d)
    assert torch.count_nonzero(dA) == 0 and torch.count_nonzero(dB) == 0
    assert torch.count_nonzero(dg) == 0


# --------------------------------------------------------------- elementwise

def test_swiglu_and_add_parity():
    g = torch.Generator().manual_seed(9)
    gate = (torch.randn(333, 136, generator=g) * 3).to(torch.bfloat16)
    up = torch.randn(333, 136, generator=g).to(torch.bfloat16)
    dh = torch.randn(333, 136, generator=g).to(torch.bfloat16)
    h = B.swiglu_fwd(gate.cuda(), up.cuda())
    dgate, dup = B.swiglu_bwd(gate.cuda(), up.cuda(), dh.cuda())
    s = B.add(gate.cuda(), up.cuda())
    G, U, D = (inputs.as_f64(t) for t in (gate, up, dh))
    assert_close("h", h, oracle.swiglu_fwd(G, U), 1e-2, 5e-3)
    og, ou = oracle.swiglu_bwd(G, U, D)
    assert_close("dgate", dgate, og, 1e-2, 5e-3)
    assert_close("dup", dup, ou, 1e-2, 5e-3)
    assert_close("add", s, G + U, 1e-2, 5e-3)


# ------------------------------------------------------- failure detection

def test_bounded_wait_reports_timeout_and_context_survives():
    ws = B.Workspace(1024)
    B.debug_wait_timeout(ws, 2000)           # 2 ms limit on a barrier nobody arrives on
    with pytest.raises(B.BoostError) as ei:
        B.check(ws)
    assert ei.value.status == 6
    B.check(ws)                              # error word was cleared
    # the context still runs real work afterwards
    _, blk, _, _ = _run_block("after_timeout", 128, 128, 64, 1, 64, 2, "silu", True)
    assert torch.isfinite(blk.y.float()).all()


def test_forward_backward_replay_from_a_cuda_graph():
    # the calls are stream-ordered, so one step captures into a CUDA graph (the
    # co-scheduled GEMMs' fork to and join from the side stream included) and replays
    # to the eager results bit for bit
    T, d, r, k, n, S = 4352, 512, 512, 2, 1024, 4
    w = inputs.make_block(T, d, r, k, n, seed=13)
    blk = Block(T, d, r, k, n, S=S, weights=w)
    x, dy = w["x"].cuda(), w["dy"].cuda()

    def step():
        blk.forward(x)
        blk.backward(x, dy)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (blk.y, blk.dx, blk.dA, blk.dB, blk.dgamma)]
    for t in (blk.y, blk.dx, blk.dA, blk.dB, blk.dgamma):
        t.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # warm-up on the capture stream
        step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (blk.y, blk.dx, blk.dA, blk.dB, blk.dgamma):
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    B.check(blk.ws)
    for a, b in zip(eager, (blk.y, blk.dx, blk.dA, blk.dB, blk.dgamma)):
        assert torch.equal(a, b)


def test_two_host_threads_on_their_own_streams_match_serial_runs():
    # calls on different workspaces may run concurrently: the library's shared fork
    # and co-scheduling streams are used one fork/join sequence at a time
    import threading

    shape = (4352, 512, 512, 2, 1024, 4)          # co-scheduled rows
    blocks, data = [], []
    for seed in (41, 42):
        T, d, r, k, n, S = shape
        w = inputs.make_block(T, d, r, k, n, seed=seed)
        blocks.append(Block(T, d, r, k, n, S=S, weights=w))
        data.append((w["x"].cuda(), w["dy"].cuda()))

    def outputs(blk):
        return [t.clone() for t in (blk.y, blk.dx, blk.dA, blk.dB, blk.dgamma)]

    serial = []
    for blk, (x, dy) in zip(blocks, data):
        blk.forward(x)
        blk.backward(x, dy)
        torch.cuda.synchronize()
        serial.append(outputs(blk))
        for t in (blk.y, blk.dx, blk.dA, blk.dB, blk.dgamma):
            t.fill_(float("nan"))
    torch.cuda.synchronize()
    errors = []

    def run(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(3):
                    blocks[i].forward(data[i][0])
                    blocks[i].backward(*data[i])
            s.synchronize()
        except Exception as ex:  # noqa: BLE001
            errors.append(ex)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for blk, want in zip(blocks, serial):
        B.check(blk.ws)
        for a, b in zip(outputs(blk), want):
            assert torch.equal(a, b)


# ------------------------------------------------------- seeded random shapes
# (drawn once from a fixed seed within the shape rules: see parity.random_block_shapes)

RANDOM_CASES = random_block_shapes()


@pytest.mark.parametrize("case", RANDOM_CASES, ids=[c[0] for c in RANDOM_CASES])
def test_seeded_random_shapes_parity(case):
    name, T, d, r, k, n, S, act, has_norm = case
    w, blk, a_fwd, a_bwd = _run_block(*case, seed=T)
    y, c, gr = oracle_block(w, act=act, has_norm=has_norm, S=S)
    assert_close("y", blk.y, y)
    assert_close("a", a_fwd, c["a"])
    assert torch.equal(a_fwd, a_bwd)
    if has_norm:
        np.testing.assert_allclose(to_np(blk.rstd), c["s"], rtol=2e-6)
        assert_close("dgamma", blk.dgamma, gr["dgamma"])
    assert_close("dx", blk.dx, gr["dx"])
    assert_close("dA", blk.dA, gr["dA"])
    assert_close("dB", blk.dB, gr["dB"])


def test_forked_backward_streams_give_the_same_results():
    # BOOST_FORK_STREAMS=1 (read once per process) runs dB and dA on forked streams beside
    # dx, and the fold beside the statistics: a child process with it set gives the
    # default one-stream results bit for bit (same kernels, same split plans)
    import hashlib
    import subprocess
    import sys

    shape = (4352, 512, 512, 2, 1024, 4)          # co-scheduled rows, split-K wgrads
    code = (
        "import hashlib, sys, torch\n"
        "sys.path.insert(0, '.')\n"
        "from rank_bottleneck_online_gb300 import inputs, binding as B\n"
        "from rank_bottleneck_online_gb300.block import Block\n"
        f"T, d, r, k, n, S = {shape}\n"
        "w = inputs.make_block(T, d, r, k, n, seed=43)\n"
        "blk = Block(T, d, r, k, n, S=S, weights=w)\n"
        "x, dy = w['x'].cuda(), w['dy'].cuda()\n"
        "blk.forward(x); blk.backward(x, dy); B.check(blk.ws)\n"
        "h = hashlib.sha256()\n"
        "for t in (blk.y, blk.dx, blk.dA, blk.dB, blk.dgamma):\n"
        "    h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())\n"
        "print(h.hexdigest())\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, BOOST_FORK_STREAMS="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    forked = r.stdout.strip().splitlines()[-1]
    T, d, r_, k, n, S = shape
    w = inputs.make_block(T, d, r_, k, n, seed=43)
    blk = Block(T, d, r_, k, n, S=S, weights=w)
    x, dy = w["x"].cuda(), w["dy"].cuda()
    blk.forward(x)
    blk.backward(x, dy)
    B.check(blk.ws)
    h = hashlib.sha256()
    for t in (blk.y, blk.dx, blk.dA, blk.dB, blk.dgamma):
        h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
    assert h.hexdigest() == forked


_HASH_CHILD = (
    "import hashlib, sys, torch\n"
    "sys.path.insert(0, '.')\n"
    "from rank_bottleneck_online_gb300 import inputs, binding as B\n"
    "from rank_bottleneck_online_gb300.block import Block, MLP\n"
    "blk_shape, mlp_shape, graph = {blk!r}, {mlp!r}, {graph!r}\n"
    "T, d, r, k, n, S = blk_shape\n"
    "w = inputs.make_block(T, d, r, k, n, seed=43)\n"
    "blk = Block(T, d, r, k, n, S=S, weights=w)\n"
    "x, dy = w['x'].cuda(), w['dy'].cuda()\n"
    "T2, d2, r2, ffn2, S2 = mlp_shape\n"
    "wm = inputs.make_mlp(T2, d2, r2, ffn2, seed=44)\n"
    "m = MLP(T2, d2, r2, ffn2, S=S2, weights=wm)\n"
    "xm, dout = wm['x'].cuda(), wm['dout'].cuda()\n"
    "def step():\n"
    "    blk.forward(x); blk.backward(x, dy)\n"
    "    m.forward(xm); m.backward(xm, dout)\n"
    "step(); torch.cuda.synchronize()\n"
    "outs = [blk.y, blk.dx, blk.dA, blk.dB, blk.dgamma, m.out, m.dy1,\n"
    "        *m.grads().values()]\n"
    "if graph:\n"
    "    g = torch.cuda.CUDAGraph()\n"
    "    with torch.cuda.graph(g):\n"
    "        step()\n"
    "    for t in outs:\n"
    "        t.zero_()\n"
    "    g.replay(); torch.cuda.synchronize()\n"
    "B.check(blk.ws); B.check(m.gu.ws); B.check(m.dn.ws)\n"
    "h = hashlib.sha256()\n"
    "for t in outs:\n"
    "    h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())\n"
    "print(h.hexdigest())\n")


def _child_hash(env_over, graph):
    import subprocess
    import sys

    code = _HASH_CHILD.format(blk=(4352, 512, 512, 2, 1024, 4),   # co-scheduled, split-K
                              mlp=(2304, 512, 256, 1536, 4), graph=graph)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root,
                       env=dict(os.environ, **env_over), capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout.strip().splitlines()[-1]


def test_programmatic_launches_give_the_same_results():
    # every kernel is a programmatic dependent launch unless BOOST_PDL=0 (read once per
    # process). A CUDA graph of the block and MLP steps replayed with them (outputs zeroed
    # first) gives plain eager launches' results bit for bit.
    plain = _child_hash({"BOOST_PDL": "0"}, graph=False)
    assert _child_hash({"BOOST_PDL": "1"}, graph=True) == plain
    assert _child_hash({"BOOST_PDL": "1"}, graph=False) == plain
