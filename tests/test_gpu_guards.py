"""Write checks standing in for a memory checker: every output buffer and the
workspace sit between guard regions filled with a sentinel byte, which forward and
backward (plain, fused SwiGLU, emulated exchange) must leave untouched; and debug
write counting shows every output element of every GEMM written exactly once. Shapes
with ragged row and column tiles, groups that are not a multiple of the tile width,
and co-scheduled row and column splits.
"""

import math

import numpy as np
import pytest
import torch

from rank_bottleneck_online_gb300 import binding as B
from rank_bottleneck_online_gb300 import build as build_mod
from rank_bottleneck_online_gb300 import inputs
from rank_bottleneck_online_gb300.block import Block

from parity import random_block_shapes

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side; keeps the interior 256-byte aligned
SENTINEL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    B.lib()


class Guarded:
    def __init__(self, shape, dtype):
        self.nbytes = math.prod(shape) * torch.tensor([], dtype=dtype).element_size()
        body = (self.nbytes + 255) // 256 * 256
        self.raw = torch.full((2 * GUARD + body,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self):
        return bool((self.raw[:GUARD] == SENTINEL).all()) and \
            bool((self.raw[GUARD + self.nbytes:] == SENTINEL).all())


def guarded_ws(desc):
    g = Guarded((B.workspace_bytes(desc),), torch.uint8)
    ws = B.Workspace.__new__(B.Workspace)
    ws.nbytes, ws.buf = g.nbytes, g.t
    B._check(B.lib().boost_block_ws_init(ws.ptr, ws.nbytes, B._stream()), "ws_init")
    return g, ws


CASES = [
    # name, T, d, r, k, n, S, has_norm
    ("ragged_rows_and_columns", 200, 192, 64, 2, 200, 4, True),
    ("rank_not_tile_multiple", 72, 128, 40, 3, 72, 2, True),
    ("no_norm_tail", 130, 128, 64, 1, 64, 2, False),
    ("co_scheduled_rows", 4352, 512, 512, 2, 1024, 4, True),
    ("co_scheduled_columns", 1024, 256, 512, 2, 8192, 4, True),
    # the down-projection and the dual kernel take the planned row split (15 rows of
    # 512-row super-tiles in the cluster launch instead of the fixed split's 16)
    ("planned_row_split", 9216, 1024, 512, 1, 2048, 4, True),
]
# and the seeded random shapes of the block parity test
CASES += [(c[0], *c[1:7], c[8]) for c in random_block_shapes()]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_no_write_outside_any_output(case):
    _, T, d, r, k, n, S, norm = case
    w = inputs.make_block(T, d, r, k, n, has_norm=norm, seed=31)
    desc = B.make_desc(T, d, r, k, n, S=S, has_norm=norm)
    bf, f32 = torch.bfloat16, torch.float32
    x, dy = w["x"].cuda(), w["dy"].cuda()
    A, Bw = w["A"].cuda(), w["B"].cuda()
    gamma = w["gamma"].cuda() if norm else None
    gws, ws = guarded_ws(desc)
    outs = {"y": Guarded((k, T, n), bf), "dx": Guarded((T, d), bf),
            "dA": Guarded((d, k * r), bf), "dB": Guarded((k, r, n), bf)}
    if norm:
        outs["rstd"] = Guarded((T,), f32)
        outs["dgamma"] = Guarded((d,), bf)
    rstd = outs["rstd"].t if norm else None
    B.block_fwd(desc, x, gamma, A, Bw, ws, y=outs["y"].t, rstd=rstd)
    B.block_bwd(desc, x, gamma, A, Bw, dy, ws, rstd=rstd, dx=outs["dx"].t,
                dgamma=outs["dgamma"].t if norm else None, dA=outs["dA"].t, dB=outs["dB"].t)
    if d % S == 0 and (d // S) % 64 == 0:
        pay = Guarded((B.btp_payload_elems(desc),), f32)
        B.block_fwd_btp(desc, x, gamma, A, Bw, ws, y=outs["y"].t, payload=pay.t)
        outs["payload"] = pay
    if k == 1:
        # the residual forms write the same outputs (plain-store epilogues)
        res_y = torch.randn(T, n, device="cuda").to(bf)
        res_x = torch.randn(T, d, device="cuda").to(bf)
        B.block_fwd(desc, x, gamma, A, Bw, ws, y=outs["y"].t, rstd=rstd, residual=res_y)
        B.block_bwd(desc, x, gamma, A, Bw, dy, ws, rstd=rstd, dx=outs["dx"].t,
                    dgamma=outs["dgamma"].t if norm else None, dA=outs["dA"].t,
                    dB=outs["dB"].t, dx_residual=res_x)
    if k == 2:
        h = Guarded((T, n), bf)
        B.block_fwd_swiglu(desc, x, gamma, A, Bw, ws, y=outs["y"].t, h=h.t, rstd=rstd)
        a = B.ws_view(ws, B.ws_layout(desc)["a"], (T, k * r), bf).clone()
        B.block_up(desc, a, Bw, ws, y=outs["y"].t, h=h.t)
        outs["h"] = h
    torch.cuda.synchronize()
    B.check(ws)
    assert gws.intact(), "workspace guard overwritten"
    for key, g in outs.items():
        assert g.intact(), f"{key} guard overwritten"


def test_no_write_outside_the_fused_swiglu_backward_outputs():
    T, d, r, ffn = 4352, 256, 128, 520          # ragged last column tile, co-scheduled rows
    w = inputs.make_mlp(T, d, r, ffn, seed=32)
    desc = B.make_desc(T, ffn, r, 1, d, S=1, has_norm=False)
    bf = torch.bfloat16
    gws, ws = guarded_ws(desc)
    h = torch.randn(T, ffn, device="cuda").to(bf)
    gate = torch.randn(T, ffn, device="cuda").to(bf)
    up = torch.randn(T, ffn, device="cuda").to(bf)
    dy = w["dout"].cuda().view(1, T, d)
    outs = {"dgate": Guarded((T, ffn), bf), "dup": Guarded((T, ffn), bf),
            "dA": Guarded((ffn, r), bf), "dB": Guarded((1, r, d), bf)}
    B.block_bwd_swiglu(desc, h, w["A2"].cuda(), w["B2"].cuda(), dy, gate, up, ws,
                       dgate=outs["dgate"].t, dup=outs["dup"].t, dA=outs["dA"].t,
                       dB=outs["dB"].t)
    torch.cuda.synchronize()
    B.check(ws)
    assert gws.intact()
    for key, g in outs.items():
        assert g.intact(), f"{key} guard overwritten"


def _check_counts(counts, log):
    c = counts.cpu().numpy()
    covered = 0
    for off, M, N, ld, planes, splits, pstride, sstride in log:
        for sp in range(splits):
            for pl in range(planes):
                base = off + sp * sstride + pl * pstride
                plane = c[base:base + (M - 1) * ld + N]
                full = np.zeros(M * ld, dtype=c.dtype)
                full[:plane.size] = plane
                grid = full.reshape(M, ld)
                assert (grid[:, :N] == 1).all(), (off, M, N, sp, pl, int(grid[:, :N].min()),
                                                   int(grid[:, :N].max()))
                assert (grid[:, N:] == 0).all(), (off, M, N, sp, pl)
                covered += M * N
    assert int(c.sum()) == covered          # nothing written outside the planes


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_every_output_element_is_written_exactly_once(case):
    # debug write counting: each GEMM's epilogues add 1 per element they write, in a
    # plane shaped like that GEMM's output (split-K partial planes included)
    _, T, d, r, k, n, S, norm = case
    w = inputs.make_block(T, d, r, k, n, has_norm=norm, seed=33)
    blk = Block(T, d, r, k, n, S=S, has_norm=norm, weights=w)
    x, dy = w["x"].cuda(), w["dy"].cuda()
    counts = torch.zeros(160 << 20, dtype=torch.int32, device="cuda")
    B.debug_count_writes(counts)
    try:
        blk.forward(x)
        blk.backward(x, dy)
        if k == 2:
            B.block_fwd_swiglu(blk.desc, x, blk.gamma, blk.A, blk.B, blk.ws)
        if d % S == 0 and (d // S) % 64 == 0:
            B.block_fwd_btp(blk.desc, x, blk.gamma, blk.A, blk.B, blk.ws)
        torch.cuda.synchronize()
        log = B.debug_count_log()
    finally:
        B.debug_count_writes(None)
    B.check(blk.ws)
    # down, up, dual, dB, dA, dx per block pass, plus the fused and exchange forwards
    assert len(log) >= 6
    _check_counts(counts, log)
