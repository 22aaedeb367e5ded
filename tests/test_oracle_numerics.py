"""Pins of the oracle's elementary pieces: bf16 rounding, SiLU, Online-RMSNorm
statistics and the exact shard/group/exchange bookkeeping.

Each pin compares against something other than the oracle itself: a
hand-derived table, an independent library routine (torch's fp32->bf16 cast,
torch.nn.functional.silu / rms_norm, autograd) or a closed form.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- bf16 ----

def _golden_bf16():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()[:2]
            want = math.inf if b == "inf" else float.fromhex(b)
            rows.append((float.fromhex(a), want, line))
    return rows


@pytest.mark.parametrize("inp,want,line", _golden_bf16())
def test_bf16_golden_table(inp, want, line):
    got = float(oracle.to_bf16(np.array([inp]))[0])
    assert got == want, line
    if want == 0.0:
        assert math.copysign(1.0, got) == math.copysign(1.0, inp)


def test_bf16_matches_torch_cast_on_fp32_values():
    # torch rounds fp32 -> bf16 to nearest even; for fp32-representable
    # inputs the direct fp64 rounding must give the same value.
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    f32 = bits.view(np.float32)
    f32 = f32[np.isfinite(f32)]
    want = torch.from_numpy(f32.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.to_bf16(f32.astype(np.float64))
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), f32[~same][:5]


def test_bf16_idempotent_and_specials():
    v = np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -2.5, 65504.0])
    r = oracle.to_bf16(v)
    assert np.array_equal(oracle.to_bf16(r), r)
    assert np.isnan(oracle.to_bf16(np.array([np.nan]))[0])
    assert math.copysign(1.0, oracle.to_bf16(np.array([-0.0]))[0]) == -1.0
    assert oracle.to_bf16(np.array([1e300]))[0] == np.inf


# ----------------------------------------------------------------- SiLU ----

def test_silu_closed_forms():
    # logistic(ln 3) = 3/4, so SiLU(ln 3) = 0.75 ln 3 and
    # SiLU'(ln 3) = 0.75 (1 + 0.25 ln 3); SiLU(0) = 0, SiLU'(0) = 1/2.
    l3 = math.log(3.0)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.silu(np.array([l3]))[0] - 0.75 * l3) < 1e-15
    assert abs(oracle.silu_grad(np.array([0.0]))[0] - 0.5) < 1e-15
    assert abs(oracle.silu_grad(np.array([l3]))[0] - 0.75 * (1 + 0.25 * l3)) < 1e-15
    # far tails: SiLU(z) -> z for z >> 0, -> 0 for z << 0
    assert oracle.silu(np.array([800.0]))[0] == 800.0
    assert oracle.silu(np.array([-800.0]))[0] == 0.0


def test_silu_matches_torch_and_autograd():
    z = torch.linspace(-12, 12, 2001, dtype=torch.float64, requires_grad=True)
    f = torch.nn.functional.silu(z)
    (gz,) = torch.autograd.grad(f.sum(), z)
    zn = z.detach().numpy()
    assert np.allclose(oracle.silu(zn), f.detach().numpy(), rtol=1e-14, atol=1e-15)
    assert np.allclose(oracle.silu_grad(zn), gz.numpy(), rtol=1e-13, atol=1e-15)


# ------------------------------------------------------- Online-RMSNorm ----

def test_bookkeeping_exact():
    assert oracle.shard_bounds(4096, 8) == [i * 512 for i in range(9)]
    assert oracle.shard_bounds(256, 4) == [0, 64, 128, 192, 256]
    assert oracle.shard_bounds(7, 1) == [0, 7]
    with pytest.raises(ValueError):
        oracle.shard_bounds(10, 4)
    with pytest.raises(ValueError):
        oracle.shard_bounds(8, 0)
    assert oracle.group_bounds(3, 512) == [0, 512, 1024, 1536]
    # payload of the fused exchange: T*(k*r+1) against T*d for a d-wide reduce
    assert oracle.exchange_elems(16384, 3, 512) == 16384 * 1537
    assert oracle.exchange_elems(1, 1, 1) == 2


def test_stats_worked_example():
    # x = 1..8, S = 4: shard sums of squares 1+4, 9+16, 25+36, 49+64.
    x = np.arange(1.0, 9.0)[None, :]
    ssq, rstd = oracle.rmsnorm_stats(x, 4, 1e-5)
    assert ssq[:, 0].tolist() == [5.0, 25.0, 61.0, 113.0]
    assert rstd[0] == 1.0 / math.sqrt(204.0 / 8.0 + 1e-5)
    # 3-4-5 row, eps = 0: mean square 12.5
    ssq, rstd = oracle.rmsnorm_stats(np.array([[3.0, 4.0]]), 2, 0.0)
    assert ssq[:, 0].tolist() == [9.0, 16.0]
    assert abs(rstd[0] - 1.0 / math.sqrt(12.5)) < 1e-16


def test_stats_constant_row_closed_form():
    # a constant row c*1 has mean square c^2, so rstd = (c^2 + eps)^-1/2
    # and every shard holds c^2 * d / S.
    d, S, eps = 64, 8, 1e-5
    for c in (0.0, 0.5, -3.0, 1e-3):
        x = np.full((1, d), c)
        ssq, rstd = oracle.rmsnorm_stats(x, S, eps)
        assert np.allclose(ssq[:, 0], c * c * d / S, rtol=1e-15, atol=0)
        assert abs(rstd[0] - 1.0 / math.sqrt(c * c + eps)) <= 1e-15 / math.sqrt(c * c + eps)


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16])
def test_sharded_stats_equal_direct(S):
    rng = np.random.default_rng(S)
    x = rng.standard_normal((37, 128))
    ssq, rstd = oracle.rmsnorm_stats(x, S, 1e-5)
    direct = 1.0 / np.sqrt(np.mean(x * x, axis=1) + 1e-5)
    assert np.allclose(rstd, direct, rtol=1e-14, atol=0)
    assert np.allclose(ssq.sum(axis=0), np.sum(x * x, axis=1), rtol=1e-14)
    assert ssq.shape == (S, 37)


def test_rmsnorm_matches_torch_library():
    # torch.nn.functional.rms_norm (fp64) is an independent implementation.
    rng = np.random.default_rng(7)
    x = rng.standard_normal((9, 48))
    g = 1.0 + 0.1 * rng.standard_normal(48)
    _, rstd = oracle.rmsnorm_stats(x, 4, 1e-5)
    want = torch.nn.functional.rms_norm(torch.from_numpy(x), (48,), torch.from_numpy(g),
                                        eps=1e-5).numpy()
    assert np.allclose(g[None, :] * x * rstd[:, None], want, rtol=1e-13, atol=1e-15)


def test_rel_errors_definition():
    o = np.array([1.0, -2.0, 0.0, 4.0])
    g = np.array([1.1, -2.0, 0.1, 4.0])
    mx, mean = oracle.rel_errors(g, o)
    rms = math.sqrt((1 + 4 + 0 + 16) / 4)
    assert abs(mx - 0.1 / rms) < 1e-15          # the 0-entry uses rms(o) as floor
    assert abs(mean - 0.2 / 7.0) < 1e-15
    assert oracle.rel_errors(np.zeros(0), np.zeros(0)) == (0.0, 0.0)
