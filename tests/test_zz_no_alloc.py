"""The allocation-free row-scale entry point, for callers that cannot call
cudaMalloc (code under a host framework whose allocator owns the device memory,
plugins handed only their input and output buffers).

It keeps the per-shard partials in one fixed array inside the library, shared
by every call, so calls in a row with different shapes must each give the row
scales the regular statistics entry point gives, and the oracle's: a later call
may not read anything an earlier one left behind. This file is collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from rank_bottleneck_online_gb300 import binding as B
from rank_bottleneck_online_gb300 import build as build_mod
from rank_bottleneck_online_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    B.lib()


def test_noalloc_rstd_matches_regular_entry_point_and_oracle_on_calls_in_a_row():
    g = torch.Generator().manual_seed(11)
    # Each call is smaller and differently sharded than the one before, so stale
    # partials from earlier calls sit in the shared array. The last shape has a shard
    # width of 3 columns (d % 8 == 0 but (d / S) % 8 != 0): the scalar path of the
    # partials kernel.
    for T, d, S in [(4096, 4096, 8), (333, 264, 3), (257, 48, 16)]:
        x = (torch.randn(T, d, generator=g) * 1.5).to(torch.bfloat16)
        xd = x.cuda()
        desc = B.make_desc(T, d, 8, 1, 8, S=S, eps=1e-5)
        _, want = B.rmsnorm_stats(desc, xd)
        got = B.rmsnorm_rstd_noalloc(desc, xd)
        torch.cuda.synchronize()
        # the regular entry point adds the same squares in another per-thread order:
        # equal up to fp32 rounding
        torch.testing.assert_close(got, want, rtol=2e-6, atol=0)
        # the oracle (fp64): fp32 accumulation of d squares, then the square root
        _, s_ref = oracle.rmsnorm_stats(inputs.as_f64(x), S, 1e-5)
        np.testing.assert_allclose(got.double().cpu().numpy(), s_ref, rtol=1e-5, atol=0)


def test_noalloc_rejects_sizes_beyond_the_fixed_array():
    L = B.lib()
    desc = B.make_desc(262144, 64, 8, 1, 8, S=8)       # S*T = 2^21 > 2^20 partials
    st = L.boost_rmsnorm_rstd_noalloc(ctypes.byref(desc), ctypes.c_void_p(0x10000),
                                      ctypes.c_void_p(0x20000), None)
    assert st == 2                                      # BOOST_ERR_UNSUPPORTED_SHAPE
    no_norm = B.make_desc(16, 64, 8, 1, 8, S=1, has_norm=False)
    st = L.boost_rmsnorm_rstd_noalloc(ctypes.byref(no_norm), ctypes.c_void_p(0x10000),
                                      ctypes.c_void_p(0x20000), None)
    assert st == 1
