"""Pins of the oracle's bottleneck-aware TP exchange (S ranks emulated on one host):
the partial products and statistics each rank sends, and the reduction that stands
in for the all-reduce ("BOOST" technical summary §2.1 and §2.2).
"""

import numpy as np
import pytest

import oracle
from rank_bottleneck_online_gb300 import inputs


def _case(T=24, d=64, r=8, k=2, n=16, seed=11):
    w = inputs.make_block(T, d, r, k, n, seed=seed)
    return {key: inputs.as_f64(v) for key, v in w.items() if v is not None}


@pytest.mark.parametrize("S", [1, 2, 4, 8])
def test_partials_sum_to_the_full_product_and_reduce_to_the_block_forward(S):
    w = _case()
    zpart, ssq = oracle.btp_shard_partials(w["x"], w["gamma"], w["A"], S, flow="exact")
    x, A, g = w["x"], w["A"], w["gamma"]
    np.testing.assert_allclose(zpart.sum(axis=0), x @ (g[:, None] * A), rtol=1e-12, atol=1e-12)
    a, srow = oracle.btp_reduce(zpart, ssq, x.shape[1], flow="exact")
    _, cache = oracle.block_fwd(x, g, A, w["B"], S=S, flow="exact")
    np.testing.assert_allclose(srow, cache["s"], rtol=1e-14)
    np.testing.assert_allclose(a, cache["a"], rtol=1e-12, atol=1e-13)
    # and the plain definition: act(RMSNorm(x) @ A)
    ref = oracle.silu((x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-5)) * g @ A)
    np.testing.assert_allclose(a, ref, rtol=1e-11, atol=1e-12)


def test_a_rank_sees_only_its_shard():
    # perturbing x outside shard s leaves rank s's contribution bit for bit unchanged
    w = _case(d=96)
    S = 3
    off = oracle.shard_bounds(96, S)
    z0, q0 = oracle.btp_shard_partials(w["x"], w["gamma"], w["A"], S, flow="exact")
    x2 = w["x"].copy()
    x2[:, off[1]:] += 1.0                      # touch shards 1 and 2 only
    z1, q1 = oracle.btp_shard_partials(x2, w["gamma"], w["A"], S, flow="exact")
    assert np.array_equal(z0[0], z1[0]) and np.array_equal(q0[0], q1[0])
    assert not np.array_equal(z0[1], z1[1])


def test_payload_is_the_fused_exchange_size():
    T, d, r, k, S = 24, 64, 8, 2, 4
    w = _case(T=T, d=d, r=r, k=k)
    zpart, ssq = oracle.btp_shard_partials(w["x"], w["gamma"], w["A"], S)
    assert zpart.size + ssq.size == S * oracle.exchange_elems(T, k, r)
    assert zpart.shape == (S, T, k * r) and ssq.shape == (S, T)
    nonorm, none = oracle.btp_shard_partials(w["x"], None, w["A"], S, has_norm=False)
    assert none is None and nonorm.size == S * T * k * r


def test_partials_brute_force_on_a_tiny_case():
    rng = np.random.default_rng(5)
    T, d, kr, S = 3, 6, 4, 3
    x = oracle.to_bf16(rng.standard_normal((T, d)))
    A = oracle.to_bf16(rng.standard_normal((d, kr)))
    g = oracle.to_bf16(1 + 0.1 * rng.standard_normal(d))
    zpart, ssq = oracle.btp_shard_partials(x, g, A, S, flow="exact")
    w = d // S
    for s in range(S):
        for t in range(T):
            q = 0.0
            for j in range(s * w, (s + 1) * w):
                q += x[t, j] * x[t, j]
            assert ssq[s, t] == pytest.approx(q, rel=1e-15)
            for m in range(kr):
                v = 0.0
                for j in range(s * w, (s + 1) * w):
                    v += x[t, j] * (g[j] * A[j, m])
                assert zpart[s, t, m] == pytest.approx(v, rel=1e-13, abs=1e-15)


def test_shard_local_mean_is_caught():
    # planted mistake: dividing each rank's statistic by its shard width instead of d
    w = _case()
    S = 4
    zpart, ssq = oracle.btp_shard_partials(w["x"], w["gamma"], w["A"], S, flow="exact")
    a_ok, _ = oracle.btp_reduce(zpart, ssq, 64, flow="exact")
    a_bad, _ = oracle.btp_reduce(zpart, ssq, 64 // S, flow="exact")
    _, cache = oracle.block_fwd(w["x"], w["gamma"], w["A"], w["B"], S=S, flow="exact")
    assert np.allclose(a_ok, cache["a"], rtol=1e-12, atol=1e-13)
    assert not np.allclose(a_bad, cache["a"], rtol=1e-3)


def test_no_norm_reduce_is_the_plain_product():
    w = _case()
    zpart, ssq = oracle.btp_shard_partials(w["x"], None, w["A"], 4, has_norm=False, flow="exact")
    a, srow = oracle.btp_reduce(zpart, ssq, 64, flow="exact")
    assert np.array_equal(srow, np.ones(24))
    np.testing.assert_allclose(a, oracle.silu(w["x"] @ w["A"]), rtol=1e-12, atol=1e-13)
