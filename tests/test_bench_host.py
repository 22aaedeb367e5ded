"""Host-side checks of bench.py: the multi-rank timing reduction over gloo ranks on
CPU (world size 2), the weak-scaling aggregate, the FLOP model, and the reference
arm's rank handling. No GPU is used."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 10.0 + 5.0 * rank           # each rank's own elapsed time
        dist.barrier()
        m = bench.max_over_ranks(local, dist, "cpu")
        out[rank] = m
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == 15.0


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5


def test_weak_scaling_aggregate():
    # N replicas each processing T*K tokens in the slowest rank's time
    assert bench.aggregate_rate(4, 16384 * 10, 2.0) == 4 * 16384 * 10 / 2.0


def test_flop_model_matches_per_block_formula():
    exe, model = bench.mlp_flops(16384, 4096, 1024, 11008)
    assert exe == 5205500362752          # 8 T d kr + 6 T kr n per block, two blocks
    assert model == (6 * 16384 * 4096 * 2048 + 6 * 16384 * 2048 * 11008 +
                     6 * 16384 * 11008 * 1024 + 6 * 16384 * 1024 * 4096)


def test_reference_arm_nonzero_ranks_do_no_work(capsys):
    class A:
        steps, warmup = 1, 0
    assert bench.reference_arm(A(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""


def test_dense_fullrank_context_is_the_textbook_mlp():
    # the full-rank comparison leg (torch) against the plain fp64 definition on a tiny
    # case: forward and every gradient
    import numpy as np

    T, d, ffn = 6, 16, 24
    step, t = bench.dense_mlp(T, d, ffn, "cpu", seed=3, dtype=torch.float64)
    out = step().detach().numpy()
    x, g, Wg, Wu, Wd, dout = (t[k].detach().numpy() for k in ("x", "gamma", "Wg", "Wu", "Wd",
                                                                 "dout"))
    rs = 1.0 / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-5)
    n = x * rs * g
    a, b = n @ Wg, n @ Wu
    sg = 1.0 / (1.0 + np.exp(-a))
    h = a * sg * b
    np.testing.assert_allclose(out, h @ Wd, rtol=1e-12, atol=1e-12)
    dh = dout @ Wd.T
    da = dh * b * sg * (1 + a * (1 - sg))
    db = dh * a * sg
    dn = da @ Wg.T + db @ Wu.T
    np.testing.assert_allclose(t["Wd"].grad.numpy(), h.T @ dout, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(t["Wg"].grad.numpy(), n.T @ da, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(t["Wu"].grad.numpy(), n.T @ db, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(t["gamma"].grad.numpy(), (dn * x * rs).sum(axis=0), rtol=1e-10,
                               atol=1e-12)
    xh = x * rs
    dxh = dn * g
    dx = rs * (dxh - xh * (dxh * xh).mean(axis=1, keepdims=True))
    np.testing.assert_allclose(t["x"].grad.numpy(), dx, rtol=1e-10, atol=1e-12)
    assert bench.dense_mlp_flops(T, d, ffn) == 6.0 * T * 3 * d * ffn


def test_workload_flop_model():
    # the default workload's model is the MLP's; a single block is 8 T d kr + 6 T kr n
    assert bench.workload_flops("llama2_7b_mlp", 16384) == bench.mlp_flops(16384, 4096, 1024,
                                                                           11008)
    exe, model = bench.workload_flops("llama2_1b_attn_block", 100)
    assert exe == 8 * 100 * 2048 * 1536 + 6 * 100 * 1536 * 2048
    assert model == 6 * 100 * 2048 * 1536 + 6 * 100 * 1536 * 2048
    # the layer: QKV + O + the MLP's two blocks
    lay, _ = bench.workload_flops("llama2_13b_layer", 1)
    d, r, f = 5120, 1280, 13824
    assert lay == sum(8 * di * kr + 6 * kr * n for di, kr, n in
                      [(d, 3 * r, d), (d, r, d), (d, 2 * r, f), (f, r, d)])


def test_dominant_kernel_skips_overlapped_operations():
    # an overlapped operation's event interval includes time shared with its concurrent
    # siblings, so it is never named the dominant kernel while a serial one exists
    prof = {"gemm_wgrad_B": (2, 9.0, 1e12, 1e9), "gemm_dual": (2, 5.0, 2e12, 1e9),
            "gemm_down_act": (2, 3.0, 1e12, 1e9)}
    name, _ = bench.dominant_kernel(prof, set(bench.OVERLAPPED_OPS))
    assert name == "gemm_dual"
    assert bench.dominant_kernel(prof, set())[0] == "gemm_wgrad_B"
    only = {"gemm_wgrad_B": (1, 1.0, 1.0, 1.0)}
    assert bench.dominant_kernel(only, set(bench.OVERLAPPED_OPS))[0] == "gemm_wgrad_B"


def test_step_spread_median_and_percentiles():
    s = bench.step_spread([5.0, 1.0, 3.0, 2.0, 4.0])
    assert s == {"median": 3.0, "p10": 1.0, "p90": 5.0, "min": 1.0, "max": 5.0, "samples": 5}
    s = bench.step_spread([float(i) for i in range(1, 11)])   # even count: mean of the middle two
    assert s["median"] == 5.5 and s["p10"] == 2.0 and s["p90"] == 9.0 and s["samples"] == 10
    assert bench.step_spread([]) is None


def test_report_line_carries_the_contract_keys(capsys):
    # one JSON line with the keys the driver reads, from a synthetic profile (no GPU)
    import argparse
    import json

    T, d, r, ffn, S, steps = 16384, 4096, 1024, 11008, 8, 10
    args = argparse.Namespace(steps=steps, warmup=5, workload=bench.WORKLOAD, skip_aux=True,
                              timing="eager",
                              step_ms=bench.step_spread([3.7] * steps))
    exe, _ = bench.workload_flops(bench.WORKLOAD, T)
    ms_total = 37.0
    # name -> (launches, ms, flops, bytes) over the timed steps
    prof = {"gemm_dual": (2 * steps, 10.0, 0.3 * exe * steps, 1e9),
            "gemm_up_swiglu": (steps, 5.0, 0.14 * exe * steps, 1e9),
            "gemm_dx_swiglu": (steps, 4.0, 0.07 * exe * steps, 1e10),
            "rmsnorm_stats": (steps, 0.3, 0.0, 1.3e9)}
    clocks = {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert bench._report(args, 1, prof, {"gemm_dual": 4 * steps}, clocks, ms_total,
                         float("nan"), 0, 0, T, d, r, ffn, S) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches", "step_ms"):
        assert key in line, key
    assert line["metric"] == bench.METRIC and line["unit"] == "tokens/s"
    assert line["value"] == pytest.approx(T * steps / (ms_total / 1e3))
    assert line["ms_per_step"] == pytest.approx(ms_total / steps)
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["n_gpus"] == 1 and line["config"]["workload"] == bench.WORKLOAD
    roof = line["roofline"]
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= set(roof)
    # the dominant kernel is taken among the operations timed alone (gemm_dual here)
    assert roof["kernel"] == "gemm_dual" and roof["bound"] == "tensor"
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    # no power-cap share in these clocks: the burst peak, both fractions printed
    peaks = bench.load_peaks()
    assert roof["peak"] == peaks["bf16_tflops"] and roof["peak_kind"].endswith("burst")
    assert roof["frac_burst"] == pytest.approx(roof["achieved"] / peaks["bf16_tflops"])
    assert roof["frac_sustained"] == pytest.approx(roof["achieved"] /
                                                   peaks["bf16_tflops_sustained"])
    assert line["gpu_launches"] == 4 * steps + 3 * steps   # kernels, not operations
    assert line["step_ms"]["median"] == pytest.approx(3.7)


def test_launch_switches_read_like_the_library(monkeypatch):
    # the library reads BOOST_PDL (default on) and BOOST_FORK_STREAMS (default off) with
    # atoi: non-zero is on; bench.py reports the same reading in its config
    monkeypatch.delenv("BOOST_PDL", raising=False)
    monkeypatch.delenv("BOOST_FORK_STREAMS", raising=False)
    assert bench._env_flag("BOOST_PDL", 1) and not bench._forked()
    monkeypatch.setenv("BOOST_PDL", "0")
    monkeypatch.setenv("BOOST_FORK_STREAMS", "1")
    assert not bench._env_flag("BOOST_PDL", 1) and bench._forked()
    monkeypatch.setenv("BOOST_PDL", "2")
    assert bench._env_flag("BOOST_PDL", 1)


def test_more_than_one_gpu_prints_unavailable_and_launches_nothing(capsys, monkeypatch):
    # the GEMMs use cluster-multicast TMA loads, which run in single-GPU processes only:
    # a request for 2 GPUs (flag or torchrun environment) prints one line and returns 0
    import json

    monkeypatch.setattr(bench, "ours_arm", lambda *a, **k: pytest.fail("kernels launched"))
    assert bench.main(["--gpus", "2"]) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert "unavailable" in line and "multicast" in line["unavailable"]
    assert line["n_gpus"] == 2 and line["metric"] == bench.METRIC
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")                # non-zero ranks print nothing
    assert bench.main([]) == 0
    assert capsys.readouterr().out == ""
    monkeypatch.setenv("RANK", "0")
    assert bench.main([]) == 0
    assert json.loads(capsys.readouterr().out.strip())["n_gpus"] == 2


def _samples(n_cap, n_free, mhz_cap=1800.0):
    return ([(mhz_cap, 2070.0, 1390.0, {"sw_power_cap"})] * n_cap +
            [(2070.0, 2070.0, 900.0, set())] * n_free)


def test_peak_follows_the_power_cap_share_of_the_timed_region():
    peaks = {"bf16_tflops": 1965.5, "bf16_tflops_sustained": 1783.2}
    # a short region at full clock: burst
    c = bench.summarize_clocks(_samples(1, 13), "nvml")
    assert c["power_cap_share"] == pytest.approx(1 / 14) and c["sm_mhz"] == 2070.0
    assert bench.choose_peak(peaks, c) == ("burst", 1965.5)
    # capped for most of the region: sustained
    c = bench.summarize_clocks(_samples(9, 5), "nvml")
    assert c["sm_mhz"] == 1800.0 and c["reasons"] == ["sw_power_cap"]
    assert bench.choose_peak(peaks, c) == ("sustained", 1783.2)
    # exactly half: sustained; no samples at all: burst
    assert bench.choose_peak(peaks, bench.summarize_clocks(_samples(2, 2), "nvml"))[0] == \
        "sustained"
    assert bench.choose_peak(peaks, bench.summarize_clocks([], "nvml")) == ("burst", 1965.5)
    assert bench.choose_peak(peaks, None) == ("burst", 1965.5)


def test_clock_samples_are_taken_from_the_timed_region_only():
    s = _samples(0, 1)[0]
    capped = _samples(1, 0)[0]
    timed = [(0.5, s), (1.0, capped), (1.5, capped), (3.0, s)]
    c = bench.ClockSampler.select(timed, 0.9, 2.0, "nvml")
    assert c["samples"] == 2 and c["power_cap_share"] == 1.0 and c["sm_mhz"] == 1800.0
    # nothing inside: the sample nearest the region's middle, flagged
    c = bench.ClockSampler.select(timed, 2.4, 2.8, "nvml")
    assert c["samples"] == 0 and "note" in c and c["sm_mhz"] == 2070.0
    assert bench.ClockSampler.select([], 0.0, 1.0, "nvml")["samples"] == 0


def test_roofline_takes_the_dominant_kernel_timed_in_the_timed_region(capsys):
    # the per-operation table comes from a second pass; the roofline line's rate comes
    # from the dominant operation's own events over the timed region (passed as `dom`)
    import argparse
    import json

    T, d, r, ffn, S, steps = 16384, 4096, 1024, 11008, 8, 10
    args = argparse.Namespace(steps=steps, warmup=5, workload=bench.WORKLOAD, skip_aux=True,
                              timing="eager", step_ms=None)
    prof = {"gemm_dual": (2 * steps, 10.0, 7.6e12 * steps, 1e9),
            "gemm_up_swiglu": (steps, 5.0, 1.5e12 * steps, 1e9)}
    dom = ("gemm_dual", (2 * steps, 9.5, 7.6e12 * steps, 1e9))
    assert bench._report(args, 1, prof, {}, {}, 36.0, float("nan"), 0, 0, T, d, r, ffn, S,
                         dom=dom) == 0
    roof = json.loads(capsys.readouterr().out.strip().splitlines()[-1])["roofline"]
    assert roof["kernel"] == "gemm_dual"
    assert roof["achieved"] == pytest.approx(7.6e12 * steps / 9.5e-3 / 1e12)
    assert roof["launches_per_step"] == 2
