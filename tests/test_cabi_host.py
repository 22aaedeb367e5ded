"""Host-side tests of the C ABI (no GPU needed): the library loads, exports every
symbol the headers declare, reports the exact shard/group/exchange bookkeeping,
and rejects bad arguments before touching CUDA.
"""

import ctypes
import glob
import os
import re

import pytest

import oracle
from rank_bottleneck_online_gb300 import binding as B
from rank_bottleneck_online_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return B.lib()


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(boost_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_abi():
    names = _declared_symbols()
    assert "boost_block_fwd" in names and "boost_block_bwd" in names
    assert set(names) == set(B.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared_symbols():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


@pytest.mark.parametrize("T,d,r,k,n,S", [(128, 256, 64, 3, 256, 4), (16384, 4096, 1024, 2, 11008, 8),
                                         (7, 24, 8, 1, 8, 3), (0, 64, 8, 5, 16, 64)])
def test_layout_bookkeeping_is_exact(L, T, d, r, k, n, S):
    desc = B.make_desc(T, d, r, k, n, S=S)
    so, go, ex = B.layout(desc)
    assert so == oracle.shard_bounds(d, S)
    assert go == oracle.group_bounds(k, r)
    assert ex == oracle.exchange_elems(T, k, r)
    # payload ratio of the fused exchange against a d-wide reduce of the same rows
    if T:
        assert ex / (T * d) == pytest.approx((k * r + 1) / d)


def test_layout_without_norm_has_one_shard(L):
    desc = B.make_desc(4, 16, 8, 2, 8, S=4, has_norm=False)
    so, go, ex = B.layout(desc)
    assert so == [0, 16]


def test_status_strings(L):
    for code in range(8):
        s = L.boost_status_string(code)
        assert s and len(s) > 1
    assert L.boost_status_string(99) == b"unknown status"


def _fake(addr):
    return ctypes.c_void_p(addr)


def _fwd(L, desc, x=0x10000, g=0x20000, A=0x30000, Bw=0x40000, y=0x50000, rstd=None,
         ws=0x100000, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = B.workspace_bytes(desc) or 1 << 20
    return L.boost_block_fwd(ctypes.byref(desc), _fake(x), _fake(g) if g else None, _fake(A),
                             _fake(Bw), _fake(y), _fake(rstd) if rstd else None, _fake(ws),
                             ws_bytes, None)


@pytest.mark.parametrize("bad,want", [
    (dict(d=250), 2),            # d not a multiple of 8
    (dict(S=3), 2),              # d % S != 0
    (dict(S=0), 1),              # no shards
    (dict(r=12), 2),             # r not a multiple of 8
    (dict(n=20), 2),             # n not a multiple of 8
    (dict(T=-1), 1),
    (dict(k=0), 1),
    (dict(act=7), 1),
])
def test_invalid_desc_rejected(L, bad, want):
    kw = dict(T=128, d=256, r=64, k=3, n=256, S=4, act="silu")
    kw.update(bad)
    desc = B.make_desc(kw["T"], kw["d"], kw["r"], kw["k"], kw["n"], S=kw["S"], act=kw["act"])
    assert _fwd(L, desc) == want
    assert L.boost_block_workspace_bytes(ctypes.byref(desc)) == 0


def test_pointer_and_workspace_checks(L):
    desc = B.make_desc(128, 256, 64, 3, 256, S=4)
    assert _fwd(L, desc, x=0x10008) == 3                       # misaligned x
    assert _fwd(L, desc, y=0) == 1                             # missing output
    assert _fwd(L, desc, g=0) == 1                             # normed block without gamma
    assert _fwd(L, desc, ws=0x100010) == 4                     # workspace not 256-aligned
    assert _fwd(L, desc, ws_bytes=1024) == 4                   # workspace too small
    nonorm = B.make_desc(128, 256, 64, 3, 256, S=4, has_norm=False)
    assert _fwd(L, nonorm) == 1                                # gamma given without norm
    assert _fwd(L, nonorm, g=0, rstd=0x60000) == 1             # rstd given without norm


def test_bwd_argument_checks(L):
    desc = B.make_desc(128, 256, 64, 3, 256, S=4)
    ws_bytes = B.workspace_bytes(desc)
    f = _fake
    # dgamma missing for a normed block
    st = L.boost_block_bwd(ctypes.byref(desc), f(0x1000), f(0x2000), f(0x3000), f(0x4000), None,
                           f(0x5000), f(0x6000), None, f(0x7000), f(0x8000), f(0x100000),
                           ws_bytes, None)
    assert st == 1
    st = L.boost_block_bwd(ctypes.byref(desc), f(0x1000), f(0x2000), f(0x3000), f(0x4000), None,
                           f(0x5004), f(0x6000), f(0x6100), f(0x7000), f(0x8000), f(0x100000),
                           ws_bytes, None)
    assert st == 3                                             # misaligned dy


def test_fused_swiglu_forward_argument_checks(L):
    f = _fake

    def fwd_glu(desc, h):
        return L.boost_block_fwd_swiglu(ctypes.byref(desc), f(0x1000), f(0x2000), f(0x3000),
                                        f(0x4000), f(0x5000), h, None, f(0x100000), 1 << 30,
                                        None)

    assert fwd_glu(B.make_desc(128, 256, 64, 3, 256, S=4), f(0x6000)) == 1   # k must be 2
    assert fwd_glu(B.make_desc(128, 256, 64, 2, 256, S=4), None) == 1        # h missing
    assert fwd_glu(B.make_desc(128, 256, 64, 2, 256, S=4), f(0x6008)) == 3   # h misaligned


def test_btp_emulation_argument_checks(L):
    f = _fake

    def fwd_btp(desc, payload):
        return L.boost_block_fwd_btp(ctypes.byref(desc), f(0x1000), f(0x2000), f(0x3000),
                                     f(0x4000), f(0x5000), None, payload, f(0x100000), 1 << 30,
                                     None)

    # shards must be whole 64-deep k-blocks: d / S = 48
    assert fwd_btp(B.make_desc(128, 192, 64, 2, 256, S=4), f(0x6000)) == 2
    assert fwd_btp(B.make_desc(128, 256, 64, 2, 256, S=4), None) == 1       # payload missing
    assert fwd_btp(B.make_desc(128, 256, 64, 2, 256, S=4), f(0x6004)) == 3  # misaligned
    assert fwd_btp(B.make_desc(128, 256, 64, 2, 256, S=3), f(0x6000)) == 2  # d % S != 0


def test_elementwise_argument_checks(L):
    assert L.boost_swiglu_fwd(4, 12, _fake(0x1000), _fake(0x2000), _fake(0x3000), None) == 2
    assert L.boost_swiglu_fwd(-1, 8, _fake(0x1000), _fake(0x2000), _fake(0x3000), None) == 1
    assert L.boost_add(12, _fake(0x1000), _fake(0x2000), _fake(0x3000), None) == 2
    assert L.boost_add(0, None, None, None, None) == 0         # empty is a no-op
    assert L.boost_debug_wait_timeout(_fake(0x100000), 256, 0, None) == 1
    assert L.boost_debug_wait_timeout(_fake(0x100010), 256, 10, None) == 4


def test_workspace_size_grows_with_shape(L):
    small = B.workspace_bytes(B.make_desc(128, 256, 64, 3, 256, S=4))
    big = B.workspace_bytes(B.make_desc(16384, 2048, 512, 3, 2048, S=4))
    assert 0 < small < big
    # a, dzs [T, kr] bf16 and A' [d, kr] bf16 at least
    assert big >= 2 * 16384 * 1536 * 2 + 2048 * 1536 * 2


def test_empty_token_batch_is_a_no_op_for_every_forward_entry(L):
    # T = 0: the [T, ...] tensors are empty and may be NULL; nothing is enqueued
    f = _fake
    desc = B.make_desc(0, 256, 64, 2, 256, S=4)
    ws_bytes = B.workspace_bytes(desc)
    assert ws_bytes > 0
    assert L.boost_block_fwd(ctypes.byref(desc), None, f(0x2000), f(0x3000), f(0x4000), None,
                             None, f(0x100000), ws_bytes, None) == 0
    assert L.boost_block_fwd_swiglu(ctypes.byref(desc), None, f(0x2000), f(0x3000), f(0x4000),
                                    None, None, None, f(0x100000), ws_bytes, None) == 0
    assert L.boost_block_fwd_btp(ctypes.byref(desc), None, f(0x2000), f(0x3000), f(0x4000),
                                 None, None, None, f(0x100000), ws_bytes, None) == 0
    assert L.boost_block_up(ctypes.byref(desc), None, f(0x4000), None, None, f(0x100000),
                            ws_bytes, None) == 0


def test_bottleneck_up_projection_argument_checks(L):
    f = _fake
    desc = B.make_desc(128, 256, 64, 3, 256, S=4)
    ws_bytes = B.workspace_bytes(desc)
    # h (the fused SwiGLU output) needs the gate and up groups: k == 2
    assert L.boost_block_up(ctypes.byref(desc), f(0x1000), f(0x2000), f(0x3000), f(0x4000),
                            f(0x100000), ws_bytes, None) == 1
    assert L.boost_block_up(ctypes.byref(desc), None, f(0x2000), f(0x3000), None, f(0x100000),
                            ws_bytes, None) == 1          # a missing
    assert L.boost_block_up(ctypes.byref(desc), f(0x1008), f(0x2000), f(0x3000), None,
                            f(0x100000), ws_bytes, None) == 3   # a misaligned
    assert L.boost_block_up(ctypes.byref(desc), f(0x1000), f(0x2000), f(0x3000), None,
                            f(0x100000), 64, None) == 4          # workspace too small


def test_profile_only_argument_checks(L):
    # one kernel id, or -1 for every kernel; anything else is rejected
    n = L.boost_profile_kernel_count()
    assert L.boost_profile_only(-2) == 1 and L.boost_profile_only(n) == 1
    assert L.boost_profile_only(n - 1) == 0 and L.boost_profile_only(-1) == 0


def test_residual_entry_point_argument_checks(L):
    # the residual forms of forward and backward reject, before enqueuing anything: more
    # than one output group, a missing residual, a misaligned residual; the forward with
    # T = 0 is a no-op (the backward's zeroed weight gradients need the device)
    f = _fake
    ok = B.make_desc(128, 256, 64, 1, 256, S=4)
    ws_bytes = B.workspace_bytes(ok)

    def fwd(desc, res, wsb=ws_bytes):
        return L.boost_block_fwd_residual(ctypes.byref(desc), f(0x10000), f(0x20000),
                                          f(0x30000), f(0x40000), f(res) if res else None,
                                          f(0x50000), None, f(0x100000), wsb, None)

    def bwd(desc, res, wsb=ws_bytes):
        return L.boost_block_bwd_residual(ctypes.byref(desc), f(0x1000), f(0x2000), f(0x3000),
                                          f(0x4000), None, f(0x5000), f(res) if res else None,
                                          f(0x6000), f(0x6100), f(0x7000), f(0x8000),
                                          f(0x100000), wsb, None)

    three = B.make_desc(128, 256, 64, 3, 256, S=4)
    assert fwd(three, 0x60000, B.workspace_bytes(three)) == 1   # k != 1
    assert fwd(ok, 0) == 1                                      # no residual
    assert fwd(ok, 0x60008) == 3                                # misaligned residual
    assert bwd(ok, 0) == 1
    assert bwd(ok, 0x60008) == 3
    # a residual that overlaps the output without being it (y at 0x50000, dx at 0x6000;
    # T * n * 2 = 64 KB): rejected; the output itself is allowed only as the same buffer
    assert fwd(ok, 0x50010) == 1
    assert bwd(ok, 0x6010) == 1
    empty = B.make_desc(0, 256, 64, 1, 256, S=4)
    wsb0 = B.workspace_bytes(empty) or 1 << 20
    assert fwd(empty, 0, wsb0) == 0


@pytest.mark.parametrize("lang,std", [("c", "-std=c11"), ("c++", "-std=c++17")])
def test_header_compiles_as_plain_c_and_cpp(lang, std):
    # the boundary header declares a C ABI: it must parse as C (and as C++) on its own
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                       "boost_block.h")
    r = subprocess.run([cc, "-fsyntax-only", "-Wall", "-Werror", "-x", lang, std, hdr],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _kernel_bodies(path):
    """name -> body text of every __global__ function in a CUDA source file."""
    text = open(path).read()
    out = {}
    for m in re.finditer(r"__global__\s+void\s+(?:__launch_bounds__\([^)]*\)\s+)?(\w+)\s*\(",
                         text):
        start = text.index("{", text.index(")", m.end()))
        depth, i = 0, start
        while True:
            depth += {"{": 1, "}": -1}.get(text[i], 0)
            i += 1
            if depth == 0:
                break
        out[m.group(1)] = text[start + 1:i - 1]
    return out


def test_programmatic_launches_wait_before_touching_memory():
    # kernels launched with the programmatic-stream-serialisation attribute may start
    # while the kernel before them runs: each must wait (griddepcontrol.wait) before any
    # global memory access. The CUDA-core kernels launched through launch_k / launch_kb
    # begin with pdl_enter(); the GEMM waits after its prologue (shared memory, TMEM and
    # the parameter-space tensor maps only), before its roles start.
    csrc = os.path.join(ROOT, "rank_bottleneck_online_gb300", "csrc")
    simple = open(os.path.join(csrc, "kernels_simple.cu")).read()
    launched = set(re.findall(r"launch_kb?\((\w+)", simple))
    launched |= set(re.findall(r"\?\s*(\w+_kernel)\b", simple))
    launched |= set(re.findall(r":\s*(\w+_kernel)\b", simple))
    launched = {k.split("<")[0] for k in launched if k.endswith("_kernel")}
    bodies = _kernel_bodies(os.path.join(csrc, "kernels_simple.cu"))
    assert launched and launched <= set(bodies), launched - set(bodies)
    for name in launched:
        first = bodies[name].strip().split(";")[0].strip()
        assert first == "pdl_enter()", f"{name} starts with {first!r}"
    assert "<<<" not in simple.split("launch_wait_timeout_probe")[0], \
        "plain launches before the probe: use launch_k"
    gemm = _kernel_bodies(os.path.join(csrc, "gemm.cuh"))["gemm_kernel"]
    wait = gemm.index("griddep_wait();")
    assert gemm.index("griddep_launch_dependents();") > wait
    assert wait < gemm.index("if (warp == 0) {\n    // ------") , \
        "the GEMM must wait before its roles start"
    for access in ("p.err", "p.out", "p.rstd", "p.qpart", "p.dgpart", "p.res"):
        pos = gemm.find(access)
        assert pos == -1 or pos > wait, f"{access} used before griddep_wait"
