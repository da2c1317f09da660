"""The C-ABI library on the CPU: it loads, exports every function include/ft_moe.h
declares, and rejects invalid arguments on the host before touching the GPU (the fake
pointers below are never dereferenced: every call fails validation first)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "ft_moe.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_mixture_experts_02_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from nvfp4_mixture_experts_02_gb300 import ftmoe
    return ftmoe


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ft_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("ft_moe_route", "ft_moe_nvfp4_decode", "ft_moe_nvfp4_prefill"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(so, name), f"{name} declared in ft_moe.h but not exported"
    assert set(declared_functions()) == set(lib.EXPORTED)


def test_version_and_status_strings(lib):
    assert lib.abi_version() == 1
    for st in range(8):
        assert lib.status_string(st).startswith(lib.STATUS_NAMES[st])


def test_workspace_bytes(lib):
    small = lib.workspace_bytes(1, 2, 8, 256, 128, False)
    assert small > 0 and small % 256 == 0
    assert lib.workspace_bytes(1, 10, 512, 4096, 1024, True) > small
    assert lib.workspace_bytes(65, 10, 512, 4096, 1024, True) == 0     # decode limit T<=64
    assert lib.workspace_bytes(1, 9, 8, 256, 128, False) == 0          # k > E


def _experts(lib, E=8, H=256, I=128, base=0x10000, **over):
    p = dict(w13=base, w13_scale=base + 0x1000, w13_gscale=base + 0x2000, w2=base + 0x3000,
             w2_scale=base + 0x4000, w2_gscale=base + 0x5000)
    p.update(over)
    return lib._Experts(E, H, I, p["w13"], p["w13_scale"], p["w13_gscale"], p["w2"],
                        p["w2_scale"], p["w2_gscale"])


def _decode(lib, ex, T=1, k=2, x=0x20000, idx=0x30000, w=0x40000, out=0x50000, ws=0x60000,
            limit=7.0, ws_bytes=1 << 30):
    return lib.lib().ft_moe_nvfp4_decode(x, T, idx, w, k, ctypes.byref(ex), None, limit, out,
                                         ws, ws_bytes, None)


@pytest.mark.parametrize("case,expect", [
    (dict(ex=dict(w13=0)), 1),                       # null weight pointer
    (dict(ex=dict(H=200)), 2),                       # H not a multiple of 128
    (dict(ex=dict(I=96)), 2),                        # I not a multiple of 128
    (dict(ex=dict(E=5000)), 2),                      # too many experts
    (dict(ex=dict(w2=0x10008)), 3),                  # misaligned weight pointer
    (dict(call=dict(k=9)), 1),                       # k > E
    (dict(call=dict(k=0)), 1),
    (dict(call=dict(T=-1)), 1),
    (dict(call=dict(T=65)), 2),                      # decode batch limit
    (dict(call=dict(limit=0.0)), 1),
    (dict(call=dict(limit=float("nan"))), 1),
    (dict(call=dict(limit=1000.0)), 1),
    (dict(call=dict(x=0x20002)), 3),                 # misaligned activations
    (dict(call=dict(ws=0x60010)), 3),                # workspace not 256-byte aligned
    (dict(call=dict(ws_bytes=16)), 4),               # workspace too small
    (dict(call=dict(out=0)), 1),
])
def test_decode_rejects_invalid_arguments(lib, case, expect):
    exargs = dict(case.get("ex", {}))
    dims = {k_: exargs.pop(k_) for k_ in ("E", "H", "I") if k_ in exargs}
    ex = _experts(lib, **dims, **exargs)
    assert _decode(lib, ex, **case.get("call", {})) == expect


def test_route_rejects_invalid_arguments(lib):
    f = lib.lib().ft_moe_route
    assert f(0, 1, 8, 2, 0x1000, 0x2000, None) == 1          # null logits
    assert f(0x1000, 1, 8, 9, 0x1000, 0x2000, None) == 1     # k > E
    assert f(0x1000, 1, 64, 33, 0x1000, 0x2000, None) == 2   # k > 32
    assert f(0x1002, 1, 8, 2, 0x1000, 0x2000, None) == 3     # misaligned
    assert f(0x1000, -1, 8, 2, 0x1000, 0x2000, None) == 1    # T < 0


def test_empty_batch_is_a_no_op(lib):
    """T = 0: FT_OK without touching any buffer (all pointers NULL), no workspace needed."""
    f = lib.lib()
    ex = _experts(lib)
    assert f.ft_moe_route(0, 0, 8, 2, 0, 0, None) == 0
    assert f.ft_moe_workspace_bytes(0, 2, 8, 256, 128, 0, 0) == 0
    assert f.ft_moe_workspace_bytes(0, 2, 8, 256, 128, 0, 1) == 0
    for fn in (f.ft_moe_nvfp4_decode, f.ft_moe_nvfp4_prefill):
        assert fn(None, 0, None, None, 2, ctypes.byref(ex), None, 7.0, None, None, 0, None) == 0
    assert f.ft_moe_nvfp4_decode_noalloc(None, 0, None, None, 2, ctypes.byref(ex), None, 7.0,
                                         None, None) == 0
    # the shape checks still apply to an empty batch
    assert f.ft_moe_nvfp4_decode(None, 0, None, None, 9, ctypes.byref(ex), None, 7.0, None,
                                 None, 0, None) == 1


def test_decode_shared_memory_fits_every_accepted_shape(lib):
    """Every shape decode accepts (T <= 64, k <= 32, E <= 4096, H <= 16384, I <= 8192) fits
    the kernel's 224 KB of shared memory per CTA: the plan, x when kept on chip, the rings."""
    f = lib.lib().ft_moe_decode_smem_bytes
    budget = 224 * 1024
    worst = 0
    for T in (1, 2, 5, 8, 16, 32, 33, 63, 64):
        for k in (1, 2, 8, 10, 16, 32):
            for E in (32, 64, 288, 512, 1024, 2048, 4096):
                if k > E:
                    continue
                for H in (128, 256, 512, 1024, 4096, 16384):
                    for I in (128, 1024, 8192):
                        for sh in (0, 1):
                            n = f(T, k, E, H, I, sh)
                            assert 0 < n <= budget, (T, k, E, H, I, sh, n)
                            worst = max(worst, n)
    assert worst == budget   # the launch asks for the whole budget
    assert f(65, 2, 8, 256, 128, 0) == 0 and f(1, 33, 64, 256, 128, 0) == 0


C_CALLER = r"""
#include <stdio.h>
#include "ft_moe.h"
int main(void) {
  /* host-side calls only: the version, a status string, a workspace size and an argument
     error that is returned before anything touches a GPU */
  ft_status st = ft_moe_route(NULL, 1, 8, 2, NULL, NULL, NULL);
  printf("%d|%s|%zu|%d\n", ft_moe_abi_version(), ft_status_string(FT_ERR_MISALIGNED),
         ft_moe_workspace_bytes(1, 2, 8, 256, 128, 0, 0), (int)st);
  return st == FT_ERR_INVALID_ARG ? 0 : 1;
}
"""


def test_header_serves_a_plain_c_caller(lib, tmp_path):
    """include/ft_moe.h compiles as strict C11 and a C program links and calls the library."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src, exe = tmp_path / "caller.c", tmp_path / "caller"
    src.write_text(C_CALLER)
    libdir = os.path.dirname(lib.LIB_PATH)
    res = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                          "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir, "-lftmoe",
                          f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, run.stdout + run.stderr
    version, status, ws, st = run.stdout.strip().split("|")
    assert int(version) == lib.abi_version() and status.startswith("FT_ERR_MISALIGNED")
    assert int(ws) == lib.workspace_bytes(1, 2, 8, 256, 128, False) and int(st) == 1


@pytest.mark.parametrize("call,expect", [
    (dict(limit=-1.0), 1),                       # SwiGLU limit out of range
    (dict(x=0x20002), 3),                        # misaligned activations
    (dict(ex=dict(H=200)), 2),                   # H not a multiple of 128
    (dict(ex=dict(w13=0)), 1),                   # null weight pointer
])
def test_noalloc_checks_every_argument_before_any_cuda_call(lib, call, expect):
    """ft_moe_nvfp4_decode_noalloc runs all the workspace entry point's host checks before
    its first CUDA call: with no GPU here, a check that came later would surface as
    FT_ERR_CUDA instead of the argument's own status."""
    call = dict(call)
    ex = _experts(lib, **call.pop("ex", {}))
    a = dict(x=0x20000, idx=0x30000, w=0x40000, out=0x50000, limit=7.0)
    a.update(call)
    st = lib.lib().ft_moe_nvfp4_decode_noalloc(a["x"], 1, a["idx"], a["w"], 2, ctypes.byref(ex),
                                               None, a["limit"], a["out"], None)
    assert st == expect, lib.status_string(st)


def test_wait_limit_hook(lib):
    assert lib.lib().ft_moe_debug_set_wait_limit(0) == 0
    assert lib.lib().ft_moe_debug_set_wait_limit(-1) == 0
    lib.debug_set_wait_limit(None)


def test_layer_from_host_rejects_invalid_arguments(lib):
    """Checked on the host before any copy is enqueued (no GPU here: a check that came after
    a CUDA call would surface as FT_ERR_CUDA)."""
    f = lib.lib().ft_moe_layer_from_host
    ex = _experts(lib)
    good = dict(xh=0x1000, lh=0x2000, T=1, k=2, oh=0x3000, xd=0x20000, ld=0x30000, idd=0,
                wd=0, od=0x50000, ws=0x60000, wsb=1 << 30, limit=7.0)

    def call(**o):
        a = dict(good, **o)
        return f(a["xh"], a["lh"], a["T"], a["k"], ctypes.byref(ex), None, a["limit"], a["oh"],
                 a["xd"], a["ld"], a["idd"], a["wd"], a["od"], a["ws"], a["wsb"], None)

    assert call(xh=0) == 1                       # null host input
    assert call(od=0) == 1                       # null device output
    assert call(limit=0.0) == 1
    assert call(xd=0x20008) == 3                 # misaligned device activations
    assert call(ws=0x60010) == 3                 # misaligned workspace
    assert call(wsb=16) == 4                     # workspace too small
    assert call(T=100) == 1                      # prefill-sized batch without slot buffers
    assert call(T=0, xh=0, lh=0, oh=0, xd=0, ld=0, od=0, ws=0) == 0   # empty batch


def test_fp8block_argument_checks(lib):
    """Host checks of the block-FP8 decode entry point (nothing reaches the GPU)."""
    f = lib.lib()
    ex = lib._F8Experts(8, 256, 128, 0x10000, 0x20000, 0x30000, 0x40000)
    call = lambda ex_, T=1, k=2, x=0x50000, limit=7.0, ws=0x60000, wsb=1 << 30: \
        f.ft_moe_fp8block_decode(x, T, 0x70000, 0x80000, k, ctypes.byref(ex_), None, limit,
                                 0x90000, ws, wsb, None)
    assert call(lib._F8Experts(8, 200, 128, 0x10000, 0x20000, 0x30000, 0x40000)) == 2   # H
    assert call(lib._F8Experts(8, 256, 128, 0, 0x20000, 0x30000, 0x40000)) == 1        # null
    assert call(lib._F8Experts(8, 256, 128, 0x10008, 0x20000, 0x30000, 0x40000)) == 3  # align
    assert call(ex, k=9) == 1
    assert call(ex, T=65) == 2
    assert call(ex, limit=-1.0) == 1
    assert call(ex, x=0x50002) == 3
    assert call(ex, wsb=16) == 4
    assert call(ex, T=0, x=0) == 0
    assert f.ft_moe_fp8block_workspace_bytes(1, 2, 8, 256, 128, 0) > 0
    assert f.ft_moe_fp8block_workspace_bytes(65, 2, 8, 256, 128, 0) == 0
    assert f.ft_moe_fp8block_workspace_bytes(1, 2, 8, 200, 128, 0) == 0


def test_router_argument_checks(lib):
    f = lib.lib()
    assert f.ft_moe_router_logits(0x1000, 0, 256, 0x2000, 8, None, 0x3000, None, None) == 0  # T=0
    assert f.ft_moe_router_logits(0x1000, 1, 250, 0x2000, 8, None, 0x3000, None, None) == 2  # H%8
    assert f.ft_moe_router_logits(0x1000, 1, 256, 0x2000, 5000, None, 0x3000, None, None) == 2
    assert f.ft_moe_router_logits(0, 1, 256, 0x2000, 8, None, 0x3000, None, None) == 1
    assert f.ft_moe_router_logits(0x1008, 1, 256, 0x2000, 8, None, 0x3000, None, None) == 3
    assert f.ft_moe_router_logits(0x1000, 1, 256, 0x2000, 8, 0x4000, 0x3000, None, None) == 1
    assert f.ft_moe_router_route(0x1000, 1, 256, 0x2000, 8, None, 9, 0x3000, None, 0x5000,
                                 0x6000, None) == 1                                   # k > E
    assert f.ft_moe_router_route(0x1000, 1, 256, 0x2000, 64, None, 33, 0x3000, None, 0x5000,
                                 0x6000, None) == 2                                   # k > 32
