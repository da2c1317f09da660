"""Helpers for the GPU tests: move a synthetic layer to the device, run the library,
and score a bf16 result against the oracle's float32 output."""
from __future__ import annotations

import contextlib
import multiprocessing
import os

import numpy as np
import torch

# Acceptance bound for the bf16 layer output against the float32 oracle (fp64 arithmetic):
# relative Frobenius error <= 5e-3 over the compared [T, H] rows, and in every token row
# max |err| <= 2e-2 * rms of that row of the oracle output. The max-abs bound is taken per
# row because one token's output is the vector the layer returns for it: over a whole
# 2048-token batch the largest outputs reach ~10x the batch rms, where rounding the exact
# value to bf16 alone (half an ulp, up to 2^-8 of it) exceeds 2e-2 of the batch rms.
REL_FRO_TOL = 5e-3
MAX_ABS_RMS_TOL = 2e-2


def ftmoe():
    from nvfp4_mixture_experts_02_gb300 import ftmoe as m   # raises if the .so is missing
    return m


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def experts_to_device(layer, device="cuda"):
    m = ftmoe()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    ex = m.NvFP4Experts(t(layer.w13), t(layer.s13), t(layer.g13), t(layer.w2), t(layer.s2),
                        t(layer.g2))
    sh = None
    if layer.shared is not None:
        s = layer.shared
        sh = m.NvFP4Shared(t(s["w13"]), t(s["s13"]), t(np.array([s["g13"]], np.float32)),
                           t(s["w2"]), t(s["s2"]), t(np.array([s["g2"]], np.float32)),
                           bf16_tensor(s["gate"], device))
    return ex, sh


def score(y_gpu: np.ndarray, y_ref: np.ndarray):
    """(relative Frobenius error, max over token rows of max |err| / rms(ref row)) in fp64;
    a 1-D input is one row."""
    y_gpu = np.atleast_2d(np.asarray(y_gpu, np.float64))
    y_ref = np.atleast_2d(np.asarray(y_ref, np.float64))
    diff = y_gpu - y_ref
    fro = np.linalg.norm(diff) / max(np.linalg.norm(y_ref), 1e-300)
    rms = np.sqrt(np.mean(y_ref ** 2, axis=-1))
    return fro, float(np.max(np.max(np.abs(diff), axis=-1) / np.maximum(rms, 1e-300)))


def assert_close(y_gpu, y_ref, what="", scale=1.0):
    """Acceptance bound (times `scale`: two results that each meet the bound against the
    oracle differ by at most twice it)."""
    fro, mx = score(y_gpu, y_ref)
    ft, mt = REL_FRO_TOL * scale, MAX_ABS_RMS_TOL * scale
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite output"
    assert fro <= ft and mx <= mt, \
        f"{what}: rel_fro={fro:.3e} (<= {ft}), max_abs/rms(row)={mx:.3e} (<= {mt})"
    return fro, mx


@contextlib.contextmanager
def oracle_pool(workers=None):
    """A map function that runs the oracle's per-expert jobs on a pool of host processes
    (spawned, never forked: the parent already holds a CUDA context), in job order."""
    n = workers or max(1, min(16, (os.cpu_count() or 2) - 1))
    with multiprocessing.get_context("spawn").Pool(n) as pool:
        yield lambda fn, it: pool.imap(fn, it, chunksize=1)
