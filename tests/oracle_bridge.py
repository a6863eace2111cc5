"""Test helpers that hand the same seeded inputs to the oracle and compare.

The oracle quantises fp32 weights itself (never the CUDA path's bytes) and routes with its
own router; the helpers only move generator output between host and device.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from quantized_routed_expert_softmax_gb300 import synth

TOL = 2e-3   # max|err| <= TOL * rms(out), fp32 accumulation against the fp64 oracle


def to_numpy_x(x: torch.Tensor) -> np.ndarray:
    """A device activation tensor as the oracle takes it: fp32 array or bf16 bits."""
    if x.dtype == torch.float32:
        return x.detach().cpu().numpy()
    return x.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_layer(w: synth.Workload, router_w: np.ndarray, gu_f32, dn_f32, experts) -> oracle.Layer:
    """An oracle.Layer holding canonical bytes (quantised by the oracle) for `experts`.

    gu_f32 / dn_f32: callables e -> fp32 numpy matrix (generator output)."""
    gu = [None] * w.E
    dn = [None] * w.E
    gts = np.ones(w.E, np.float32)
    dts = np.ones(w.E, np.float32)
    for e in sorted(set(int(v) for v in experts)):
        a, b = gu_f32(e), dn_f32(e)
        if w.wfmt == "q8_0":
            gu[e] = oracle.q8_0_quantize(a)
            dn[e] = oracle.q8_0_quantize(b)
        else:
            gu[e], gts[e] = oracle.nvfp4_quantize(a)
            dn[e], dts[e] = oracle.nvfp4_quantize(b)
    act = oracle.ACT_SWIGLU if w.act == "swiglu" else oracle.ACT_RELU2
    fmt = oracle.W_Q8_0 if w.wfmt == "q8_0" else oracle.W_NVFP4
    return oracle.Layer(w.d, w.f, w.E, w.k, act, fmt, router_w, gu, dn,
                        gts if w.wfmt == "nvfp4" else None, dts if w.wfmt == "nvfp4" else None)


def assert_close(got: np.ndarray, ref: np.ndarray, tol: float = TOL, what: str = "out") -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.abs(got - ref).max())
    assert err <= tol * rms, f"{what}: max|err| {err:.3e} > {tol} * rms {rms:.3e} (ratio {err / rms:.2e})"
    return err / rms if rms > 0 else 0.0
