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
        elif w.wfmt == "int8pc":
            gu[e] = oracle.int8pc_quantize(a)
            dn[e] = oracle.int8pc_quantize(b)
        else:
            gu[e], gts[e] = oracle.nvfp4_quantize(a)
            dn[e], dts[e] = oracle.nvfp4_quantize(b)
    act = oracle.ACT_SWIGLU if w.act == "swiglu" else oracle.ACT_RELU2
    fmt = {"q8_0": oracle.W_Q8_0, "nvfp4": oracle.W_NVFP4, "int8pc": oracle.W_INT8PC}[w.wfmt]
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


def coded_q8_0(x32: np.ndarray) -> np.ndarray:
    """The values the oracle's Q8_0 codes of each row stand for (exact in fp32)."""
    rows, cols = x32.shape
    return np.stack([oracle.q8_0_dequant(oracle.q8_0_quantize(x32[r:r + 1]), 1, cols)[0]
                     for r in range(rows)]).astype(np.float32)


def check_act_quant(w: synth.Workload, ol: oracle.Layer, rows, out: np.ndarray, tr: dict, ref: dict) -> None:
    """The activation-quantised path (orc_layer_forward_ex with act_q8) at the sampled tokens.

    The coded h that the down projection reads is a quantisation decision taken on an fp32 h
    that the two sides accumulate in different orders, so a code may differ by one step where
    h falls next to a rounding boundary.  Hence three checks:
      1. the GPU's coded h against the oracle's h coded by the oracle's codec: one code step at
         most per element, and below 5% of the elements differing at all;
      2. out against the oracle's down projection and combine applied to the GPU's own coded h
         (each block's code products are exact integers times both fp16 scales: the dense
         product of the dequantised weights with the coded h, in fp64): max|err| <= TOL * rms;
      3. out against the oracle's end-to-end out, within TOL * rms plus the most the differing
         codes can move it: sum over them of |w| * step * max |down column|."""
    k, f = w.k, w.f
    T_s = len(rows)
    pos = tr["pos"].cpu().numpy()
    h_dev = tr["h"].cpu().numpy()
    idx = ref["idx"]
    wts = ref["w"].astype(np.float64)
    h_gpu = np.stack([h_dev[pos[t * k + j]] for t in rows for j in range(k)])       # pair order
    h_orc = coded_q8_0(ref["h"].astype(np.float32))
    step = np.repeat(np.abs(ref["h"].astype(np.float32)).reshape(T_s * k, -1, 32).max(axis=2) / 127.0, 32, axis=1)
    diff = h_gpu != h_orc
    assert (np.abs(h_gpu - h_orc) <= 1.01 * step + 1e-30).all(), "coded h differs by more than one code step"
    # (a few percent at K = 6144 on the tensor cores, whose fp32 accumulation aligns each group
    # of products to its largest term; a systematic fault would move most codes)
    assert diff.mean() < 0.05, f"{diff.mean():.4f} of the coded h differ"
    chk = np.zeros((T_s, w.d))
    bound = np.zeros(T_s)
    for e in sorted(set(int(v) for v in idx.ravel())):
        Wd = oracle.q8_0_dequant(ol.down[e], w.d, f)                    # fp64 [d, f], exact
        colmax = np.abs(Wd).max(axis=0)
        for i in range(T_s):
            for j in range(k):
                if idx[i, j] != e:
                    continue
                p = i * k + j
                chk[i] += wts[i, j] * (Wd @ h_gpu[p].astype(np.float64))
                bound[i] += abs(wts[i, j]) * float((diff[p] * step[p] * colmax).sum())
    assert_close(out, chk, what="out vs the oracle's down and combine on the coded h")
    rms = float(np.sqrt(np.mean(ref["out"] ** 2)))
    err = np.abs(out.astype(np.float64) - ref["out"]).max(axis=1)
    assert (err <= TOL * rms + bound).all(), (float(err.max()), TOL * rms, float(bound.max()))
