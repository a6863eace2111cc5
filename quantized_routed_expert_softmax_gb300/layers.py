"""Assemble device-resident layers of a workload from the seeded generator.

Weights are drawn as fp32 (on the device for the large shapes), packed by libmoe's own
packers into the layouts moe_layer_forward reads, and the fp32 copies are dropped.
"""
from __future__ import annotations

import torch

from . import native, synth


def build_layer(w: synth.Workload, layer: int = 0, source: str = "cuda", keep_fp32: bool = False,
                path: str = "auto", E_chunk: int = 16, act_quant: str = "none", host_weights: str = "none"):
    """A native.MoELayer for `w`, layer `layer`.

    source = "cuda": fp32 weights drawn on the device, E_chunk experts at a time;
    source = "numpy": drawn on the host with the numpy generator (small shapes), the
    same numbers the oracle tests draw.  keep_fp32 keeps the fp32 stacks on the layer
    (attributes gate_up_f32 / down_f32) for tests that hand them to the oracle.  act_quant
    "q8_0" selects the activation-quantised expert path (Q8_0 weights only).  host_weights "down"
    moves the packed down stack, "all" both stacks, to page-locked host memory that the kernels
    read in place.
    """
    dev = torch.device("cuda")
    router_w = torch.from_numpy(synth.router_weight(w, layer)).to(dev)
    rows = w.rows_gu
    if w.wfmt == "q8_0":
        gu = torch.empty((w.E, native.q8_0_bytes(rows, w.d)), dtype=torch.uint8, device=dev)
        dn = torch.empty((w.E, native.q8_0_bytes(w.d, w.f)), dtype=torch.uint8, device=dev)
    elif w.wfmt == "int8pc":
        gu = torch.empty((w.E, native.int8pc_bytes(rows, w.d)), dtype=torch.uint8, device=dev)
        dn = torch.empty((w.E, native.int8pc_bytes(w.d, w.f)), dtype=torch.uint8, device=dev)
    else:
        gu = torch.empty((w.E, native.nvfp4_bytes(rows, w.d)), dtype=torch.uint8, device=dev)
        dn = torch.empty((w.E, native.nvfp4_bytes(w.d, w.f)), dtype=torch.uint8, device=dev)
    gts = torch.empty(w.E, dtype=torch.float32, device=dev) if w.wfmt == "nvfp4" else None
    dts = torch.empty(w.E, dtype=torch.float32, device=dev) if w.wfmt == "nvfp4" else None
    keep_gu, keep_dn = [], []
    for e0 in range(0, w.E, E_chunk):
        ex = range(e0, min(w.E, e0 + E_chunk))
        if source == "cuda":
            a = synth.expert_stack_cuda(w, layer, "gate_up", ex)
            b = synth.expert_stack_cuda(w, layer, "down", ex)
        else:
            pairs = [synth.expert_weights(w, layer, e) for e in ex]
            a = torch.from_numpy(__import__("numpy").stack([p[0] for p in pairs])).to(dev)
            b = torch.from_numpy(__import__("numpy").stack([p[1] for p in pairs])).to(dev)
        sl = slice(ex.start, ex.stop)
        if w.wfmt == "q8_0":
            native.quantize_q8_0(a, "device", out=gu[sl])
            native.quantize_q8_0(b, "device", out=dn[sl])
        elif w.wfmt == "int8pc":
            native.quantize_int8pc(a, "device", out=gu[sl])
            native.quantize_int8pc(b, "device", out=dn[sl])
        else:
            native.pack_nvfp4(a, "device", out=gu[sl], tscale=gts[sl])
            native.pack_nvfp4(b, "neuron", out=dn[sl], tscale=dts[sl])
        if keep_fp32:
            keep_gu.append(a)
            keep_dn.append(b)
        else:
            del a, b
    def to_host(t):   # packed on the device, then moved to page-locked host memory
        h = torch.empty(t.shape, dtype=torch.uint8, pin_memory=True)
        h.copy_(t)
        return h
    if host_weights in ("down", "all"):
        dn = to_host(dn)
    if host_weights == "all":
        gu = to_host(gu)
    layer_obj = native.MoELayer(w.d, w.f, w.E, w.k, w.act, w.wfmt, router_w, gu, dn, gts, dts, path=path,
                                act_quant=act_quant, host_weights=host_weights)
    if keep_fp32:
        layer_obj.gate_up_f32 = torch.cat(keep_gu)
        layer_obj.down_f32 = torch.cat(keep_dn)
    return layer_obj
