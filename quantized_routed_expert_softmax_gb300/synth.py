"""Seeded synthetic inputs for the routed MoE layer.

This module only draws numbers and shapes them (sizes, value distributions, the bias
channel that makes the latent experts sparse, Zipf routing); it holds none of the
layer's arithmetic, and it is the one piece that both the CUDA path and the CPU oracle
consume.  Every tensor has its own seed derived from (workload, layer, tensor, expert)
so any slice can be regenerated on its own.

Workload shapes follow the models the pages run:
  tiny      d=256,  E=8,   k=2,  f=512,  SwiGLU, Q8_0, x fp32 N(0,1)
  gemma     d=2816, E=128, k=8,  f=704,  SwiGLU, Q8_0, 30 layers (Gemma-4-26B-A4B:
            "Running Gemma 4 26B at 5 tokens/s on a 13-year-old Xeon", and the
            Inferentia page, "Wall 1": 128 experts, top-8, 30 layers)
  nemotron  d=1024, E=512, k=22, f=2688, ReLU^2 gateless, NVFP4, 40 layers, ~92.5 % of
            neurons zero after ReLU^2 (Nemotron page, "bytes per token" and step 4)
  minimax   d=6144, E=128, k=4,  f=3072, SwiGLU, Q8_0, 8 resident layers (MiniMax-M3:
            "Why can super-large MoE be distributed for inference", section 1)
  zipf      the gemma shape with Zipf(s=1.1) routing supplied by the caller
  gemma_int8pc  the gemma shape with per-channel int8 experts
"""
from __future__ import annotations

import statistics
import zlib
from dataclasses import dataclass, field

import numpy as np

BASE_SEED = 0


@dataclass(frozen=True)
class Workload:
    name: str
    d: int
    f: int
    E: int
    k: int
    act: str            # "swiglu" | "relu2"
    wfmt: str           # "q8_0" | "nvfp4"
    x_dtype: str        # "f32" | "bf16"
    layers: int
    tokens: tuple = ()
    rms_norm_input: bool = True
    zero_fraction: float | None = None   # target fraction of exact zeros after ReLU^2
    router_std: float = 0.05
    weight_std: float = 0.02
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def rows_gu(self) -> int:
        return 2 * self.f if self.act == "swiglu" else self.f


WORKLOADS = {
    "tiny": Workload("tiny", d=256, f=512, E=8, k=2, act="swiglu", wfmt="q8_0", x_dtype="f32", layers=1,
                     tokens=(16,), rms_norm_input=False),
    "gemma": Workload("gemma", d=2816, f=704, E=128, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=30,
                      tokens=(1, 4, 512)),
    "nemotron": Workload("nemotron", d=1024, f=2688, E=512, k=22, act="relu2", wfmt="nvfp4", x_dtype="bf16",
                         layers=40, tokens=(1, 32), zero_fraction=0.925),
    "minimax": Workload("minimax", d=6144, f=3072, E=128, k=4, act="swiglu", wfmt="q8_0", x_dtype="bf16",
                        layers=8, tokens=(1, 8, 4096)),
    "zipf": Workload("zipf", d=2816, f=704, E=128, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=1,
                     tokens=(1, 8, 64, 512, 2048, 8192)),
    "zipf_nvfp4": Workload("zipf_nvfp4", d=2816, f=704, E=128, k=8, act="swiglu", wfmt="nvfp4", x_dtype="bf16",
                           layers=1, tokens=(1, 8, 64, 512, 2048, 8192)),
    # the Gemma layer shape with per-channel int8 experts (Inferentia page, "Wall 1": about
    # 11.4 GB of int8 experts per rank of two)
    "gemma_int8pc": Workload("gemma_int8pc", d=2816, f=704, E=128, k=8, act="swiglu", wfmt="int8pc", x_dtype="bf16",
                             layers=30, tokens=(1, 4, 64)),
}


def sub_seed(*parts) -> int:
    """A stable 63-bit seed from BASE_SEED and the parts (workload, layer, tensor, expert)."""
    key = "/".join(str(p) for p in (BASE_SEED,) + parts).encode()
    return (zlib.crc32(key) << 31) ^ zlib.crc32(key[::-1])


def rng(*parts) -> np.random.Generator:
    return np.random.default_rng(sub_seed(*parts))


def bias_shift(w: Workload) -> float:
    """Magnitude of the bias weight that makes ~zero_fraction of the pre-activations
    negative.  Pre-activations are a sum of d-1 terms N(0, weight_std^2) * x with x of
    unit RMS, so they are ~N(0, weight_std^2 (d-1)); the bias channel x[0] = 1 with
    weight -beta moves the mean to -beta."""
    sigma = w.weight_std * float(np.sqrt(w.d - 1))
    return sigma * statistics.NormalDist().inv_cdf(w.zero_fraction)


# ----------------------------------------------------------------------------- CPU (numpy)
def router_weight(w: Workload, layer: int = 0) -> np.ndarray:
    """W [d, E] fp32 ~ N(0, router_std^2)."""
    g = rng(w.name, layer, "router")
    return (g.standard_normal((w.d, w.E), dtype=np.float32) * np.float32(w.router_std)).astype(np.float32)


def expert_weights(w: Workload, layer: int, expert: int) -> tuple[np.ndarray, np.ndarray]:
    """(gate_up [rows_gu, d], down [d, f]) fp32 ~ N(0, weight_std^2) for one expert.

    SwiGLU: rows 0..f-1 of gate_up are the gate, f..2f-1 the up projection (the fused
    [n_embd, 2 n_ff, n_experts] tensor, gate first).  With a zero-fraction target the
    bias weight -beta is written into column 0 of every row of the up projection."""
    g1 = rng(w.name, layer, "gate_up", expert)
    g2 = rng(w.name, layer, "down", expert)
    gu = g1.standard_normal((w.rows_gu, w.d), dtype=np.float32) * np.float32(w.weight_std)
    dn = g2.standard_normal((w.d, w.f), dtype=np.float32) * np.float32(w.weight_std)
    if w.zero_fraction is not None:
        up0 = w.f if w.act == "swiglu" else 0
        gu[up0:up0 + w.f, 0] = np.float32(-bias_shift(w))
    return gu.astype(np.float32), dn.astype(np.float32)


def tokens_f32(w: Workload, T: int, layer: int = 0, tag: str = "x") -> np.ndarray:
    """x [T, d] fp32 ~ N(0,1); RMS-normalised per token when the workload says so; the
    bias channel x[:, 0] = 1 when it has a zero-fraction target."""
    g = rng(w.name, layer, tag, T)
    x = g.standard_normal((T, w.d), dtype=np.float32)
    if w.rms_norm_input:
        x = x / np.sqrt(np.mean(x.astype(np.float64) ** 2, axis=1, keepdims=True) + 1e-6)
        x = x.astype(np.float32)
    if w.zero_fraction is not None:
        x[:, 0] = 1.0
    return x


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even, via torch's conversion) as uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def tokens(w: Workload, T: int, layer: int = 0, tag: str = "x") -> np.ndarray:
    """Layer input in the workload's activation type: fp32 array, or bf16 as uint16 bits."""
    x = tokens_f32(w, T, layer, tag)
    return x if w.x_dtype == "f32" else to_bf16_bits(x)


def zipf_routing(T: int, E: int, k: int, s: float = 1.1, seed_tag: str = "zipf") -> tuple[np.ndarray, np.ndarray]:
    """Precomputed routing: each token draws k distinct experts without replacement with
    probability proportional to rank^-s over a seeded permutation of the experts; the
    weights are a softmax of seeded N(0,1) scores (positive, summing to one)."""
    g = rng(seed_tag, T, E, k)
    order = g.permutation(E)
    p_rank = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    p = np.empty(E)
    p[order] = p_rank / p_rank.sum()
    idx = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        idx[t] = g.choice(E, size=k, replace=False, p=p)
    z = g.standard_normal((T, k))
    wts = np.exp(z - z.max(axis=1, keepdims=True))
    wts = (wts / wts.sum(axis=1, keepdims=True)).astype(np.float32)
    return idx, wts


# ----------------------------------------------------------------------------- GPU (torch)
def cuda_generator(*parts):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(sub_seed(*parts) & ((1 << 63) - 1))
    return g


def expert_stack_cuda(w: Workload, layer: int, which: str, experts: range | None = None):
    """A stack of expert matrices generated on the device (for full-size workloads whose
    fp32 weights do not fit the host comfortably): which = "gate_up" -> [n, rows_gu, d],
    "down" -> [n, d, f], fp32 ~ N(0, weight_std^2), one generator per expert."""
    import torch
    experts = range(w.E) if experts is None else experts
    shape = (w.rows_gu, w.d) if which == "gate_up" else (w.d, w.f)
    out = torch.empty((len(experts),) + shape, dtype=torch.float32, device="cuda")
    for i, e in enumerate(experts):
        g = cuda_generator(w.name, layer, which + "_cuda", e)
        out[i].normal_(0.0, w.weight_std, generator=g)
    if which == "gate_up" and w.zero_fraction is not None:
        up0 = w.f if w.act == "swiglu" else 0
        out[:, up0:up0 + w.f, 0] = -bias_shift(w)
    return out


def tokens_cuda(w: Workload, T: int, layer: int = 0, tag: str = "x"):
    """x [T, d] on the device in the workload's activation dtype (torch fp32 or bf16)."""
    import torch
    g = cuda_generator(w.name, layer, tag + "_cuda", T)
    x = torch.randn((T, w.d), generator=g, device="cuda", dtype=torch.float32)
    if w.rms_norm_input:
        x = x * torch.rsqrt(x.double().pow(2).mean(dim=1, keepdim=True) + 1e-6).float()
    if w.zero_fraction is not None:
        x[:, 0] = 1.0
    return x if w.x_dtype == "f32" else x.to(torch.bfloat16)
