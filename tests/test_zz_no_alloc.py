"""moe_layer_forward_noalloc against moe_layer_forward, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device memory (they
are handed only input/output buffers and a stream, or must not allocate while serving
or during stream capture).  It must give the same results as the workspace entry point,
call after call, from its fixed in-library scratch.  This file is collected last so that
a run stopping at the first failure has already run everything else.
"""
import numpy as np
import pytest
import torch

from oracle_bridge import TOL
from quantized_routed_expert_softmax_gb300 import layers, native, synth

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_q8_swiglu": (synth.WORKLOADS["tiny"], [1, 16]),
    "small_nvfp4_relu2": (synth.Workload("noalloc_nvfp4_relu2", d=256, f=512, E=16, k=4, act="relu2", wfmt="nvfp4",
                                         x_dtype="bf16", layers=1, zero_fraction=0.925), [1, 7]),
}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_softmax_gb300 import build
    build.build()
    native.lib()


def _close(a: torch.Tensor, b: torch.Tensor) -> None:
    a, b = a.cpu().numpy().astype(np.float64), b.cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(b ** 2)))
    assert np.isfinite(a).all()
    assert float(np.abs(a - b).max()) <= TOL * rms


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_entry_point_twice(name):
    w, Ts = CASES[name]
    L = layers.build_layer(w, source="numpy")
    for T in Ts:
        x = synth.tokens_cuda(w, T, tag="noalloc")
        ref = L.forward(x)
        first = L.forward_noalloc(x)
        second = L.forward_noalloc(x)          # the scratch keeps the last call's contents
        torch.cuda.synchronize()
        _close(first, ref)
        _close(second, ref)
        # a different input right after must not see the previous call's state
        x2 = synth.tokens_cuda(w, T, tag="noalloc2")
        _close(L.forward_noalloc(x2), L.forward(x2))


def test_noalloc_rejects_problems_beyond_the_scratch():
    w = synth.WORKLOADS["tiny"]
    L = layers.build_layer(w, source="numpy")
    T = 1
    scratch = 16 * 1024 * 1024                       # MOE_NOALLOC_SCRATCH_BYTES
    while L.workspace_bytes(T) <= scratch:
        T *= 2
    x = torch.zeros((T, w.d), dtype=torch.float32, device="cuda")
    with pytest.raises(native.MoeError) as exc:
        L.forward_noalloc(x)
    assert exc.value.status == 4          # MOE_ERR_WORKSPACE
