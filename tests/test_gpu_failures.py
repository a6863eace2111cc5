"""Device-side failure detection, made to happen without faulting or hanging the GPU.

Every wait in libmoe's kernels is bounded.  The one-kernel decode layer's grid barriers
normally wait at most a second; a test can shorten that limit through the workspace header
(the int64 at byte 32, in ns) and make every barrier wait run out by setting the barrier's
arrival counter (the int32 at byte 16) to a value its targets never reach.  The kernel must
then record device error 2, give up waiting for the rest of the launch (it raises the counter
past every target, so no later barrier waits), leave its counters zero for the next call, and
return within the limit; the next call on the same workspace must give the normal result bit
for bit.  Error 3 (an activation beyond the f16
range of the tensor-core operands) needs no wait at all: a host-made input of 1e5 on the
GEMM path triggers it.  The pages have no counterpart to these checks: they guard the GPU
and the caller, not the method.
"""
import time

import numpy as np
import pytest
import torch

from quantized_routed_expert_softmax_gb300 import layers, native, synth

pytestmark = pytest.mark.gpu

BAR_WORD = 4        # int32 index of the one-kernel layer's barrier arrival counter (byte 16)
DONE_WORD = 5       # ... and of its finished-CTA counter
LIMIT_QWORD = 4     # int64 index of the barrier wait limit (byte 32)
UNREACHABLE = -(1 << 30)

Q8 = synth.Workload("fail_q8", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=3)
NV = synth.Workload("fail_nv", d=512, f=256, E=32, k=6, act="relu2", wfmt="nvfp4", x_dtype="bf16", layers=1,
                    zero_fraction=0.925)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_softmax_gb300 import build
    build.build()
    native.lib()


def _poison(ws: torch.Tensor, limit_ns: int) -> None:
    ws.view(torch.int32)[BAR_WORD] = UNREACHABLE
    ws.view(torch.int64)[LIMIT_QWORD] = limit_ns
    torch.cuda.synchronize()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("wl", [Q8, NV], ids=["q8_swiglu", "nvfp4_relu2"])
def test_grid_barrier_timeout_stops_the_layer_and_reports_error_2(wl):
    L = layers.build_layer(wl, source="numpy")
    assert L.launches(1) == 1                           # the one-kernel layer
    x = synth.tokens_cuda(wl, 1, tag="fail")
    ws = torch.zeros(L.workspace_bytes(1), dtype=torch.uint8, device="cuda")
    ref = L.forward(x, workspace=ws).clone()
    assert native.device_status(ws) == 0
    _poison(ws, 100_000)                                # 100 us per wait
    out = torch.full((1, wl.d), float("nan"), device="cuda")
    t0 = time.perf_counter()
    L.forward(x, out=out, workspace=ws)
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert native.device_status(ws) == 2
    assert took < 0.5, took                             # the short limit, not the default second
    # the counters are zero again, so the workspace serves the next call as it is
    assert int(ws.view(torch.int32)[BAR_WORD]) == 0 and int(ws.view(torch.int32)[DONE_WORD]) == 0
    ws.view(torch.int64)[LIMIT_QWORD] = 0
    again = L.forward(x, workspace=ws)
    assert np.array_equal(_bits(again), _bits(ref))
    assert native.device_status(ws) == 0


def test_grid_barrier_timeout_in_a_stack():
    stack = native.MoEStack([layers.build_layer(Q8, layer=l, source="numpy") for l in range(Q8.layers)])
    assert stack.launches() == 1
    x = synth.tokens_cuda(Q8, 1, tag="fail_stack")
    ws = stack.workspace()
    ref = stack.forward(x).clone()
    _poison(ws, 100_000)
    stack.forward(x)
    assert native.device_status(ws) == 2
    ws.view(torch.int64)[LIMIT_QWORD] = 0
    assert np.array_equal(_bits(stack.forward(x)), _bits(ref))
    assert native.device_status(ws) == 0


def test_activation_beyond_f16_range_reports_error_3():
    wl = synth.WORKLOADS["tiny"]
    L = layers.build_layer(wl, source="numpy", path="gemm")
    x = synth.tokens_cuda(wl, 64, tag="range")
    ws = L.workspace(64)
    L.forward(x, workspace=ws)
    assert native.device_status(ws) == 0
    bad = x.clone()
    bad[3, 5] = 1e5                                     # beyond +-65504
    L.forward(bad, workspace=ws)
    assert native.device_status(ws) == 3
    assert native.device_status(ws) == 0                # reading clears the word
    L.forward(x, workspace=ws)
    assert native.device_status(ws) == 0
