"""Host-resident expert weights read in place (MOE_FLAG_HOST_WEIGHTS), through the C ABI.

"Running NVIDIA's new 120B Nemotron-3.5-Super on an 8GB GPU" keeps the experts in host RAM
and reads the down projection over the bus in place, only its active 16-neuron groups ("How
the engine works", step 4).  On GB300 the host memory is the Grace memory behind NVLink-C2C:
the expert stacks sit in page-locked host memory and the weight-streaming kernels load them
directly.  The arithmetic is unchanged, so every result must be bitwise the one of the same
weights in device memory (whose oracle parity the other tests establish); the tensor-core
path, which loads by TMA, is refused, and memory the device cannot address is rejected before
anything is launched."""
import numpy as np
import pytest
import torch

from oracle_bridge import assert_close, oracle_layer
from quantized_routed_expert_softmax_gb300 import layers, native, synth

pytestmark = pytest.mark.gpu

Q8 = synth.Workload("hw_q8", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=3)
NV = synth.Workload("hw_nv", d=512, f=256, E=32, k=6, act="relu2", wfmt="nvfp4", x_dtype="bf16", layers=1,
                    zero_fraction=0.925)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_softmax_gb300 import build
    build.build()
    native.lib()


def _bits(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("where", ["all", "down"])
@pytest.mark.parametrize("wl,T", [(Q8, 1), (Q8, 16), (NV, 1), (NV, 32)])
def test_host_weights_equal_device_weights(wl, T, where):
    dev = layers.build_layer(wl, source="numpy")
    host = layers.build_layer(wl, source="numpy", host_weights=where)
    assert not host.down.is_cuda and host.down.is_pinned()
    assert host.gate_up.is_cuda == (where == "down")
    assert host.launches(T) == dev.launches(T)
    x = synth.tokens_cuda(wl, T, tag="hostw")
    tr = {}
    out = host.forward(x, trace=tr)
    assert np.array_equal(_bits(out), _bits(dev.forward(x)))
    assert host.device_status() == 0
    if T == 1:   # and against the oracle directly
        ol = oracle_layer(wl, synth.router_weight(wl), lambda e: synth.expert_weights(wl, 0, e)[0],
                          lambda e: synth.expert_weights(wl, 0, e)[1], range(wl.E))
        xs = x.cpu().view(torch.int16).numpy().view(np.uint16)
        ref = ol.forward(xs)
        assert np.array_equal(tr["idx"].cpu().numpy(), ref["idx"])
        assert_close(out.cpu().numpy(), ref["out"])


def test_host_weights_stack_is_one_kernel_and_bitwise_equal():
    dev = native.MoEStack([layers.build_layer(Q8, layer=l, source="numpy") for l in range(Q8.layers)])
    host = native.MoEStack([layers.build_layer(Q8, layer=l, source="numpy", host_weights="all")
                            for l in range(Q8.layers)])
    assert host.launches() == dev.launches() == 1
    x = synth.tokens_cuda(Q8, 1, tag="hostw_stack")
    assert np.array_equal(_bits(host.forward(x)), _bits(dev.forward(x)))


def test_host_weights_refuse_the_tensor_core_path_and_unmapped_memory():
    L = layers.build_layer(NV, source="numpy", host_weights="all")
    x = synth.tokens_cuda(NV, 64, tag="hostw_gemm")
    L.set_path("gemm")
    with pytest.raises(native.MoeError) as exc:   # refused by the descriptor check, before the workspace
        L.forward(x, workspace=torch.zeros(256, dtype=torch.uint8, device="cuda"))
    assert exc.value.status == 5          # MOE_ERR_UNSUPPORTED
    L.set_path("auto")                    # AUTO keeps host weights on the weight-streaming kernels
    ref = layers.build_layer(NV, source="numpy", path="gemv").forward(x)
    assert np.array_equal(_bits(L.forward(x)), _bits(ref))
    # pageable host memory is not addressable by the device: rejected before any launch
    pageable = torch.empty(L.gate_up.shape, dtype=torch.uint8)
    pageable.copy_(L.gate_up)
    bad = native.MoELayer(NV.d, NV.f, NV.E, NV.k, NV.act, NV.wfmt, L.router_w, pageable, L.down,
                          L.gate_up_tscale, L.down_tscale, host_weights="all")
    with pytest.raises(native.MoeError) as exc:
        bad.forward(x)
    assert exc.value.status == 1          # MOE_ERR_INVALID_ARG
    # device memory flagged as host memory is rejected too
    bad = native.MoELayer(NV.d, NV.f, NV.E, NV.k, NV.act, NV.wfmt, L.router_w, L.gate_up.cuda(), L.down.cuda(),
                          L.gate_up_tscale, L.down_tscale, host_weights="down")
    with pytest.raises(native.MoeError) as exc:
        bad.forward(x)
    assert exc.value.status == 1          # MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("where", ["all", "down"])
def test_nemotron_layer_full_size_from_host_memory(where):
    w = synth.WORKLOADS["nemotron"]
    host = layers.build_layer(w, host_weights=where)
    dev_gu, dev_dn = host.gate_up.cuda(), host.down.cuda()
    dev = native.MoELayer(w.d, w.f, w.E, w.k, w.act, w.wfmt, host.router_w, dev_gu, dev_dn, host.gate_up_tscale,
                          host.down_tscale)
    for T in (1, 32):
        x = synth.tokens_cuda(w, T, tag="hostw_full")
        assert np.array_equal(_bits(host.forward(x)), _bits(dev.forward(x)))
