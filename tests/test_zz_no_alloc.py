"""moe_layer_forward_noalloc against moe_layer_forward, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device memory: a plugin
that is handed only its input/output buffers and a stream by an engine that owns every
allocation, or a server that must not allocate once it is serving (an allocation can
synchronise the device, and none is allowed while a stream is being captured).  It runs
the same kernels as the workspace entry point on the same arguments, so its output must be
bit-identical to a call with a fresh workspace, call after call, whatever the previous call
on the shared in-library scratch was (another layer shape, another token count, a device
error).  This file is collected last so that a run stopping at the first failure has
already run everything else.
"""
import numpy as np
import pytest
import torch

from quantized_routed_expert_softmax_gb300 import layers, native, synth

pytestmark = pytest.mark.gpu

NV_SMALL = synth.Workload("noalloc_nvfp4_relu2", d=256, f=512, E=16, k=4, act="relu2", wfmt="nvfp4",
                          x_dtype="bf16", layers=1, zero_fraction=0.925)
# Layer shapes whose workspaces differ in every region after the control words: d = 256, 1024
# and the Gemma width 2816 (the fused combine's row-tile counters reach index d/32 - 1 = 87).
D256 = synth.WORKLOADS["tiny"]
D1024 = synth.Workload("noalloc_d1024", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16",
                       layers=1)
D2816 = synth.Workload("noalloc_d2816", d=2816, f=704, E=16, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16",
                       layers=1)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_softmax_gb300 import build
    build.build()
    native.lib()


@pytest.fixture(scope="module")
def built():
    return {w.name: layers.build_layer(w, source="numpy") for w in (D256, D1024, D2816, NV_SMALL)}


def _fresh(L, x, idx_in=None, w_in=None):
    """The workspace entry point on a freshly zeroed workspace."""
    ws = torch.zeros(L.workspace_bytes(x.shape[0]), dtype=torch.uint8, device="cuda")
    return L.forward(x, idx_in=idx_in, w_in=w_in, workspace=ws)


def _same_bits(a: torch.Tensor, b: torch.Tensor) -> None:
    a, b = a.cpu().numpy(), b.cpu().numpy()
    assert np.isfinite(a).all()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), float(np.abs(a - b).max())


@pytest.mark.parametrize("name,Ts", [(D256.name, [1, 16]), (NV_SMALL.name, [1, 7])])
def test_noalloc_equals_workspace_entry_point_twice(built, name, Ts):
    L = built[name]
    wl = D256 if name == D256.name else NV_SMALL
    for T in Ts:
        x = synth.tokens_cuda(wl, T, tag="noalloc")
        ref = _fresh(L, x)
        first = L.forward_noalloc(x)
        second = L.forward_noalloc(x)          # the scratch keeps the last call's contents
        _same_bits(first, ref)
        _same_bits(second, ref)
        # a different input right after must not see the previous call's state
        x2 = synth.tokens_cuda(wl, T, tag="noalloc2")
        _same_bits(L.forward_noalloc(x2), _fresh(L, x2))


def test_noalloc_layers_of_different_widths_share_the_scratch(built):
    # d = 256, 1024 and 2816 in turn, at 1 to 8 tokens (the fused combine's counters in use),
    # and both orders: each call's output must equal a fresh-workspace call bit for bit
    seq = [D256, D2816, D1024, D256, D1024, D2816, D256]
    for T in (1, 2, 5, 8):
        for i, wl in enumerate(seq):
            L = built[wl.name]
            x = synth.tokens_cuda(wl, T, tag=f"mix{i}")
            _same_bits(L.forward_noalloc(x), _fresh(L, x))
    assert native.MoELayer.noalloc_status() == 0


def test_noalloc_token_counts_in_any_order(built):
    L = built[D256.name]
    x = synth.tokens_cuda(D256, 16, tag="order")
    ref16 = _fresh(L, x)
    ref1 = _fresh(L, x[:1].contiguous())
    for _ in range(2):
        _same_bits(L.forward_noalloc(x), ref16)
        _same_bits(L.forward_noalloc(x[:1].contiguous()), ref1)


def test_noalloc_status_reports_a_clamped_expert(built):
    L = built[D256.name]
    x = synth.tokens_cuda(D256, 4, tag="bad")
    idx = torch.tensor([[0, 1], [2, 999], [3, -5], [4, 5]], dtype=torch.int32, device="cuda")
    wts = torch.full((4, 2), 0.5, dtype=torch.float32, device="cuda")
    out = L.forward_noalloc(x, idx_in=idx, w_in=wts)
    assert native.MoELayer.noalloc_status() == 1
    assert native.MoELayer.noalloc_status() == 0       # reading clears the word
    _same_bits(out, _fresh(L, x, idx_in=idx, w_in=wts))
    # the next call starts clean
    _same_bits(L.forward_noalloc(x), _fresh(L, x))
    assert native.MoELayer.noalloc_status() == 0


def test_noalloc_rejects_problems_beyond_the_scratch(built):
    L = built[D256.name]
    T = 1
    scratch = 16 * 1024 * 1024                       # MOE_NOALLOC_SCRATCH_BYTES
    while L.workspace_bytes(T) <= scratch:
        T *= 2
    x = torch.zeros((T, D256.d), dtype=torch.float32, device="cuda")
    with pytest.raises(native.MoeError) as exc:
        L.forward_noalloc(x)
    assert exc.value.status == 4          # MOE_ERR_WORKSPACE
