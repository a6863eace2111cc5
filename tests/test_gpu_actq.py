"""The activation-quantised Q8_0 expert path (MOE_ACTQ_Q8_0) against the oracle, through the C ABI.

The CPU engines of "Running Gemma 4 26B at 5 tokens/s on a 13-year-old Xeon without a GPU"
(sections "A three-step fix" and "Narrowing down the cause") quantise every expert input to
Q8_0 blocks and take Q8_0 x Q8_0 block dots.  The oracle's orc_layer_forward_ex(act_q8) is that
path: each block's 32 code products summed as integers, times both fp16 scales, in fp64.
Bit-exact here: the activation codes (as the values they stand for) against the oracle's Q8_0
codec, and routing.  The coded h the down projection reads is a rounding decision on an fp32
h the two sides accumulate in different orders, so it may differ by one code step; the
outputs are checked against the oracle's down and combine on the GPU's own coded h (2e-3 *
rms) and end to end within 2e-3 * rms plus what the differing codes can move
(oracle_bridge.check_act_quant).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle_bridge import assert_close, check_act_quant, coded_q8_0, oracle_layer, to_numpy_x
from quantized_routed_expert_softmax_gb300 import layers, native, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_softmax_gb300 import build
    build.build()
    native.lib()


def _edge_rows(cols, seed):
    g = np.random.default_rng(seed)
    m = (g.standard_normal((6, cols)) * 3).astype(np.float32)
    m[0, :32] = 0.0                                        # an all-zero block
    m[1, :32] = -0.3                                       # a constant block
    m[2, :8] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, 126.5, -0.49]
    m[3, :3] = [1.0, 0.49997, -0.49997]                    # the fp32 scale decides, not the fp16 one
    m[4, :64] *= 1e4
    m[5, :64] *= 1e-30
    return m


@pytest.mark.parametrize("cols", [256, 2816, 3072])
def test_activation_codes_bitexact(cols):
    x = np.concatenate([_edge_rows(cols, cols), np.random.default_rng(1).standard_normal((37, cols)).astype(np.float32)])
    got = native.quantize_act_q8_0(torch.from_numpy(x).cuda()).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), coded_q8_0(x).view(np.uint32))
    # bf16 activations are coded from their exact fp32 values
    xb = torch.from_numpy(x).cuda().to(torch.bfloat16)
    got_b = native.quantize_act_q8_0(xb).cpu().numpy()
    assert np.array_equal(got_b.view(np.uint32), coded_q8_0(xb.float().cpu().numpy()).view(np.uint32))


SMALL = {
    "tiny_q8_swiglu": synth.WORKLOADS["tiny"],
    "small_q8_relu2": synth.Workload("aq_q8_relu2", d=512, f=256, E=12, k=3, act="relu2", wfmt="q8_0",
                                     x_dtype="bf16", layers=1, zero_fraction=0.8),
    "k8_e64": synth.Workload("aq_k8", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=1),
}


def _run(w, T, path):
    L = layers.build_layer(w, source="numpy", path=path, act_quant="q8_0")
    x = synth.tokens(w, T, tag="actq")
    xt = torch.from_numpy(x).cuda()
    if x.dtype == np.uint16:
        xt = xt.view(torch.bfloat16)
    tr = {}
    out = L.forward(xt, trace=tr).cpu().numpy()
    ol = oracle_layer(w, synth.router_weight(w), lambda e: synth.expert_weights(w, 0, e)[0],
                      lambda e: synth.expert_weights(w, 0, e)[1], range(w.E))
    ref = ol.forward(x, act_q8=True)
    return L, xt, out, tr, ref, ol


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("T,path", [(1, "auto"), (3, "auto"), (16, "auto"), (100, "auto"), (300, "gemm")])
def test_layer_activation_quantised_parity(name, T, path):
    w = SMALL[name]
    L, xt, out, tr, ref, ol = _run(w, T, path)
    assert np.array_equal(tr["idx"].cpu().numpy(), ref["idx"])
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert np.allclose(tr["w"].cpu().numpy(), ref["w"], rtol=1e-6, atol=0)
    check_act_quant(w, ol, np.arange(T), out, tr, ref)
    # deterministic: a second call is bit-identical
    assert np.array_equal(L.forward(xt).cpu().numpy().view(np.uint32), out.view(np.uint32))
    if T == 1 and path == "auto" and w.act == "swiglu":
        assert L.launches(T) == 1   # the one-kernel layer codes x and h itself
    else:   # two more launches than the unquantised path on the same kernels
        plain = native.MoELayer(w.d, w.f, w.E, w.k, w.act, w.wfmt, L.router_w, L.gate_up, L.down,
                                path="gemv" if (T == 1 and path == "auto") else path)
        assert L.launches(T) == plain.launches(T) + 2


def test_activation_quantised_differs_from_plain():
    # the coded path is a different numeric contract: both match their own oracle, not each other
    w = SMALL["k8_e64"]
    L, xt, out, tr, ref, ol = _run(w, 4, "auto")
    plain = ol.forward(synth.tokens(w, 4, tag="actq"))["out"]
    rms = float(np.sqrt(np.mean(plain ** 2)))
    assert float(np.abs(ref["out"] - plain).max()) > 2e-3 * rms
    check_act_quant(w, ol, np.arange(4), out, tr, ref)


def test_activation_quantised_noalloc_and_stack():
    w = SMALL["k8_e64"]
    L = layers.build_layer(w, source="numpy", act_quant="q8_0")
    x = synth.tokens_cuda(w, 1, tag="actq1")
    a = L.forward(x)
    assert np.array_equal(L.forward_noalloc(x).cpu().numpy().view(np.uint32), a.cpu().numpy().view(np.uint32))
    st = native.MoEStack([L])
    assert st.launches() == 1                   # the one-kernel layer codes x and h itself
    assert np.array_equal(st.forward(x).cpu().numpy().view(np.uint32), a.cpu().numpy().view(np.uint32))
    # the separate kernels on the same layer: the same codes and routing, outputs within tolerance
    tr1, tr2 = {}, {}
    a1 = L.forward(x, trace=tr1).cpu().numpy()
    L.set_path("gemv")
    assert L.launches(1) > 1
    a2 = L.forward(x, trace=tr2).cpu().numpy()
    assert np.array_equal(tr1["idx"].cpu().numpy(), tr2["idx"].cpu().numpy())
    assert_close(a1, a2.astype(np.float64), what="one kernel vs separate kernels")


# A stack of coded layers as one kernel: bitwise equal to its layers glued by the stand-alone
# RMS-norm, each layer against the oracle's coded path on its own input.  A stack whose layers
# code differently runs layer by layer.
def test_activation_quantised_stack_one_kernel():
    w = synth.Workload("aq_st", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=3)
    n = 3
    ls = [layers.build_layer(w, layer=l, source="numpy", act_quant="q8_0") for l in range(n)]
    st = native.MoEStack(ls)
    assert st.launches(True) == 1
    x0 = synth.tokens_cuda(w, 1, tag="aq_stack")
    xn = torch.zeros((n, w.d), dtype=torch.bfloat16, device="cuda")
    outs = torch.full((n, w.d), float("nan"), device="cuda")
    routing = {}
    st.forward(x0, outs=outs, x_next=xn, routing=routing)
    x = x0
    for l, L in enumerate(ls):
        tr = {}
        o = L.forward(x, trace=tr)
        assert np.array_equal(o.cpu().numpy().view(np.uint32), outs[l:l + 1].cpu().numpy().view(np.uint32)), l
        assert np.array_equal(tr["idx"].cpu().numpy(), routing["idx"][l:l + 1].cpu().numpy())
        ol = oracle_layer(w, synth.router_weight(w, l), lambda e, l=l: synth.expert_weights(w, l, e)[0],
                          lambda e, l=l: synth.expert_weights(w, l, e)[1], range(w.E))
        ref = ol.forward(to_numpy_x(x), act_q8=True)
        assert np.array_equal(tr["idx"].cpu().numpy(), ref["idx"])
        check_act_quant(w, ol, np.arange(1), o.cpu().numpy(), tr, ref)
        x = native.rmsnorm_bf16(o)
        assert torch.equal(x.view(torch.int16), xn[l:l + 1].view(torch.int16)), l
    assert torch.equal(st.forward(x0).view(torch.int32), outs.view(torch.int32))
    # mixed: the first layer coded, the others not
    plain = [layers.build_layer(w, layer=l, source="numpy") for l in range(1, n)]
    mixed = native.MoEStack([ls[0]] + plain)
    assert mixed.launches(True) == 1 + 1 + 2 * 2   # one kernel per layer, a norm after each
    mo = torch.full((n, w.d), float("nan"), device="cuda")
    mixed.forward(x0, outs=mo)
    x = x0
    for l, L in enumerate([ls[0]] + plain):
        o = L.forward(x)
        assert np.array_equal(o.cpu().numpy().view(np.uint32), mo[l:l + 1].cpu().numpy().view(np.uint32)), l
        x = native.rmsnorm_bf16(o)


@pytest.mark.parametrize("name,T,tile", [("gemma", 1, None), ("gemma", 4, None), ("minimax", 4096, 64)])
def test_activation_quantised_full_size(name, T, tile):
    from test_gpu_parity import _full_case
    _full_case(name, T, tile=tile, act_quant="q8_0")
