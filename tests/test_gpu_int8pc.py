"""Per-channel int8 experts (MOE_W_INT8PC) against the oracle, through the C ABI.

"Squeezing a 26B MoE onto the cheapest Inferentia instance", section "Wall 1: the memory
math": the experts quantised to int8 with one scale per output channel.  Bit-exact here: the
packed bytes in both layouts against orc_int8pc_quantize (and the oracle's own device-layout
permutation), and routing.  Outputs and h: max|err| <= 2e-3 * rms against the oracle's
dequantise-then-fp64 layer.  The weight-streaming kernels read the codes as exact f16 and
apply each row's fp32 scale to every 32-column panel's product (the same sum up to fp32
rounding as scaling once at the end).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle_bridge import assert_close, oracle_layer
from quantized_routed_expert_softmax_gb300 import layers, native, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_softmax_gb300 import build
    build.build()
    native.lib()


def _edge_matrix(rows, cols, seed):
    g = np.random.default_rng(seed)
    m = (g.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    m[0] = 0.0                                        # an all-zero row: s = 0, codes 0
    m[1] = 0.3                                        # a constant row: codes 127
    m[2, :] = 0.0
    m[2, :8] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, 126.5, -0.49]   # s = 1: half-way values round away
    m[3] *= 1e4                                       # large values
    m[4] *= 1e-30                                     # tiny values (a subnormal scale)
    return m


@pytest.mark.parametrize("rows,cols", [(64, 256), (96, 2816), (2816, 704)])
def test_int8pc_packer_bitexact(rows, cols):
    mats = np.stack([_edge_matrix(rows, cols, s) for s in range(3)])
    src = torch.from_numpy(mats).cuda()
    got_c = native.quantize_int8pc(src, "canonical").cpu().numpy()
    got_d = native.quantize_int8pc(src, "device").cpu().numpy()
    for i in range(3):
        canon = oracle.int8pc_quantize(mats[i])
        assert np.array_equal(got_c[i], canon), (i, int((got_c[i] != canon).sum()))
        assert np.array_equal(got_d[i], oracle.int8pc_to_device(canon, rows, cols))


SMALL = {
    "tiny_int8pc": synth.Workload("pc_tiny", d=256, f=512, E=8, k=2, act="swiglu", wfmt="int8pc", x_dtype="f32",
                                  layers=1, rms_norm_input=False),
    "relu2_int8pc": synth.Workload("pc_relu2", d=512, f=256, E=12, k=3, act="relu2", wfmt="int8pc", x_dtype="bf16",
                                   layers=1, zero_fraction=0.8),
    "k8_e64_int8pc": synth.Workload("pc_k8", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="int8pc", x_dtype="bf16",
                                    layers=1),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("T", [1, 3, 16, 100])
def test_layer_int8pc_parity(name, T):
    w = SMALL[name]
    L = layers.build_layer(w, source="numpy")
    x = synth.tokens(w, T, tag="pc")
    xt = torch.from_numpy(x).cuda()
    if x.dtype == np.uint16:
        xt = xt.view(torch.bfloat16)
    tr = {}
    out = L.forward(xt, trace=tr).cpu().numpy()
    ol = oracle_layer(w, synth.router_weight(w), lambda e: synth.expert_weights(w, 0, e)[0],
                      lambda e: synth.expert_weights(w, 0, e)[1], range(w.E))
    ref = ol.forward(x)
    assert np.array_equal(tr["idx"].cpu().numpy(), ref["idx"])
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert np.allclose(tr["w"].cpu().numpy(), ref["w"], rtol=1e-6, atol=0)
    assert_close(tr["h"].cpu().numpy(), ref["h"][ref["perm"]], what="h")
    assert_close(out, ref["out"])
    # the packed bytes of one expert, as the oracle lays them out
    e = int(ref["idx"][0, 0])
    assert np.array_equal(L.gate_up[e].cpu().numpy(), oracle.int8pc_to_device(ol.gate_up[e], w.rows_gu, w.d))
    assert np.array_equal(L.down[e].cpu().numpy(), oracle.int8pc_to_device(ol.down[e], w.d, w.f))
    # bitwise deterministic, fully written
    o2 = torch.full((T, w.d), float("nan"), device="cuda")
    L.forward(xt, out=o2)
    assert np.array_equal(o2.cpu().numpy().view(np.uint32), out.view(np.uint32))


def test_int8pc_tensor_core_path_is_not_built():
    w = SMALL["tiny_int8pc"]
    L = layers.build_layer(w, source="numpy", path="gemm")
    with pytest.raises(native.MoeError) as exc:
        L.forward(torch.zeros((16, w.d), device="cuda"))
    assert exc.value.status == 5          # MOE_ERR_UNSUPPORTED
    L.set_path("auto")                    # AUTO keeps per-channel int8 on the weight-streaming kernels
    assert L.forward(torch.zeros((600, w.d), device="cuda")).abs().max().item() == 0.0


@pytest.mark.parametrize("T", [1, 4, 64])
def test_gemma_int8pc_full_size(T):
    from test_gpu_parity import _full_case
    _full_case("gemma_int8pc", T)
