"""GPU parity: libmoe's CUDA path against the CPU oracle, through the C ABI.

Bit-exact: quantised bytes (every layout), tensor scales, router logits, top-k indices,
expert offsets and the permutation.  Floating point: combine weights to 1e-6 relative,
layer outputs to max|err| <= 2e-3 * rms(out).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle_bridge import TOL, assert_close, check_act_quant, oracle_layer, to_numpy_x
from quantized_routed_expert_softmax_gb300 import layers, native, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_softmax_gb300 import build
    build.build()
    native.lib()


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _edge_matrix(rows, cols, seed):
    g = np.random.default_rng(seed)
    m = (g.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    m[0, :32] = 0.0                                    # an all-zero block
    m[1, :32] = 0.3                                    # a constant block
    m[2, :8] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, 126.5, -0.49]    # half-way codes
    m[3, :3] = [1.0, 0.49997, -0.49997]                # fp32-vs-fp16 scale sensitivity
    m[4, :64] = g.standard_normal(64).astype(np.float32) * 1e3      # large values
    m[5, :64] = g.standard_normal(64).astype(np.float32) * 1e-30    # tiny (subnormal scales)
    return m


# ------------------------------------------------------------------ packers
@pytest.mark.parametrize("rows,cols", [(64, 256), (96, 2816)])
def test_q8_0_packer_bitexact(rows, cols):
    mats = np.stack([_edge_matrix(rows, cols, s) for s in range(3)])
    canon = np.stack([oracle.q8_0_quantize(m) for m in mats])
    got_c = native.quantize_q8_0(_f32(mats), "canonical").cpu().numpy()
    got_d = native.quantize_q8_0(_f32(mats), "device").cpu().numpy()
    assert np.array_equal(got_c, canon)
    for i in range(3):
        assert np.array_equal(got_d[i], oracle.q8_0_to_device(canon[i], rows, cols))


@pytest.mark.parametrize("rows,cols", [(64, 256), (64, 2688), (2688, 1024)])
def test_nvfp4_packer_bitexact(rows, cols):
    g = np.random.default_rng(rows + cols)
    mats = [(g.standard_normal((rows, cols)) * 0.02).astype(np.float32) for _ in range(3)]
    mats[1] = _edge_matrix(rows, cols, 7)
    mats[2][:] = 0.0                                  # an all-zero matrix: s_t = 1
    src = _f32(np.stack(mats))
    ref = [oracle.nvfp4_quantize(m) for m in mats]
    for layout in ("canonical", "device", "neuron"):
        got, ts = native.pack_nvfp4(src, layout)
        got, ts = got.cpu().numpy(), ts.cpu().numpy()
        for i, (q, st) in enumerate(ref):
            assert ts[i] == np.float32(st)
            want = {"canonical": q, "device": oracle.nvfp4_to_panels(q, rows, cols),
                    "neuron": oracle.nvfp4_to_neuron(q, rows, cols)}[layout]
            assert np.array_equal(got[i], want), (layout, i, int((got[i] != want).sum()))


# ------------------------------------------------------------------ router
@pytest.mark.parametrize("name", ["tiny", "gemma", "nemotron"])
@pytest.mark.parametrize("T", [1, 3, 16, 37, 512, 4096])
def test_router_topk_bitexact(name, T):
    w = synth.WORKLOADS[name]
    x = synth.tokens(w, T, tag="router")
    W = synth.router_weight(w)
    xt = torch.from_numpy(x).cuda()
    if x.dtype == np.uint16:
        xt = xt.view(torch.bfloat16)
    idx, wt, lg = native.router_topk(xt, _f32(W), w.k, return_logits=True)
    ref_lg = oracle.router_logits(x, W)
    assert np.array_equal(lg.cpu().numpy().view(np.uint32), ref_lg.view(np.uint32))
    ref_idx, ref_w = oracle.topk_softmax(ref_lg, w.k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.allclose(wt.cpu().numpy(), ref_w, rtol=1e-6, atol=0)


def test_router_ties_take_lowest_index():
    w = synth.WORKLOADS["gemma"]
    x = torch.zeros((4, w.d), dtype=torch.bfloat16, device="cuda")
    idx, wt = native.router_topk(x, _f32(synth.router_weight(w)), w.k)
    assert (idx.cpu().numpy() == np.arange(w.k)).all()
    assert (wt.cpu().numpy() == np.float32(1.0 / w.k)).all()


# ------------------------------------------------------------------ the layer, small shapes
SMALL = {
    "tiny_q8_swiglu": synth.WORKLOADS["tiny"],
    "small_nvfp4_relu2": synth.Workload("small_nvfp4_relu2", d=256, f=512, E=16, k=4, act="relu2", wfmt="nvfp4",
                                        x_dtype="bf16", layers=1, zero_fraction=0.925),
    "small_q8_relu2": synth.Workload("small_q8_relu2", d=512, f=256, E=12, k=3, act="relu2", wfmt="q8_0",
                                     x_dtype="bf16", layers=1, zero_fraction=0.8),
    "small_nvfp4_swiglu": synth.Workload("small_nvfp4_swiglu", d=512, f=320, E=8, k=2, act="swiglu", wfmt="nvfp4",
                                         x_dtype="f32", layers=1),
}
# Many experts: up to 4096 logits the one-launch routing selects the top-k through segment
# candidates once E > 256 (T = 1, 3, 8 here); T = 16 goes through the separate kernels.
WIDE = synth.Workload("wide_e512", d=256, f=128, E=512, k=6, act="relu2", wfmt="q8_0", x_dtype="bf16", layers=1,
                      zero_fraction=0.8)


@pytest.mark.parametrize("T", [1, 3, 8, 16])
def test_layer_many_experts_parity(T):
    L, out, tr, ref = _run_small(WIDE, T)
    assert np.array_equal(tr["logits"].cpu().numpy().view(np.uint32), ref["logits"].view(np.uint32))
    assert np.array_equal(tr["idx"].cpu().numpy(), ref["idx"])
    assert np.allclose(tr["w"].cpu().numpy(), ref["w"], rtol=1e-6, atol=0)
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert_close(out, ref["out"])


def test_many_experts_ties_take_lowest_indices():
    # all logits equal (x = 0): the k lowest expert indices, uniform weights
    L = layers.build_layer(WIDE, source="numpy")
    x = torch.zeros((3, WIDE.d), dtype=torch.bfloat16, device="cuda")
    tr = {}
    L.forward(x, trace=tr)
    assert (tr["idx"].cpu().numpy() == np.arange(WIDE.k)).all()
    assert (tr["w"].cpu().numpy() == np.float32(1.0 / WIDE.k)).all()


def _run_small(w, T, idx_in=None, w_in=None, path="auto"):
    L = layers.build_layer(w, source="numpy", path=path)
    x = synth.tokens(w, T, tag="parity")
    xt = torch.from_numpy(x).cuda()
    if x.dtype == np.uint16:
        xt = xt.view(torch.bfloat16)
    tr = {}
    ii = None if idx_in is None else torch.from_numpy(idx_in).cuda()
    ww = None if w_in is None else torch.from_numpy(w_in).cuda()
    out = L.forward(xt, idx_in=ii, w_in=ww, trace=tr).cpu().numpy()
    ol = oracle_layer(w, synth.router_weight(w), lambda e: synth.expert_weights(w, 0, e)[0],
                      lambda e: synth.expert_weights(w, 0, e)[1], range(w.E))
    ref = ol.forward(x, idx_in=idx_in, w_in=w_in)
    return L, out, tr, ref


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("T", [1, 3, 16, 33, 100])
def test_layer_small_parity(name, T):
    w = SMALL[name]
    L, out, tr, ref = _run_small(w, T)
    assert np.array_equal(tr["idx"].cpu().numpy(), ref["idx"])
    assert np.allclose(tr["w"].cpu().numpy(), ref["w"], rtol=1e-6, atol=0)
    assert np.array_equal(tr["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(tr["pos"].cpu().numpy(), ref["pos"])
    assert np.array_equal(tr["logits"].cpu().numpy().view(np.uint32), ref["logits"].view(np.uint32))
    # activations in sorted-row order
    h_ref = ref["h"][ref["perm"]]
    assert_close(tr["h"].cpu().numpy(), h_ref, what="h")
    assert_close(out, ref["out"])


# NVFP4 down at two or more tokens, the GEMV path forced: on the tensor cores in passes of 8,
# 16 and 32 tokens with ragged last passes (T = 300 puts about 75 rows on each of the 8
# experts), ReLU^2 with 92.5% zeros (inactive groups skipped, uneven halves) and SwiGLU with 20
# groups; and the CUDA-core kernel for a wide f.
NV_DOWN = {
    "small_nvfp4_relu2": SMALL["small_nvfp4_relu2"],
    "small_nvfp4_swiglu": SMALL["small_nvfp4_swiglu"],
    # f = 2688: the h planes of 8 tokens would leave one CTA per SM, so the CUDA-core kernel
    # (2-token tiles) runs the down projection at every T here
    "wide_f_relu2": synth.Workload("nv_wide_f", d=256, f=2688, E=16, k=4, act="relu2", wfmt="nvfp4", x_dtype="bf16",
                                   layers=1, zero_fraction=0.925),
}


@pytest.mark.parametrize("name", list(NV_DOWN))
@pytest.mark.parametrize("T", [2, 9, 40, 300])
def test_nvfp4_down_tensor_core_parity(name, T):
    w = NV_DOWN[name]
    L, out, tr, ref = _run_small(w, T, path="gemv")
    assert np.array_equal(tr["idx"].cpu().numpy(), ref["idx"])
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert_close(tr["h"].cpu().numpy(), ref["h"][ref["perm"]], what="h")
    assert_close(out, ref["out"])


# The tensor-core GEMM path forced on the same layers: token tiles of 128 with ragged tails
# (T=700 puts about 175 rows on each expert of the 8-expert layers), fp32 inputs split hi/lo.
@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("T", [1, 16, 100, 700])
def test_layer_small_gemm_parity(name, T):
    w = SMALL[name]
    L, out, tr, ref = _run_small(w, T, path="gemm")
    assert np.array_equal(tr["idx"].cpu().numpy(), ref["idx"])
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert_close(tr["h"].cpu().numpy(), ref["h"][ref["perm"]], what="h")
    assert_close(out, ref["out"])
    # no atomics on this path either: a second call is bit-identical
    out2 = L.forward(torch.from_numpy(synth.tokens(w, T, tag="parity")).cuda().view(
        torch.bfloat16 if w.x_dtype == "bf16" else torch.float32)).cpu().numpy()
    assert np.array_equal(out.view(np.uint32), out2.view(np.uint32))


def test_layer_gemm_skewed_routing():
    # Zipf-skewed supplied routing: the hottest experts get several token tiles, some none
    w = SMALL["small_nvfp4_relu2"]
    T = 900
    idx, wts = synth.zipf_routing(T, w.E, w.k, seed_tag="gemm-skew")
    L, out, tr, ref = _run_small(w, T, idx_in=idx, w_in=wts, path="gemm")
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert np.bincount(idx.ravel(), minlength=w.E).max() > 2 * 128
    assert_close(out, ref["out"])


# One token, Q8_0 SwiGLU, k in {1, 2, 4, 8}: the down kernel owns 16 output rows for every
# routed expert and combines in place.  k = 1 gives eight warps per expert; a supplied routing
# that names one expert twice must take the general path (two rows in one slot).
@pytest.mark.parametrize("k", [1, 4])
def test_one_token_row_tile_down(k):
    w = synth.Workload(f"t1_k{k}", d=512, f=256, E=8, k=k, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=1)
    L, out, tr, ref = _run_small(w, 1, path="gemv")
    assert L.launches(1) == 3
    assert np.array_equal(tr["idx"].cpu().numpy(), ref["idx"])
    assert_close(out, ref["out"])


# One token, routing computed: the whole layer as one cooperative kernel (router, top-k,
# softmax, gate.up, down, combine; three grid barriers).  The shapes cover
# k = 1 .. 8, 22 and 32, E from 4 to 1024 (1024 experts: 8 per routing CTA), Q8_0 SwiGLU and NVFP4
# ReLU^2 with 80-92.5% zeros, fp32 and bf16 inputs,
# panel ranges that split items across warps and warps that span several items; every case
# is checked against the oracle and against the separate-kernel path, and the output must
# be completely written and bitwise identical over three calls.
ONE_KERNEL = {
    "tiny_f32": synth.WORKLOADS["tiny"],
    "k1": synth.Workload("ok_k1", d=512, f=256, E=8, k=1, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=1),
    "k8_e64": synth.Workload("ok_k8", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=1),
    "k3_e12_f32": synth.Workload("ok_k3", d=768, f=96, E=12, k=3, act="swiglu", wfmt="q8_0", x_dtype="f32",
                                 layers=1),
    "k32_e1024": synth.Workload("ok_k32", d=256, f=64, E=1024, k=32, act="swiglu", wfmt="q8_0", x_dtype="bf16",
                                layers=1),
    "e4_k4": synth.Workload("ok_e4", d=256, f=32, E=4, k=4, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=1),
    # NVFP4 ReLU^2 (gateless latent experts, neuron-contiguous down, all-zero groups skipped)
    "nv_k6_e32": synth.Workload("ok_nv6", d=512, f=256, E=32, k=6, act="relu2", wfmt="nvfp4", x_dtype="bf16",
                                layers=1, zero_fraction=0.925),
    "nv_k22_e512_f32": synth.Workload("ok_nv22", d=256, f=128, E=512, k=22, act="relu2", wfmt="nvfp4",
                                      x_dtype="f32", layers=1, zero_fraction=0.8),
    # NVFP4 SwiGLU (16-neuron gate + up items, every down group active, down prefetched)
    "nv_swiglu_k4": synth.Workload("ok_nvsw4", d=512, f=320, E=16, k=4, act="swiglu", wfmt="nvfp4",
                                   x_dtype="bf16", layers=1),
    "nv_swiglu_k8_f32": synth.Workload("ok_nvsw8", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="nvfp4",
                                       x_dtype="f32", layers=1),
    # per-channel int8 SwiGLU (the Q8_0 panels with one fp32 scale per row)
    "pc_k8_e64": synth.Workload("ok_pc8", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="int8pc", x_dtype="bf16",
                                layers=1),
    "pc_k3_e12_f32": synth.Workload("ok_pc3", d=768, f=96, E=12, k=3, act="swiglu", wfmt="int8pc", x_dtype="f32",
                                    layers=1),
    "pc_k22_e512": synth.Workload("ok_pc22", d=256, f=64, E=512, k=22, act="swiglu", wfmt="int8pc",
                                  x_dtype="bf16", layers=1),
}


@pytest.mark.parametrize("name", list(ONE_KERNEL))
def test_one_token_one_kernel(name):
    w = ONE_KERNEL[name]
    L, out, tr, ref = _run_small(w, 1)
    assert L.launches(1) == 1
    assert np.array_equal(tr["logits"].cpu().numpy().view(np.uint32), ref["logits"].view(np.uint32))
    assert np.array_equal(tr["idx"].cpu().numpy(), ref["idx"])
    assert np.allclose(tr["w"].cpu().numpy(), ref["w"], rtol=1e-6, atol=0)
    assert np.array_equal(tr["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(tr["pos"].cpu().numpy(), ref["pos"])
    assert_close(tr["h"].cpu().numpy(), ref["h"][ref["perm"]], what="h")
    assert_close(out, ref["out"])
    x = torch.from_numpy(synth.tokens(w, 1, tag="parity")).cuda()
    if w.x_dtype == "bf16":
        x = x.view(torch.bfloat16)
    outs = []
    for _ in range(3):
        o = torch.full((1, w.d), float("nan"), device="cuda")
        L.forward(x, out=o)
        outs.append(o.cpu().numpy())
    assert np.isfinite(outs[0]).all()
    for o in outs:
        assert np.array_equal(o.view(np.uint32), out.view(np.uint32))
    assert L.device_status() == 0
    L.set_path("gemv")
    assert L.launches(1) > 1
    assert_close(L.forward(x).cpu().numpy(), ref["out"])


# Supplied routing at one token: the same kernel without the router and the selection.  The
# trace copies idx and w exactly; the permutation follows them bit for bit; h and out agree
# with the oracle and with the separate kernels on the same routing.
@pytest.mark.parametrize("name", ["tiny_f32", "k1", "k8_e64", "k32_e1024", "nv_k6_e32", "nv_k22_e512_f32",
                                  "nv_swiglu_k4", "pc_k8_e64"])
def test_one_token_one_kernel_supplied_routing(name):
    w = ONE_KERNEL[name]
    idx, wts = synth.zipf_routing(1, w.E, w.k, seed_tag="one-kernel")
    L, out, tr, ref = _run_small(w, 1, idx_in=idx, w_in=wts)
    assert L.launches(1, routing_supplied=True) == 1
    assert np.array_equal(tr["idx"].cpu().numpy(), idx)
    assert np.array_equal(tr["w"].cpu().numpy().view(np.uint32), wts.view(np.uint32))
    assert np.array_equal(tr["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(tr["pos"].cpu().numpy(), ref["pos"])
    assert_close(tr["h"].cpu().numpy(), ref["h"][ref["perm"]], what="h")
    assert_close(out, ref["out"])
    assert L.device_status() == 0
    x = torch.from_numpy(synth.tokens(w, 1, tag="parity")).cuda()
    if w.x_dtype == "bf16":
        x = x.view(torch.bfloat16)
    ii, ww = torch.from_numpy(idx).cuda(), torch.from_numpy(wts).cuda()
    o = torch.full((1, w.d), float("nan"), device="cuda")
    L.forward(x, idx_in=ii, w_in=ww, out=o)
    assert np.array_equal(o.cpu().numpy().view(np.uint32), out.view(np.uint32))   # deterministic, fully written
    L.set_path("gemv")
    assert L.launches(1, routing_supplied=True) > 1
    assert_close(L.forward(x, idx_in=ii, w_in=ww).cpu().numpy(), ref["out"])


# An expert repeated in the supplied routing takes one slot per pair (pair order), and an index
# outside [0, E) is clamped and reported as device error 1, in the one-kernel layer as in the
# separate kernels.
def test_one_token_one_kernel_repeated_and_bad_experts():
    w = ONE_KERNEL["k8_e64"]
    rep = np.array([[5, 40, 5, 63, 0, 5, 17, 40]], dtype=np.int32)
    wts = np.array([[0.05, 0.1, 0.15, 0.2, 0.05, 0.25, 0.1, 0.1]], dtype=np.float32)
    L, out, tr, ref = _run_small(w, 1, idx_in=rep, w_in=wts)
    assert L.launches(1, routing_supplied=True) == 1
    assert np.array_equal(tr["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(tr["pos"].cpu().numpy(), ref["pos"])
    assert_close(tr["h"].cpu().numpy(), ref["h"][ref["perm"]], what="h")
    assert_close(out, ref["out"])
    assert L.device_status() == 0
    x = torch.from_numpy(synth.tokens(w, 1, tag="parity")).cuda().view(torch.bfloat16)
    bad = np.array([[5, 40, 5, 999, -7, 5, 17, 40]], dtype=np.int32)   # 999 -> 63, -7 -> 0
    o_bad = L.forward(x, idx_in=torch.from_numpy(bad).cuda(), w_in=torch.from_numpy(wts).cuda())
    assert L.device_status() == 1
    assert L.device_status() == 0
    assert np.array_equal(o_bad.cpu().numpy().view(np.uint32), out.view(np.uint32))


# One workspace serves calls of any token count in any order: its control words (the one-kernel
# layer's barrier counters among them) sit at offsets that do not depend on T, so a one-token
# call after a 16-token call (whose activations fill the bytes a one-token layout places later)
# starts from clean counters.
def test_one_workspace_serves_calls_of_any_token_count():
    w = SMALL["tiny_q8_swiglu"]
    L = layers.build_layer(w, source="numpy")
    x = torch.from_numpy(synth.tokens(w, 16, tag="mixed")).cuda()
    fresh16 = layers.build_layer(w, source="numpy").forward(x).cpu().numpy()
    fresh1 = layers.build_layer(w, source="numpy").forward(x[:1].contiguous()).cpu().numpy()
    assert L.launches(1) == 1
    ws = L.workspace(16)
    for _ in range(2):
        o16 = L.forward(x, workspace=ws).cpu().numpy()
        o1 = L.forward(x[:1].contiguous(), workspace=ws).cpu().numpy()
        assert np.array_equal(o16.view(np.uint32), fresh16.view(np.uint32))
        assert np.array_equal(o1.view(np.uint32), fresh1.view(np.uint32))
    assert L.device_status() == 0


def test_one_token_repeated_expert_in_supplied_routing():
    w = SMALL["tiny_q8_swiglu"]
    idx = np.array([[3, 3]], dtype=np.int32)
    wts = np.array([[0.25, 0.75]], dtype=np.float32)
    L, out, tr, ref = _run_small(w, 1, idx_in=idx, w_in=wts)
    assert_close(out, ref["out"])


@pytest.mark.parametrize("T", [5, 64])
def test_layer_supplied_routing(T):
    w = SMALL["tiny_q8_swiglu"]
    idx, wts = synth.zipf_routing(T, w.E, w.k, seed_tag="parity")
    L, out, tr, ref = _run_small(w, T, idx_in=idx, w_in=wts)
    assert np.array_equal(tr["perm"].cpu().numpy(), ref["perm"])
    assert_close(out, ref["out"])


def test_bad_expert_index_is_clamped_and_reported():
    w = SMALL["tiny_q8_swiglu"]
    L = layers.build_layer(w, source="numpy")
    x = torch.from_numpy(synth.tokens(w, 4, tag="bad")).cuda()
    idx = torch.tensor([[0, 1], [2, 999], [3, -5], [4, 5]], dtype=torch.int32, device="cuda")
    wts = torch.full((4, 2), 0.5, dtype=torch.float32, device="cuda")
    out = L.forward(x, idx_in=idx, w_in=wts)
    assert torch.isfinite(out).all()
    assert L.device_status() == 1
    assert L.device_status() == 0          # reading clears the word


def test_output_is_fully_written_and_deterministic():
    w = SMALL["small_nvfp4_relu2"]
    L = layers.build_layer(w, source="numpy")
    x = torch.from_numpy(synth.tokens(w, 33, tag="det")).cuda().view(torch.bfloat16)
    outs = []
    for _ in range(3):
        o = torch.full((33, w.d), float("nan"), device="cuda")
        L.forward(x, out=o)
        outs.append(o.cpu().numpy())
    assert np.isfinite(outs[0]).all()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(outs[0].view(np.uint32), outs[2].view(np.uint32))


def test_zero_input_gives_zero_output():
    for name in ("tiny_q8_swiglu", "small_nvfp4_swiglu"):
        w = SMALL[name]
        L = layers.build_layer(w, source="numpy")
        x = torch.zeros((3, w.d), dtype=torch.float32, device="cuda")
        assert (L.forward(x) == 0).all()


def test_empty_batch_is_a_no_op():
    w = SMALL["tiny_q8_swiglu"]
    L = layers.build_layer(w, source="numpy")
    out = torch.full((1, w.d), 7.0, device="cuda")
    L.forward(torch.zeros((0, w.d), device="cuda"), out=out[:0])
    assert (out == 7.0).all()


def test_rmsnorm_bf16():
    g = np.random.default_rng(3)
    x = (g.standard_normal((5, 2816)) * 3).astype(np.float32)
    got = native.rmsnorm_bf16(_f32(x)).float().cpu().numpy()
    ref = x / np.sqrt((x.astype(np.float64) ** 2).mean(axis=1, keepdims=True) + 1e-6)
    assert np.abs(got - ref).max() <= 2 ** -8 * np.abs(ref).max()


# ------------------------------------------------------------------ the layer, full shapes
def dense_sample(tr, T, k, tile, n_min=64):
    """Tokens to check against the oracle at a full size: the first token of every token tile
    of the hottest expert (tiles of `tile` sorted rows) and of its last row, the last (ragged)
    row of the 16 busiest experts whose row count is not a multiple of the tile, then evenly
    spaced tokens up to n_min.  Every sampled token's output spans every row tile of the
    weights."""
    off = tr["offsets"].cpu().numpy()
    perm = tr["perm"].cpu().numpy()
    cnt = np.diff(off)
    rows = set()
    hot = int(np.argmax(cnt))
    for i in range(0, int(cnt[hot]), tile):
        rows.add(int(perm[off[hot] + i]) // k)
    rows.add(int(perm[off[hot + 1] - 1]) // k)
    ragged = [int(e) for e in np.argsort(-cnt, kind="stable") if cnt[e] % tile]
    for e in ragged[:16]:
        rows.add(int(perm[off[e + 1] - 1]) // k)
    for t in np.linspace(0, T - 1, num=n_min).astype(int):
        if len(rows) >= n_min:
            break
        rows.add(int(t))
    return sorted(rows)


def _full_case(name, T, sample=None, idx_in=None, w_in=None, path="auto", tile=None, act_quant="none"):
    """One full-size layer against the oracle: every token (sample None), the listed tokens,
    or (tile given) the dense_sample of the layer's own permutation.  act_quant "q8_0": the
    activation-quantised expert path on both sides."""
    w = synth.WORKLOADS[name]
    L = layers.build_layer(w, keep_fp32=True, path=path, act_quant=act_quant)
    x = synth.tokens_cuda(w, T, tag="parity")
    tr = {}
    ii = None if idx_in is None else torch.from_numpy(idx_in).cuda()
    ww = None if w_in is None else torch.from_numpy(w_in).cuda()
    out = L.forward(x, idx_in=ii, w_in=ww, trace=tr).cpu().numpy()
    if tile is not None:
        sample = dense_sample(tr, T, w.k, tile)
        assert len(sample) >= 64
    rows = np.arange(T) if sample is None else np.asarray(sample)
    xs = to_numpy_x(x)[rows]
    W = L.router_w.cpu().numpy()
    if idx_in is None:
        lg = oracle.router_logits(xs, W)
        need, _ = oracle.topk_softmax(lg, w.k)
    else:
        need = idx_in[rows]
    ol = oracle_layer(w, W, lambda e: L.gate_up_f32[e].cpu().numpy(), lambda e: L.down_f32[e].cpu().numpy(),
                      need.ravel())
    ref = ol.forward(xs, idx_in=None if idx_in is None else idx_in[rows],
                     w_in=None if w_in is None else w_in[rows], act_q8=act_quant == "q8_0")
    # the packed bytes of the experts used, bit for bit
    for e in sorted(set(int(v) for v in need.ravel()))[:3]:
        if w.wfmt == "q8_0":
            assert np.array_equal(L.gate_up[e].cpu().numpy(), oracle.q8_0_to_device(ol.gate_up[e], w.rows_gu, w.d))
            assert np.array_equal(L.down[e].cpu().numpy(), oracle.q8_0_to_device(ol.down[e], w.d, w.f))
        elif w.wfmt == "int8pc":
            assert np.array_equal(L.gate_up[e].cpu().numpy(), oracle.int8pc_to_device(ol.gate_up[e], w.rows_gu, w.d))
            assert np.array_equal(L.down[e].cpu().numpy(), oracle.int8pc_to_device(ol.down[e], w.d, w.f))
        else:
            assert np.array_equal(L.gate_up[e].cpu().numpy(), oracle.nvfp4_to_panels(ol.gate_up[e], w.rows_gu, w.d))
            assert np.array_equal(L.down[e].cpu().numpy(), oracle.nvfp4_to_neuron(ol.down[e], w.d, w.f))
    if idx_in is None:
        assert np.array_equal(tr["logits"].cpu().numpy()[rows].view(np.uint32), ref["logits"].view(np.uint32))
    assert np.array_equal(tr["idx"].cpu().numpy()[rows], ref["idx"])
    assert np.allclose(tr["w"].cpu().numpy()[rows], ref["w"], rtol=1e-6, atol=0)
    if act_quant == "q8_0":
        check_act_quant(w, ol, rows, out[rows], tr, ref)
        ratio = None
    else:
        ratio = assert_close(out[rows], ref["out"])
    # invariants of the full-size permutation
    off = tr["offsets"].cpu().numpy()
    perm = tr["perm"].cpu().numpy()
    pos = tr["pos"].cpu().numpy()
    assert off[0] == 0 and off[-1] == T * w.k
    assert np.array_equal(perm[pos], np.arange(T * w.k))
    idx_all = tr["idx"].cpu().numpy().ravel()
    assert np.array_equal(np.diff(off), np.bincount(idx_all, minlength=w.E))
    assert np.array_equal(perm, np.argsort(idx_all, kind="stable"))
    del L
    torch.cuda.empty_cache()
    return ratio


@pytest.mark.parametrize("T", [1, 4])
def test_gemma_layer_full_size(T):
    _full_case("gemma", T)


# Token tiles: the GEMV kernels stage up to 8 tokens of an expert, the tensor-core GEMMs 64 to
# 192 sorted rows; sampling every 8th / 64th row of the hottest expert meets every tile of both.
@pytest.mark.parametrize("path,tile", [("gemv", 8), ("gemm", 64)])
def test_gemma_layer_prefill_512_sampled(path, tile):
    _full_case("gemma", 512, path=path, tile=tile)


@pytest.mark.parametrize("T", [1, 32])
def test_nemotron_layer_full_size(T):
    _full_case("nemotron", T)


@pytest.mark.parametrize("T", [1, 8])
def test_minimax_layer_full_size(T):
    _full_case("minimax", T)


def test_minimax_layer_prefill_4096_sampled():
    _full_case("minimax", 4096, tile=64)


# The skewed-routing sweep's sizes up to its largest, T = 8192 (65,536 pairs; the hottest
# expert gets a pair from most tokens, over a hundred 64-row tiles)
@pytest.mark.parametrize("name,T", [("zipf", 64), ("zipf_nvfp4", 64), ("zipf", 2048), ("zipf_nvfp4", 2048),
                                    ("zipf", 8192)])
def test_zipf_routing_full_size(name, T):
    w = synth.WORKLOADS[name]
    idx, wts = synth.zipf_routing(T, w.E, w.k)
    _full_case(name, T, idx_in=idx, w_in=wts, tile=8 if T * w.k < 8 * w.E else 64)


# One token of the sweep's layer shape with supplied routing: the one-kernel layer for Q8_0
# and for NVFP4 SwiGLU (every token of the call checked)
@pytest.mark.parametrize("name", ["zipf", "zipf_nvfp4"])
def test_zipf_one_token_full_size(name):
    w = synth.WORKLOADS[name]
    idx, wts = synth.zipf_routing(1, w.E, w.k)
    _full_case(name, 1, idx_in=idx, w_in=wts)
    L = layers.build_layer(w)
    assert L.launches(1, routing_supplied=True) == 1
    del L
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ the benchmarked stacks, full shape
# The call bench.py times at one token: moe_stack_forward over the Gemma-shaped (Q8_0 SwiGLU)
# and Nemotron-shaped (NVFP4 ReLU^2, 92.5% zeros) stacks, built by the bench's own builder
# (device-drawn weights, each layer warming L2 with the next one's router).  Each layer's
# routing must match the oracle's bit for bit and its output to the tolerance, on the bf16
# input that layer consumed; a second call must be bitwise identical (Nemotron page, "How we
# check correctness": compared against a reference, the same input run repeatedly).
@pytest.mark.parametrize("name,n", [("gemma", 4), ("nemotron", 4)])
def test_benchmarked_stack_full_shape(name, n):
    import bench
    w = synth.WORKLOADS[name]
    stack_layers, inputs = bench.build_stack(w, 1, n, 0)
    st = native.MoEStack(stack_layers)
    assert st.launches() == 1
    x0 = inputs[0]
    xn = torch.empty((n, w.d), dtype=torch.bfloat16, device="cuda")
    routing = {}
    outs = st.forward(x0, x_next=xn, routing=routing).clone()
    for l in range(n):
        xs = to_numpy_x(x0 if l == 0 else xn[l - 1:l])
        W = stack_layers[l].router_w.cpu().numpy()
        need, _ = oracle.topk_softmax(oracle.router_logits(xs, W), w.k)
        ol = oracle_layer(w, W, lambda e: synth.expert_stack_cuda(w, l, "gate_up", [e])[0].cpu().numpy(),
                          lambda e: synth.expert_stack_cuda(w, l, "down", [e])[0].cpu().numpy(), need.ravel())
        ref = ol.forward(xs)
        assert np.array_equal(routing["idx"][l:l + 1].cpu().numpy(), ref["idx"]), l
        assert np.allclose(routing["w"][l:l + 1].cpu().numpy(), ref["w"], rtol=1e-6, atol=0), l
        assert_close(outs[l:l + 1].cpu().numpy(), ref["out"], what=f"layer {l}")
    again = st.forward(x0)
    assert torch.equal(outs.view(torch.int32), again.view(torch.int32))
    del stack_layers, st
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ a stack of layers, one token
# moe_stack_forward: x_{l+1} = bf16(RMSNorm(out_l)).  On Q8_0 SwiGLU layers the whole stack is
# one kernel; it must equal the layers called one by one with moe_rmsnorm_bf16 between them bit
# for bit (the same arithmetic per layer, the same reduction order in the norm), and every layer
# must match the oracle on the input that layer consumed.  path GEMV takes the layer-by-layer
# fallback inside the library.
STACKS = {
    "k8_e64_bf16": (synth.Workload("st_k8", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16",
                                   layers=4), 4),
    "tiny_f32_input": (synth.WORKLOADS["tiny"], 3),
    "nv_relu2": (synth.Workload("st_nv", d=512, f=256, E=32, k=6, act="relu2", wfmt="nvfp4", x_dtype="bf16",
                                layers=3, zero_fraction=0.925), 3),
    "nv_swiglu": (synth.Workload("st_nvsw", d=768, f=256, E=32, k=8, act="swiglu", wfmt="nvfp4",
                                 x_dtype="bf16", layers=3), 3),
    "int8pc": (synth.Workload("st_pc", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="int8pc", x_dtype="bf16",
                              layers=3), 3),
}


@pytest.mark.parametrize("name", list(STACKS))
@pytest.mark.parametrize("path", ["auto", "gemv"])
def test_stack_one_token(name, path):
    w, n = STACKS[name]
    layers_ = [layers.build_layer(w, layer=l, source="numpy", path=path) for l in range(n)]
    stack = native.MoEStack(layers_)
    if path == "auto":
        assert stack.launches(True) == 1
    else:   # each layer's own launches, then the norm
        assert stack.launches(True) == n * (layers_[0].launches(1) + 1)
    x0 = torch.from_numpy(synth.tokens(w, 1, tag="stack")).cuda()
    if w.x_dtype == "bf16":
        x0 = x0.view(torch.bfloat16)
    xn = torch.full((n, w.d), 0, dtype=torch.bfloat16, device="cuda")
    outs = torch.full((n, w.d), float("nan"), device="cuda")
    routing = {}
    stack.forward(x0, outs=outs, x_next=xn, routing=routing)
    # layer by layer through the single-layer calls and the stand-alone norm
    x = x0
    for l, L in enumerate(layers_):
        tr = {}
        o = L.forward(x, trace=tr)
        assert np.array_equal(o.cpu().numpy().view(np.uint32), outs[l:l + 1].cpu().numpy().view(np.uint32)), l
        assert np.array_equal(tr["idx"].cpu().numpy(), routing["idx"][l:l + 1].cpu().numpy())
        assert np.array_equal(tr["w"].cpu().numpy().view(np.uint32), routing["w"][l:l + 1].cpu().numpy().view(np.uint32))
        x = native.rmsnorm_bf16(o)
        assert torch.equal(x.view(torch.int16), xn[l:l + 1].view(torch.int16)), l
    # each layer against the oracle on its own input
    for l in range(n):
        xl = x0 if l == 0 else xn[l - 1:l]
        xs = to_numpy_x(xl)
        ol = oracle_layer(w, synth.router_weight(w, l), lambda e: synth.expert_weights(w, l, e)[0],
                          lambda e: synth.expert_weights(w, l, e)[1], range(w.E))
        ref = ol.forward(xs)
        assert np.array_equal(routing["idx"][l:l + 1].cpu().numpy(), ref["idx"])
        assert_close(outs[l:l + 1].cpu().numpy(), ref["out"])
    # run to run: bitwise identical
    outs2 = stack.forward(x0)
    assert torch.equal(outs.view(torch.int32), outs2.view(torch.int32))
