"""The expert ranks' evaluator of ep.py on the GPU, without a collective.

In expert-parallel decoding (the distributed page, "Why can super-large MoE be distributed for
inference", the swarm section) every rank evaluates the experts it holds on the rows other
ranks send it.  ep.LocalExperts does it with libmoe: a layer over the rank's experts with one
expert per row and weight 1 (supplied routing).  Here both ranks of a two-way split run in one
process on one GPU, the rows routed to each as the dispatch would send them, and the slot-order
combine of their outputs must match the oracle's layer (and the single-GPU layer) to the
tolerance.  The all-to-all exchange itself is tested on CPU ranks (test_ep_gloo.py)."""
import numpy as np
import pytest
import torch

from oracle_bridge import assert_close, oracle_layer
from quantized_routed_expert_softmax_gb300 import ep, layers, native, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_softmax_gb300 import build
    build.build()
    native.lib()


@pytest.mark.parametrize("T", [1, 6, 40])
def test_local_experts_of_two_ranks_combine_to_the_layer(T):
    w = synth.Workload("ep_gpu", d=1024, f=192, E=64, k=8, act="swiglu", wfmt="q8_0", x_dtype="bf16", layers=1)
    G = 2
    L = layers.build_layer(w, source="numpy")
    x = torch.from_numpy(synth.tokens(w, T, tag="ep")).cuda().view(torch.bfloat16)
    tr = {}
    out = L.forward(x, trace=tr)
    idx = tr["idx"].cpu().numpy()
    flat = idx.ravel()
    y_pair = torch.zeros((T * w.k, w.d), dtype=torch.float32, device="cuda")
    order, counts = ep.dispatch_plan(idx, G)
    start = 0
    for r in range(G):   # the rows rank r would receive, in send order
        pairs = order[start:start + counts[r]]
        start += counts[r]
        le = ep.LocalExperts(w.d, w.f, w.E // G, w.act, w.wfmt, L.gate_up[r::G].contiguous(),
                             L.down[r::G].contiguous())
        pt = torch.from_numpy(pairs).cuda()
        ids = torch.from_numpy(ep.local_expert(flat[pairs], G).astype(np.int64)).cuda()
        y_pair[pt] = le(x[pt // w.k].contiguous(), ids)
    got = ep.combine(tr["w"], y_pair, w.k).cpu().numpy()
    ol = oracle_layer(w, synth.router_weight(w), lambda e: synth.expert_weights(w, 0, e)[0],
                      lambda e: synth.expert_weights(w, 0, e)[1], range(w.E))
    ref = ol.forward(synth.tokens(w, T, tag="ep"))
    assert np.array_equal(idx, ref["idx"])
    assert_close(got, ref["out"])
    assert_close(got, out.cpu().numpy().astype(np.float64), what="against the single-GPU layer")
