"""Expert-parallel dispatch and combine (ep.py) on CPU ranks over gloo.

The distributed page ("Why can super-large MoE be distributed for inference", the swarm
section) keeps the router on the backbone and sends the expert work to the machines that hold
the experts.  With expert e on rank e mod G, each rank's tokens routed on that rank, the rows
shipped out and back by all-to-all and combined in slot order, every rank's output must equal
the single-rank oracle's output for its tokens bit for bit: the experts are evaluated by the
oracle on the rank that holds them, and the combine adds the same fp64 terms in the same
order.  World sizes 2 and 3 (with 3, ranks hold different numbers of experts); one rank has
no tokens of its own and still serves its experts."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

D, F, E, K = 256, 128, 14, 3
TOKENS = [5, 0, 9]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    from quantized_routed_expert_softmax_gb300 import synth
    return synth.Workload("ep_gloo", d=D, f=F, E=E, k=K, act="swiglu", wfmt="q8_0", x_dtype="f32", layers=1)


def _oracle_layer(w, experts, n_layer_experts, k, router):
    """An oracle layer holding `experts` ((index in this layer, global expert) pairs)."""
    import oracle
    from quantized_routed_expert_softmax_gb300 import synth
    gu = [None] * n_layer_experts
    dn = [None] * n_layer_experts
    for le, e in experts:
        a, b = synth.expert_weights(w, 0, e)
        gu[le] = oracle.q8_0_quantize(a)
        dn[le] = oracle.q8_0_quantize(b)
    return oracle.Layer(w.d, w.f, n_layer_experts, k, oracle.ACT_SWIGLU, oracle.W_Q8_0, router, gu, dn)


def _tokens(w, rank):
    from quantized_routed_expert_softmax_gb300 import synth
    T = TOKENS[rank]
    return synth.tokens_f32(w, max(T, 1), tag=f"ep{rank}")[:T]


def _rank_main(rank, world, port, out_dir):
    import oracle
    from quantized_routed_expert_softmax_gb300 import ep, synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _workload()
        x = _tokens(w, rank)
        if len(x):   # the router on this rank's tokens
            idx, wts = oracle.topk_softmax(oracle.router_logits(x, synth.router_weight(w)), K)
        else:
            idx, wts = np.zeros((0, K), np.int32), np.zeros((0, K), np.float32)
        mine = list(enumerate(range(rank, E, world)))           # this rank's experts: e = rank (mod G)
        local = _oracle_layer(w, mine, len(mine), 1, np.zeros((D, len(mine)), np.float32))

        def run_local(rows, ids):
            got = local.forward(rows.numpy(), idx_in=ids.numpy().astype(np.int32).reshape(-1, 1),
                                w_in=np.ones((rows.shape[0], 1), np.float32))
            return torch.from_numpy(got["out"])                 # 0.0 + 1.0 * y: the expert's y exactly

        out = ep.ep_forward(torch.from_numpy(x), idx, torch.from_numpy(wts.astype(np.float64)), run_local)
        np.save(os.path.join(out_dir, f"rank{rank}.npy"), out.numpy())
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_expert_parallel_equals_single_rank_oracle(tmp_path, world):
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    from quantized_routed_expert_softmax_gb300 import synth
    w = _workload()
    full = _oracle_layer(w, [(e, e) for e in range(E)], E, K, synth.router_weight(w))
    for r in range(world):
        x = _tokens(w, r)
        got = np.load(tmp_path / f"rank{r}.npy")
        if len(x) == 0:
            assert got.shape == (0, D)
            continue
        ref = full.forward(x)["out"]
        assert np.array_equal(got.view(np.uint64), ref.view(np.uint64)), (r, float(np.abs(got - ref).max()))


def test_dispatch_plan_orders_by_rank_expert_pair():
    from quantized_routed_expert_softmax_gb300 import ep
    idx = np.array([[5, 2, 7], [2, 4, 5], [7, 0, 3]])
    order, counts = ep.dispatch_plan(idx, 2)
    flat = idx.ravel()
    assert counts.tolist() == [np.sum(flat % 2 == 0), np.sum(flat % 2 == 1)]
    keys = [(flat[p] % 2, flat[p], p) for p in order]
    assert keys == sorted(keys)                           # rank, then expert, then pair id
    assert sorted(order.tolist()) == list(range(flat.size))
    assert ep.local_expert(7, 2) == 3 and ep.expert_rank(7, 2) == 1
