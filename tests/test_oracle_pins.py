"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle function to an independent fact: a number the pages print
(tests/golden/page_numbers.json), a library routine (numpy's float16, torch's
float8_e4m3fn, scipy's expit), a value worked out by hand from the format definition,
an invariant (round trips, permutations), a special case with a closed form, or brute
force on tiny inputs.  None of them needs a GPU.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_routed_expert_softmax_gb300 import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


def page(key):
    return GOLDEN[key]["value"]


# ------------------------------------------------------------------ byte counts (pages)
def test_nemotron_expert_bytes_match_page():
    up = oracle.nvfp4_bytes(2688, 1024)
    down = oracle.nvfp4_bytes(1024, 2688)
    assert up + down == page("nemotron_expert_bytes")
    assert (up + down) % 4096 == 0 and (up + down) // 4096 == page("nemotron_expert_pages_4kib")
    assert round((up + down) / 1e6, 2) == page("nemotron_expert_mb")
    assert round(up / 1e6, 2) == page("nemotron_up_mb")
    s = page("nemotron_shape")
    per_token = s["top_k"] * s["moe_layers"] * (up + down)
    assert abs(per_token / 1e9 - page("nemotron_gb_per_token")) < 0.05
    routed = s["experts"] * s["moe_layers"] * (up + down)
    assert round(routed / 2**30) == page("nemotron_routed_gib")


def test_gemma_shapes_match_page():
    w = synth.WORKLOADS["gemma"]
    bf16_bytes = w.layers * w.E * (w.rows_gu * w.d + w.d * w.f) * 2
    assert abs(bf16_bytes / 1e9 - page("gemma_bf16_experts_gb")) / page("gemma_bf16_experts_gb") < 0.005
    assert w.layers * w.k == page("gemma_uncomputed_tensors_per_forward")
    # Q8_0: 34 bytes per 32 weights
    per_expert = oracle.q8_0_bytes(w.rows_gu, w.d) + oracle.q8_0_bytes(w.d, w.f)
    assert per_expert == (w.rows_gu * w.d + w.d * w.f) // 32 * 34 == 6_319_104


def test_minimax_and_nemotron_workloads_match_pages():
    m = page("minimax_experts")
    w = synth.WORKLOADS["minimax"]
    assert (w.d, w.f, w.E, w.k) == (m["n_embd"], m["ffn"], m["experts"], m["top_k"])
    assert m["moe_layers"] * m["experts"] == m["held"] and m["moe_layers"] * m["top_k"] == m["computed_per_token"]
    n = page("nemotron_shape")
    w = synth.WORKLOADS["nemotron"]
    assert (w.d, w.f, w.E, w.k, w.layers) == (n["latent"], n["ffn"], n["experts"], n["top_k"], n["moe_layers"])
    assert w.zero_fraction == page("nemotron_zero_fraction")


# ------------------------------------------------------------------ scalar codecs
def test_fp16_encode_matches_numpy():
    g = np.random.default_rng(1)
    vals = np.concatenate([
        g.standard_normal(4000).astype(np.float32) * np.float32(1e-3),
        g.standard_normal(2000).astype(np.float32),
        (g.random(2000) * 6e-5).astype(np.float32),          # subnormal range
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e-8, 6.1035156e-05], np.float32),
    ])
    # exact half-way points between adjacent fp16 values
    h = np.arange(0x0400, 0x7bff, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    h2 = (np.arange(0x0400, 0x7bff, 37, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    vals = np.concatenate([vals, ((h + h2) / 2).astype(np.float32)])
    for v in vals:
        ref = int(np.array([v], np.float32).astype(np.float16).view(np.uint16)[0])
        assert oracle.f32_to_f16_bits(float(v)) == ref, v


def test_fp16_decode_all_codes():
    codes = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    for c in range(0, 0x10000, 7):
        got = oracle.f16_bits_to_f64(c)
        if np.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c]


def test_e4m3_decode_all_256_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_to_f64(c)
        if np.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c], c


def test_e4m3_encode_matches_torch_in_range():
    g = np.random.default_rng(2)
    vals = np.concatenate([
        g.random(3000) * 448.0, g.random(2000) * 0.02, g.random(500) * 2.0 ** -8,
        np.array([0.0, 448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11, 240.0, 232.0, 15.5])])
    # midpoints between adjacent finite codes
    dec = np.array([oracle.e4m3_to_f64(c) for c in range(0x7f)])
    vals = np.concatenate([vals, (dec[:-1] + dec[1:]) / 2]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, r in zip(vals, ref):
        assert oracle.f32_to_e4m3(float(v)) == int(r), v


def test_e4m3_saturates():
    assert oracle.f32_to_e4m3(1000.0) == 0x7e        # 448, the largest finite code
    assert oracle.e4m3_to_f64(0x7e) == 448.0


E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_decode_table():
    # OCP microscaling FP4 E2M1 value table (1 sign, 2 exponent bits with bias 1, 1 mantissa bit)
    for c, v in enumerate(E2M1_TABLE):
        assert oracle.e2m1_to_f64(c) == v and math.copysign(1, oracle.e2m1_to_f64(c)) == math.copysign(1, v)


def test_e2m1_encode_is_nearest_ties_to_even_code():
    mags = E2M1_TABLE[:8]
    grid = sorted(set([i / 64 for i in range(0, 64 * 8)] + [(a + b) / 2 for a, b in zip(mags, mags[1:])]))
    for x in grid + [-v for v in grid] + [7.0, 100.0, -9.0]:
        # brute force over the 8 magnitudes: nearest, ties to the even code (even mantissa bit)
        a = abs(x)
        best = min(range(8), key=lambda c: (abs(mags[c] - a), c & 1))
        if a > 6.0:
            best = 7
        want = best if (best == 0 or x >= 0) else best | 8
        assert oracle.f32_to_e2m1(x) == want, x


# ------------------------------------------------------------------ Q8_0
def _q8_block(vals):
    x = np.zeros((1, 32), np.float32)
    x[0, : len(vals)] = vals
    return oracle.q8_0_quantize(x)


def test_q8_0_all_zero_block():
    b = _q8_block([])
    assert b.shape == (34,) and not b.any()


def test_q8_0_constant_block():
    b = oracle.q8_0_quantize(np.full((1, 32), 0.3, np.float32))
    d = np.float32(0.3) / np.float32(127.0)
    assert int(b[0]) | (int(b[1]) << 8) == int(np.array([d], np.float32).astype(np.float16).view(np.uint16)[0])
    assert (b[2:].view(np.int8) == 127).all()
    b = oracle.q8_0_quantize(np.full((1, 32), -0.3, np.float32))
    assert (b[2:].view(np.int8) == -127).all()


def test_q8_0_rounds_half_away_from_zero():
    # amax 127 -> d = 1, 1/d = 1: the codes are round-half-away of the values themselves
    b = _q8_block([127.0, 2.5, -2.5, 0.5, -0.5, 1.5, 126.5, -0.49])
    q = b[2:].view(np.int8)
    assert list(q[:8]) == [127, 3, -3, 1, -1, 2, 127, 0]
    assert int(b[0]) | (int(b[1]) << 8) == 0x3C00   # fp16 1.0


def test_q8_0_codes_use_the_fp32_scale_not_the_stored_fp16_one():
    # amax 1: d = 1/127 in fp32 (0.0078740157), stored as fp16 0.00787353515625 (smaller by
    # 6e-5 relative).  0.49997 * 127 = 63.496 -> code 63 with the fp32 scale; dividing by
    # the fp16 scale would give 63.50007 -> 64.
    b = _q8_block([1.0, 0.49997, -0.49997])
    assert int(b[0]) | (int(b[1]) << 8) == 0x2008          # fp16 0.00787353515625
    assert oracle.f16_bits_to_f64(0x2008) == 0.00787353515625
    assert list(b[2:5].view(np.int8)) == [127, 63, -63]


def test_q8_0_roundtrip_fixed_point_and_error_bound():
    g = np.random.default_rng(3)
    x = (g.standard_normal((16, 256)) * 0.02).astype(np.float32)
    q = oracle.q8_0_quantize(x)
    dq = oracle.q8_0_dequant(q, 16, 256)
    assert np.array_equal(oracle.q8_0_quantize(dq.astype(np.float32)), q)
    # |x - dequant| <= half a step, step = d (fp32), plus the fp16 rounding of d times |q|
    blocks = x.reshape(16, 8, 32)
    d32 = np.abs(blocks).max(axis=2, keepdims=True).astype(np.float64) / 127.0
    err = np.abs(dq.reshape(16, 8, 32) - blocks.astype(np.float64))
    assert (err <= d32 * 0.5 * (1 + 1e-6) + 127 * d32 * 2.0 ** -11).all()


def test_q8_0_device_layout_is_a_byte_permutation():
    g = np.random.default_rng(4)
    rows, cols = 24, 96
    x = (g.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    c = oracle.q8_0_quantize(x)
    d = oracle.q8_0_to_device(c, rows, cols)
    assert np.array_equal(oracle.q8_0_from_device(d, rows, cols), c)
    assert np.array_equal(np.sort(c), np.sort(d))
    # hand check: panel 1 (columns 32..63), row 5 starts at 1*rows*34 + 5*32 and holds
    # the 32 codes of block (5, 1); its scale is at 1*rows*34 + rows*32 + 5*2
    nb = cols // 32
    blk = c[(5 * nb + 1) * 34:(5 * nb + 2) * 34]
    assert np.array_equal(d[rows * 34 + 5 * 32: rows * 34 + 6 * 32], blk[2:])
    assert np.array_equal(d[rows * 34 + rows * 32 + 10: rows * 34 + rows * 32 + 12], blk[:2])


def test_int8pc_device_layout_is_a_byte_permutation():
    # per-channel int8 (Inferentia page, "Wall 1: the memory math"): the device layout the
    # weight-streaming kernels read holds the same bytes in another order
    g = np.random.default_rng(5)
    rows, cols = 40, 96
    x = (g.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    c = oracle.int8pc_quantize(x)
    d = oracle.int8pc_to_device(c, rows, cols)
    assert np.array_equal(oracle.int8pc_from_device(d, rows, cols), c)
    assert np.array_equal(np.sort(c), np.sort(d))
    # hand check: row 7's fp32 scale is bytes 28..31; panel 2 (columns 64..95) starts at
    # 4*rows + 2*rows*32 and row 7's 32 codes there are the canonical codes (7, 64..95)
    assert np.array_equal(d[28:32], c[rows * cols + 28: rows * cols + 32])
    p2 = 4 * rows + 2 * rows * 32
    assert np.array_equal(d[p2 + 7 * 32: p2 + 8 * 32], c[7 * cols + 64: 7 * cols + 96])
    # a planted mistake fails it: swapping two rows of a panel
    bad = d.copy()
    bad[p2: p2 + 32], bad[p2 + 32: p2 + 64] = d[p2 + 32: p2 + 64], d[p2: p2 + 32]
    assert not np.array_equal(oracle.int8pc_from_device(bad, rows, cols), c)


# ------------------------------------------------------------------ NVFP4
def test_nvfp4_hand_worked_block():
    # Row 0 holds 10.5, so s_t = 10.5 / 2688 = 2^-8 exactly.  Row 1's first block has
    # amax 6: sb = E4M3(6 / (6 * 2^-8)) = 256 and dec(sb) * s_t = 1, so its codes are the
    # plain E2M1 roundings of the values, ties to the even code.
    x = np.zeros((2, 16), np.float32)
    x[0, 0] = 10.5
    x[1] = [6, -6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, 0.3, -0.2, 4, 3, 2, 1, 0.5]
    q, st = oracle.nvfp4_quantize(x)
    assert st == 2.0 ** -8
    vals, scales = q[:16], q[16:]
    codes = [(vals[i // 2] >> (4 * (i % 2))) & 0xF for i in range(32)]
    assert codes[16:] == [0x7, 0xF, 0x0, 0x2, 0x2, 0x4, 0x4, 0x6, 0x6, 0x1, 0x0, 0x6, 0x5, 0x4, 0x2, 0x1]
    # row 0: sb = E4M3(10.5 / (6/256)) = 448 -> dec*st = 1.75 -> 10.5/1.75 = 6 -> code 7
    assert codes[0] == 0x7 and all(c == 0 for c in codes[1:16])
    assert oracle.e4m3_to_f64(int(scales[0])) == 448.0 and oracle.e4m3_to_f64(int(scales[1])) == 256.0


def test_nvfp4_nibble_order_low_is_even_element():
    x = np.zeros((1, 16), np.float32)
    x[0, 0], x[0, 1] = 1.0, -6.0     # amax 6: s_t = 6/2688, block scale 448
    q, st = oracle.nvfp4_quantize(x)
    dq = oracle.nvfp4_dequant(q, 1, 16, st)
    assert q[0] == 0xF2
    assert abs(dq[0, 0] - 1.0) < 1e-6 and abs(dq[0, 1] + 6.0) < 1e-6


def test_nvfp4_all_zero_matrix():
    q, st = oracle.nvfp4_quantize(np.zeros((4, 32), np.float32))
    assert st == 1.0 and not q.any()


def test_nvfp4_dequant_matches_library_decoders():
    g = np.random.default_rng(5)
    x = (g.standard_normal((8, 64)) * 0.02).astype(np.float32)
    q, st = oracle.nvfp4_quantize(x)
    vals, scales = q[: 8 * 32], q[8 * 32:]
    codes = np.stack([vals & 0xF, vals >> 4], axis=1).reshape(8, 64)
    e2m1 = np.array(E2M1_TABLE)[codes]
    sc = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).double().numpy().reshape(8, 4)
    ref = e2m1 * np.repeat(sc, 16, axis=1) * np.float64(np.float32(st))
    assert np.array_equal(oracle.nvfp4_dequant(q, 8, 64, st), ref)
    # quantisation error is within half an E2M1 step of the block's scale (step <= 2 at 4..6)
    assert np.abs(ref - x).max() <= np.abs(x).max()


def test_nvfp4_nibble_swap_must_fail():
    """Swapping the two nibbles of every byte must break the result (Nemotron page,
    'How we check correctness': the swap sent perplexity to 18,784)."""
    w = synth.WORKLOADS["tiny"]
    g = np.random.default_rng(6)
    W = (g.standard_normal((64, 256)) * 0.02).astype(np.float32)
    q, st = oracle.nvfp4_quantize(W)
    sw = q.copy()
    nv = 64 * 256 // 2
    sw[:nv] = ((q[:nv] & 0xF) << 4) | (q[:nv] >> 4)
    good = oracle.nvfp4_dequant(q, 64, 256, st)
    bad = oracle.nvfp4_dequant(sw, 64, 256, st)
    x = synth.tokens_f32(w, 4)
    rel = np.linalg.norm(x @ bad.T - x @ good.T) / np.linalg.norm(x @ good.T)
    assert rel > 0.5


def test_nvfp4_panel_layout_roundtrip():
    g = np.random.default_rng(7)
    rows, cols = 16, 128
    q, _ = oracle.nvfp4_quantize((g.standard_normal((rows, cols)) * 0.02).astype(np.float32))
    p = oracle.nvfp4_to_panels(q, rows, cols)
    assert np.array_equal(oracle.nvfp4_from_panels(p, rows, cols), q)
    assert np.array_equal(np.sort(p), np.sort(q))
    # panel 1, row 3: code bytes 32..63 of row 3, then its 4 scale bytes at 1*rows*36 + rows*32 + 3*4
    assert np.array_equal(p[rows * 36 + 3 * 32: rows * 36 + 4 * 32], q[3 * 64 + 32: 3 * 64 + 64])
    sbase = rows * cols // 2
    assert np.array_equal(p[rows * 36 + rows * 32 + 12: rows * 36 + rows * 32 + 16], q[sbase + 3 * 8 + 4: sbase + 3 * 8 + 8])


def test_nvfp4_neuron_relayout_is_an_invertible_byte_permutation():
    g = np.random.default_rng(8)
    rows, cols = 32, 64        # a down matrix [d, f]
    q, _ = oracle.nvfp4_quantize((g.standard_normal((rows, cols)) * 0.02).astype(np.float32))
    n = oracle.nvfp4_to_neuron(q, rows, cols)
    assert n.size == q.size
    assert np.array_equal(oracle.nvfp4_from_neuron(n, rows, cols), q)
    # nibble multiset of the codes and byte multiset of the scales are preserved
    nv = rows * cols // 2
    canon_codes = np.sort(np.concatenate([q[:nv] & 0xF, q[:nv] >> 4]))
    rec = 16 * rows // 2 + rows
    neur_vals = np.concatenate([n[g_ * rec: g_ * rec + 16 * rows // 2] for g_ in range(cols // 16)])
    assert np.array_equal(canon_codes, np.sort(np.concatenate([neur_vals & 0xF, neur_vals >> 4])))
    # hand check: neuron n = 16*2 + 5 (group 2, member 5), row r = 7 (odd: high nibble of byte 3)
    r, nn = 7, 37
    cbyte = q[(r * cols + nn) // 2]
    ccode = (cbyte >> 4) if nn & 1 else (cbyte & 0xF)
    nbyte = n[2 * rec + 5 * (rows // 2) + r // 2]
    assert (nbyte >> 4) == ccode
    # the scale of (row 7, group 2) sits after the group's 16 neuron records
    assert n[2 * rec + 16 * rows // 2 + 7] == q[nv + 7 * (cols // 16) + 2]


def test_nvfp4_round_trip_over_200_experts_of_relayout():
    """The page compares the repack and relayout byte for byte over 200 experts; here
    200 small random down matrices go through the relayout and back."""
    g = np.random.default_rng(9)
    for _ in range(200):
        q = g.integers(0, 256, size=oracle.nvfp4_bytes(16, 32), dtype=np.uint8)
        assert np.array_equal(oracle.nvfp4_from_neuron(oracle.nvfp4_to_neuron(q, 16, 32), 16, 32), q)


# ------------------------------------------------------------------ router
def test_router_zero_input_picks_lowest_indices_uniformly():
    x = np.zeros((3, 256), np.float32)
    W = np.random.default_rng(10).standard_normal((256, 8)).astype(np.float32)
    lg = oracle.router_logits(x, W)
    assert not lg.any()
    idx, w = oracle.topk_softmax(lg, 3)
    assert (idx == [0, 1, 2]).all() and (w == 1.0 / 3.0).all()


def test_router_k1_weight_is_one():
    g = np.random.default_rng(11)
    lg = g.standard_normal((5, 8)).astype(np.float32)
    idx, w = oracle.topk_softmax(lg, 1)
    assert (w == 1.0).all() and (idx[:, 0] == lg.argmax(axis=1)).all()


def test_topk_tie_break_lower_index_and_slot_order():
    lg = np.array([[1.0, 3.0, 3.0, 2.0], [0.0, -0.0, 5.0, -0.0]], np.float32)
    idx, w = oracle.topk_softmax(lg, 3)
    assert idx[0].tolist() == [1, 2, 3]
    assert idx[1].tolist() == [2, 0, 1]
    e = np.exp([0.0, 0.0, -1.0])
    assert np.allclose(w[0], e / e.sum(), rtol=1e-15, atol=0)


def test_softmax_weights_survive_large_logits():
    # the maximum (slot 0) is subtracted before exponentiating
    lg = np.array([[800.0, 799.0, -5.0, 790.0]], np.float32)
    idx, w = oracle.topk_softmax(lg, 2)
    assert idx[0].tolist() == [0, 1]
    assert np.allclose(w[0], [1 / (1 + math.exp(-1)), math.exp(-1) / (1 + math.exp(-1))], rtol=1e-15, atol=0)


def test_topk_brute_force_against_a_full_sort():
    g = np.random.default_rng(12)
    lg = g.standard_normal((64, 128)).astype(np.float32)
    lg[:, 5] = lg[:, 9]                                   # some exact ties
    for k in (1, 2, 8, 22):
        idx, w = oracle.topk_softmax(lg, k)
        for t in range(64):
            order = np.lexsort((np.arange(128), -lg[t].astype(np.float64)))  # value desc, index asc
            assert idx[t].tolist() == order[:k].tolist()
            sel = lg[t, order[:k]].astype(np.float64)
            sm = np.exp(sel - sel.max())
            assert np.allclose(w[t], sm / sm.sum(), rtol=1e-14, atol=0)
        # the softmax over the k selected equals the full softmax renormalised on them
        full = np.exp(lg.astype(np.float64) - lg.max(axis=1, keepdims=True))
        full /= full.sum(axis=1, keepdims=True)
        sel = np.take_along_axis(full, idx.astype(np.int64), axis=1)
        assert np.allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12, atol=0)


def test_router_canonical_order_hand_cases():
    # d = 512, one expert.  Chain l sums i = l, l+256 in order; the tree merges chain l+h
    # into chain l for h = 128, ..., 1.
    big = 2.0 ** 24
    W = np.zeros((512, 1), np.float32)
    x = np.zeros((1, 512), np.float32)
    x[0, [0, 1, 257]] = 1.0
    W[[0, 1, 257], 0] = [big, 1.0, 1.0]
    # chain 1 = 1 + 1 = 2 first, then 2^24 + 2 is exact
    assert oracle.router_logits(x, W)[0, 0] == big + 2
    # a left-to-right sum would have lost both ones: 2^24 + 1 rounds to 2^24 (tie, even)
    x2 = np.zeros((1, 512), np.float32)
    W2 = np.zeros((512, 1), np.float32)
    x2[0, [0, 1, 128]] = 1.0
    W2[[0, 1, 128], 0] = [big, 1.0, 1.0]
    # chain 128 meets chain 0 at h = 128 (2^24 + 1 -> 2^24), chain 1 meets it at h = 1
    assert oracle.router_logits(x2, W2)[0, 0] == big


def test_router_tree_pairs_chain_l_with_chain_l_plus_h():
    # big value in chain 2, ones in chains 1 and 3: the tree's h = 2 level adds chain 3 to
    # chain 1 (1 + 1 = 2) and chain 2 to chain 0; h = 1 then gives 2^24 + 2 exactly.
    # Pairing chains differently, or summing left to right, loses both ones.
    big = 2.0 ** 24
    W = np.zeros((256, 1), np.float32)
    x = np.zeros((1, 256), np.float32)
    x[0, [1, 2, 3]] = 1.0
    W[[1, 2, 3], 0] = [1.0, big, 1.0]
    assert oracle.router_logits(x, W)[0, 0] == big + 2


def test_router_logits_within_fp32_error_bound_of_exact_dot():
    w = synth.WORKLOADS["gemma"]
    x = synth.tokens(w, 8)
    W = synth.router_weight(w)
    lg = oracle.router_logits(x, W).astype(np.float64)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    exact = xf @ W.astype(np.float64)
    bound = (w.d / 256 + 8 + 2) * 2.0 ** -24 * (np.abs(xf) @ np.abs(W.astype(np.float64)))
    assert (np.abs(lg - exact) <= bound).all()


# ------------------------------------------------------------------ permutation
def test_permute_brute_force_and_invariants():
    g = np.random.default_rng(13)
    T, k, E = 50, 4, 16
    idx = np.stack([g.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    offsets, perm, pos = oracle.permute(idx, E)
    flat = idx.ravel()
    assert offsets[0] == 0 and offsets[E] == T * k
    assert np.array_equal(np.diff(offsets), np.bincount(flat, minlength=E))
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(perm[pos], np.arange(T * k)) and np.array_equal(pos[perm], np.arange(T * k))


# ------------------------------------------------------------------ experts and the layer
def _tiny_layer(act="swiglu", wfmt="q8_0", E=8, k=2, d=256, f=512, zero_fraction=None, seed_name="tiny"):
    w = synth.Workload(seed_name, d=d, f=f, E=E, k=k, act=act, wfmt=wfmt, x_dtype="f32", layers=1,
                       rms_norm_input=zero_fraction is not None, zero_fraction=zero_fraction)
    gu, dn, gts, dts = [], [], [], []
    for e in range(E):
        a, b = synth.expert_weights(w, 0, e)
        if wfmt == "q8_0":
            gu.append(oracle.q8_0_quantize(a))
            dn.append(oracle.q8_0_quantize(b))
        else:
            qa, sa = oracle.nvfp4_quantize(a)
            qb, sb = oracle.nvfp4_quantize(b)
            gu.append(qa), dn.append(qb), gts.append(sa), dts.append(sb)
    L = oracle.Layer(d, f, E, k, oracle.ACT_SWIGLU if act == "swiglu" else oracle.ACT_RELU2,
                     oracle.W_Q8_0 if wfmt == "q8_0" else oracle.W_NVFP4, synth.router_weight(w), gu, dn,
                     gts or None, dts or None)
    return w, L


def _dequant_all(L):
    rows = 2 * L.f if L.act == oracle.ACT_SWIGLU else L.f
    if L.wfmt == oracle.W_Q8_0:
        gu = [oracle.q8_0_dequant(L.gate_up[e], rows, L.d) for e in range(L.E)]
        dn = [oracle.q8_0_dequant(L.down[e], L.d, L.f) for e in range(L.E)]
    else:
        gu = [oracle.nvfp4_dequant(L.gate_up[e], rows, L.d, L.gate_up_tscale[e]) for e in range(L.E)]
        dn = [oracle.nvfp4_dequant(L.down[e], L.d, L.f, L.down_tscale[e]) for e in range(L.E)]
    return gu, dn


@pytest.mark.parametrize("wfmt", ["q8_0", "nvfp4"])
def test_fused_gate_up_equals_two_mul_mat_id_and_fused_mul_silu(wfmt):
    """Xeon page, 'A three-step fix' / 'Runtime graph fallback': the fused
    [n_embd, 2 n_ff, n_experts] tensor split into two views (gate first, up second),
    one expert-indexed matmul on each, then SiLU(gate) * up."""
    w, L = _tiny_layer(wfmt=wfmt)
    x = synth.tokens(w, 16)
    res = L.forward(x)
    gu, _ = _dequant_all(L)
    xd = x.astype(np.float64)
    gate = oracle.mul_mat_id(gu, 0, L.f, xd, res["idx"])
    up = oracle.mul_mat_id(gu, L.f, L.f, xd, res["idx"])
    h = oracle.fused_mul_silu(gate, up).reshape(16 * L.k, L.f)
    assert np.array_equal(h, res["h"])
    # swapping the halves gives a different result (the order is pinned, not assumed)
    assert not np.allclose(oracle.fused_mul_silu(up, gate).reshape(16 * L.k, L.f), res["h"])


def test_silu_matches_scipy():
    from scipy.special import expit
    for v in [-30.0, -3.0, -0.5, 0.0, 0.5, 2.0, 30.0]:
        assert oracle.lib().orc_silu(v) == pytest.approx(v * expit(v), rel=1e-15, abs=1e-300)


def test_sparse_down_equals_dense_down_with_relu2_zeros():
    """Nemotron page, step 4: skipping 16-neuron groups that are all zero changes nothing."""
    w, L = _tiny_layer(act="relu2", wfmt="nvfp4", zero_fraction=0.925, seed_name="relu2-tiny")
    x = synth.tokens_f32(w, 16)
    a = L.forward(x, sparse_down=True)
    b = L.forward(x, sparse_down=False)
    assert np.array_equal(a["out"], b["out"])
    h = a["h"]
    groups = (h.reshape(h.shape[0], -1, 16) != 0).any(axis=2)
    assert (~groups).any(), "some groups must be all zero for the test to mean anything"


def test_dense_experts_identity():
    """Inferentia page, 'Honest caveats': evaluating all experts with zero weight off the
    selected set gives the routed layer's result."""
    w, L = _tiny_layer()
    x = synth.tokens(w, 16)
    res = L.forward(x)
    wfull = np.zeros((16, L.E))
    np.put_along_axis(wfull, res["idx"].astype(np.int64), res["w"], axis=1)
    dense = L.forward_dense_experts(x, wfull)
    assert np.allclose(dense, res["out"], rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("act", ["swiglu", "relu2"])
def test_zero_input_gives_zero_output(act):
    w, L = _tiny_layer(act=act, wfmt="q8_0" if act == "swiglu" else "nvfp4")
    out = L.forward(np.zeros((4, L.d), np.float32))["out"]
    assert (out == 0).all()


@pytest.mark.parametrize("act,wfmt", [("swiglu", "q8_0"), ("relu2", "nvfp4"), ("swiglu", "nvfp4")])
def test_layer_brute_force_numpy(act, wfmt):
    """An independent numpy evaluation of the whole layer from the dequantised weights:
    dense matmuls, softmax over the top-k of a full sort, weighted sum."""
    w, L = _tiny_layer(act=act, wfmt=wfmt)
    x = synth.tokens(w, 16)
    res = L.forward(x)
    gu, dn = _dequant_all(L)
    xd = x.astype(np.float64)
    lg = res["logits"].astype(np.float64)
    out = np.zeros((16, L.d))
    for t in range(16):
        order = np.lexsort((np.arange(L.E), -lg[t]))[: L.k]
        sm = np.exp(lg[t, order] - lg[t, order].max())
        sm /= sm.sum()
        for j, e in enumerate(order):
            z = gu[e] @ xd[t]
            if act == "swiglu":
                g, u = z[: L.f], z[L.f:]
                h = g / (1 + np.exp(-g)) * u
            else:
                h = np.maximum(z, 0) ** 2
            out[t] += sm[j] * (dn[e] @ h)
    assert np.allclose(res["out"], out, rtol=1e-9, atol=1e-12 * np.abs(out).max())


def test_precomputed_routing_is_used_as_given():
    w, L = _tiny_layer()
    x = synth.tokens(w, 8)
    idx, wts = synth.zipf_routing(8, L.E, L.k, seed_tag="pin")
    res = L.forward(x, idx_in=idx, w_in=wts)
    assert np.array_equal(res["idx"], idx) and np.array_equal(res["w"], wts.astype(np.float64))
    base = L.forward(x)
    swap = L.forward(x, idx_in=base["idx"], w_in=base["w"].astype(np.float32))
    assert np.allclose(swap["out"], base["out"], rtol=1e-6, atol=1e-9)


def test_relu2_bias_channel_gives_the_page_zero_fraction():
    """Nemotron page, step 4: ~92.5 % of neurons are exactly zero after ReLU^2.  The
    synthetic latent layer gets that from its bias channel; measured on the oracle."""
    w = synth.WORKLOADS["nemotron"]
    E_s = 4
    gu, dn, gts, dts = [], [], [], []
    for e in range(E_s):
        a, b = synth.expert_weights(w, 0, e)
        qa, sa = oracle.nvfp4_quantize(a)
        qb, sb = oracle.nvfp4_quantize(b)
        gu.append(qa), dn.append(qb), gts.append(sa), dts.append(sb)
    L = oracle.Layer(w.d, w.f, E_s, 2, oracle.ACT_RELU2, oracle.W_NVFP4,
                     np.zeros((w.d, E_s), np.float32), gu, dn, gts, dts)
    x = synth.tokens(w, 16)
    idx = np.tile(np.arange(2, dtype=np.int32), (16, 1))
    res = L.forward(x, idx_in=idx, w_in=np.full((16, 2), 0.5, np.float32))
    frac = float((res["h"] == 0).mean())
    assert abs(frac - 0.925) < 0.015, frac


# ------------------------------------------------------------------ activation-quantised Q8_0
# The CPU engines' Q8_0 x Q8_0 path (Xeon page, "A three-step fix" and "Narrowing down the
# cause"): the expert's input vector is quantised with the same Q8_0 block codec as the
# weights, and each weight row is dotted with it block by block: exact integer code sums,
# both fp16 scales.  Pinned below by definitions written from the codec alone.
def test_q8_0_vec_dot_is_the_dot_of_the_dequantised_rows():
    g = np.random.default_rng(11)
    for cols in (32, 256, 2816):
        a = oracle.q8_0_quantize((g.standard_normal((1, cols)) * 0.02).astype(np.float32))
        b = oracle.q8_0_quantize(g.standard_normal((1, cols)).astype(np.float32))
        da, db = oracle.q8_0_dequant(a, 1, cols)[0], oracle.q8_0_dequant(b, 1, cols)[0]
        terms = da * db                       # each exact in fp64
        got = oracle.q8_0_vec_dot(a, b)
        assert abs(got - math.fsum(terms)) <= 1e-13 * np.abs(terms).sum()


def test_q8_0_vec_dot_closed_forms():
    nb = 4
    ones = oracle.q8_0_quantize(np.full((1, 32 * nb), 1.0, np.float32))
    twos = oracle.q8_0_quantize(np.full((1, 32 * nb), 2.0, np.float32))
    # constant blocks code to +127 with the fp16 of amax/127 as scale
    s1 = oracle.f16_bits_to_f64(oracle.f32_to_f16_bits(np.float32(1.0) / np.float32(127.0)))
    s2 = oracle.f16_bits_to_f64(oracle.f32_to_f16_bits(np.float32(2.0) / np.float32(127.0)))
    assert oracle.q8_0_vec_dot(ones, twos) == nb * 32 * 127 * 127 * s1 * s2
    # alternating signs against a constant: every block's integer sum is zero
    alt = np.tile(np.array([1.0, -1.0], np.float32), 16 * nb)[None]
    assert oracle.q8_0_vec_dot(ones, oracle.q8_0_quantize(alt)) == 0.0
    # a zero activation block has scale 0 and codes 0
    zero = oracle.q8_0_quantize(np.zeros((1, 32 * nb), np.float32))
    assert oracle.q8_0_vec_dot(ones, zero) == 0.0
    # one block of x against e_i picks the weight's code i times both scales
    x = np.zeros((1, 32), np.float32)
    x[0, 5] = 3.0
    w = (np.arange(32, dtype=np.float32) - 16.0)[None] * 0.01
    qw, qx = oracle.q8_0_quantize(w), oracle.q8_0_quantize(x)
    sw = oracle.f16_bits_to_f64(int(qw[0]) | (int(qw[1]) << 8))
    sx = oracle.f16_bits_to_f64(int(qx[0]) | (int(qx[1]) << 8))
    assert oracle.q8_0_vec_dot(qw, qx) == float(np.int8(qw[2 + 5])) * 127 * sw * sx


def test_q8_0_activation_quantisation_error_bound():
    """|dot(Q(w), Q(x)) - dot(deq(Q(w)), x)| is bounded by the codec: each element of x is
    off by at most d/2 (rounding with the fp32 scale d) plus 127 |d - fp16(d)| (the stored
    scale), with d = amax(block)/127."""
    g = np.random.default_rng(12)
    cols = 1024
    for trial in range(5):
        w = (g.standard_normal((1, cols)) * 0.02).astype(np.float32)
        x = (g.standard_normal((1, cols)) * (10.0 ** (trial - 2))).astype(np.float32)
        qw, qx = oracle.q8_0_quantize(w), oracle.q8_0_quantize(x)
        dw = oracle.q8_0_dequant(qw, 1, cols)[0]
        exact = math.fsum(dw * x[0].astype(np.float64))
        bound = 0.0
        for b in range(cols // 32):
            blk = x[0, 32 * b: 32 * b + 32]
            d = np.float32(np.abs(blk).max()) / np.float32(127.0)
            dh = oracle.f16_bits_to_f64(oracle.f32_to_f16_bits(d))
            e = float(d) / 2 + 127 * abs(float(d) - dh) + 1e-7 * float(d)
            bound += np.abs(dw[32 * b: 32 * b + 32]).sum() * e
        err = abs(oracle.q8_0_vec_dot(qw, qx) - exact)
        assert err <= bound, (trial, err, bound)
        assert err > 0.0   # the activations really are quantised


def test_activation_quantised_layer_composes_the_pinned_pieces():
    """The layer with act_q8: x quantised per token, gate/up by block dots, SwiGLU in fp64,
    h rounded to fp32 and quantised, down by block dots, the fixed-order combine.  Rebuilt
    here from the pinned codec (quantise, dequantise) and plain numpy dots."""
    w, L = _tiny_layer()
    T = 6
    x = synth.tokens(w, T)
    idx, wts = synth.zipf_routing(T, L.E, L.k, seed_tag="q8act")
    res = L.forward(x, idx_in=idx, w_in=wts, act_q8=True)
    gu, dn = _dequant_all(L)
    out = np.zeros((T, L.d))
    for t in range(T):
        xq = oracle.q8_0_dequant(oracle.q8_0_quantize(x[t][None].astype(np.float32)), 1, L.d)[0]
        for j in range(L.k):
            e = int(idx[t, j])
            z = gu[e] @ xq
            g_, u_ = z[: L.f], z[L.f:]
            h = g_ / (1 + np.exp(-g_)) * u_
            hq = oracle.q8_0_dequant(oracle.q8_0_quantize(h.astype(np.float32)[None]), 1, L.f)[0]
            out[t] += float(wts[t, j]) * (dn[e] @ hq)
    assert np.allclose(res["out"], out, rtol=1e-9, atol=1e-12 * np.abs(out).max())
    # against the float-activation layer: the same routing, close but not equal
    ref = L.forward(x, idx_in=idx, w_in=wts)
    rel = np.abs(res["out"] - ref["out"]).max() / np.sqrt((ref["out"] ** 2).mean())
    assert 0.0 < rel < 0.05, rel


def test_activation_quantised_path_refuses_nvfp4():
    w, L = _tiny_layer(act="relu2", wfmt="nvfp4")
    with pytest.raises(ValueError):
        L.forward(synth.tokens(w, 2), act_q8=True)


# ------------------------------------------------------------------ per-channel int8 (NEXT-4)
# Inferentia page, 'Wall 1: the memory math': the experts quantised to int8 with one scale per
# output channel.  The page gives no recipe; the oracle takes s = amax(row)/127 in fp32 and
# q = round(x/s), half away from zero, and stores the codes row-major, then the fp32 scales.
def test_int8_per_channel_bytes_match_page():
    w = synth.WORKLOADS["gemma"]
    params = w.layers * w.E * (w.rows_gu * w.d + w.d * w.f)
    assert abs(params * 2 / 2 / 1e9 - page("gemma_bf16_experts_gb_per_core_tp2")) < 0.05   # bf16, two cores
    per_expert = oracle.int8pc_bytes(w.rows_gu, w.d) + oracle.int8pc_bytes(w.d, w.f)
    assert per_expert == (w.rows_gu * w.d + w.d * w.f) + 4 * (w.rows_gu + w.d)
    per_rank = w.layers * w.E * per_expert / 2
    assert abs(per_rank / 1e9 - page("gemma_int8_experts_gb_per_rank")) / page("gemma_int8_experts_gb_per_rank") < 0.01


def test_int8_per_channel_hand_rows():
    m = np.array([[0.0, 0.0, 0.0, 0.0],           # all zero: scale 0, codes 0
                  [0.3, 0.3, -0.3, 0.3],          # constant magnitude: codes +-127
                  [127.0, 2.5, -2.5, 0.5],        # scale exactly 1: half-way values round away
                  [127.0, -0.49, 63.5, -126.5]], np.float32)
    q = oracle.int8pc_quantize(m)
    codes = q[:16].view(np.int8).reshape(4, 4)
    scales = q[16:].view(np.float32)
    assert (codes[0] == 0).all() and scales[0] == 0.0
    assert list(codes[1]) == [127, 127, -127, 127] and scales[1] == np.float32(0.3) / np.float32(127.0)
    assert list(codes[2]) == [127, 3, -3, 1] and scales[2] == 1.0
    assert list(codes[3]) == [127, 0, 64, -127] and scales[3] == 1.0
    assert np.array_equal(oracle.int8pc_dequant(q, 4, 4), codes.astype(np.float64) * scales[:, None].astype(np.float64))


def test_int8_per_channel_scale_is_per_row_and_error_bound():
    g = np.random.default_rng(21)
    m = (g.standard_normal((16, 704)) * np.logspace(-3, 1, 16)[:, None]).astype(np.float32)
    q = oracle.int8pc_quantize(m)
    scales = q[16 * 704:].view(np.float32).astype(np.float64)
    amax = np.abs(m).max(axis=1)
    assert np.array_equal(scales.astype(np.float32), (amax / np.float32(127.0)).astype(np.float32))
    err = np.abs(oracle.int8pc_dequant(q, 16, 704) - m.astype(np.float64))
    assert (err <= scales[:, None] * (0.5 + 1e-6)).all()
    # a per-tensor scale would leave the small rows with almost no resolution
    assert (err.max(axis=1) <= amax / 127 * 0.5 * (1 + 1e-6)).all()


def test_int8_per_channel_layer_brute_force():
    """The layer over per-channel int8 experts against a numpy evaluation from the
    dequantised weights (the same expert arithmetic as the other formats)."""
    w = synth.Workload("int8pc", d=256, f=512, E=8, k=2, act="swiglu", wfmt="q8_0", x_dtype="f32", layers=1,
                       rms_norm_input=False)
    gu, dn = [], []
    for e in range(w.E):
        a, b = synth.expert_weights(w, 0, e)
        gu.append(oracle.int8pc_quantize(a))
        dn.append(oracle.int8pc_quantize(b))
    L = oracle.Layer(w.d, w.f, w.E, w.k, oracle.ACT_SWIGLU, oracle.W_INT8PC, synth.router_weight(w), gu, dn)
    x = synth.tokens(w, 8)
    res = L.forward(x)
    lg = res["logits"].astype(np.float64)
    out = np.zeros((8, w.d))
    for t in range(8):
        order = np.lexsort((np.arange(w.E), -lg[t]))[: w.k]
        sm = np.exp(lg[t, order] - lg[t, order].max())
        sm /= sm.sum()
        for j, e in enumerate(order):
            z = oracle.int8pc_dequant(gu[e], 2 * w.f, w.d) @ x[t].astype(np.float64)
            h = z[: w.f] / (1 + np.exp(-z[: w.f])) * z[w.f:]
            out[t] += sm[j] * (oracle.int8pc_dequant(dn[e], w.d, w.f) @ h)
    assert np.allclose(res["out"], out, rtol=1e-9, atol=1e-12 * np.abs(out).max())


def test_oracle_results_do_not_depend_on_the_thread_count():
    """Xeon page, 'Clues in the garbled output' and 'Narrowing down the cause': single- and
    multi-thread runs are byte-identical.
    Every oracle output is computed by one thread in a fixed order, so the thread count of
    its parallel loops must not change a bit of the result (codecs and the layer)."""
    threads = oracle.num_threads()
    w, L = _tiny_layer()
    x = synth.tokens(w, 12)
    m = (np.random.default_rng(31).standard_normal((96, 2816)) * 0.02).astype(np.float32)
    runs = []
    try:
        for n in (1, 2, max(threads, 3)):
            oracle.set_num_threads(n)
            r = L.forward(x)
            q8 = oracle.q8_0_quantize(m)
            nv, _ = oracle.nvfp4_quantize(m)
            runs.append((r["out"].tobytes(), r["h"].tobytes(), r["idx"].tobytes(), q8.tobytes(), nv.tobytes()))
    finally:
        oracle.set_num_threads(threads)
    assert runs[0] == runs[1] == runs[2]
