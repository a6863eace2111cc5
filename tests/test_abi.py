"""The C ABI on the host: the library loads, exports every symbol include/moe.h declares,
and rejects bad arguments with the documented status before launching anything.
No test here touches a GPU."""
import ctypes
import os
import re
import shutil

import pytest

from quantized_routed_expert_softmax_gb300 import native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(native.LIB_PATH):
        if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("libmoe.so not built and no nvcc to build it")
        from quantized_routed_expert_softmax_gb300 import build
        build.build()
    return native.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    declared = header_functions()
    assert declared == sorted(native.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def test_abi_version_and_status_strings(L):
    assert L.moe_abi_version() == 10300
    for s in range(8):
        assert L.moe_status_string(s).decode().startswith(native.STATUS_NAMES[s])


def test_size_queries(L):
    assert L.moe_q8_0_bytes(1408, 2816) == 4_212_736
    assert L.moe_q8_0_bytes(2816, 704) == 2_106_368
    assert L.moe_nvfp4_bytes(2688, 1024) + L.moe_nvfp4_bytes(1024, 2688) == 3_096_576
    assert L.moe_q8_0_bytes(10, 33) == 0 and L.moe_nvfp4_bytes(0, 64) == 0
    assert L.moe_router_workspace_bytes(3, 8) == 256


FAKE = 0x10000   # an aligned address that is never dereferenced: validation fails first


def test_packer_validation(L):
    S = L.moe_quantize_q8_0
    assert S(None, 1, 32, 32, 1, FAKE, None) == 1
    assert S(FAKE, 1, 33, 32, 1, FAKE, None) == 2
    assert S(FAKE, 1, 32, 48, 1, FAKE, None) == 2
    assert S(FAKE, 1, 32, 32, 7, FAKE, None) == 1
    assert S(FAKE + 4, 1, 32, 32, 1, FAKE, None) == 3
    assert S(FAKE, 0, 32, 32, 1, FAKE, None) == 0          # nothing to do, nothing launched
    P = L.moe_pack_nvfp4
    assert P(FAKE, 1, 32, 32, 1, FAKE, FAKE, None) == 2      # cols must be a multiple of 64
    assert P(FAKE, 1, 32, 64, 1, FAKE, None, None) == 1
    assert P(FAKE, 1, 32, 64, 9, FAKE, FAKE, None) == 1


def test_activation_quantiser_validation(L):
    Q = L.moe_quantize_act_q8_0
    assert Q(None, 0, 4, 64, FAKE, None) == 1
    assert Q(FAKE, 2, 4, 64, FAKE, None) == 1       # bad dtype
    assert Q(FAKE, 0, 4, 48, FAKE, None) == 2       # cols a multiple of 32
    assert Q(FAKE + 4, 0, 4, 64, FAKE, None) == 3
    assert Q(FAKE, 1, 0, 64, FAKE, None) == 0       # nothing to do, nothing launched


def test_activation_quantised_layer_workspace(L):
    # the coded expert input takes T * d fp32 more
    plain = L.moe_layer_workspace_bytes(ctypes.byref(_desc()), 64)
    coded = L.moe_layer_workspace_bytes(ctypes.byref(_desc(act_quant=1)), 64)
    assert coded >= plain + 64 * 256 * 4


def test_router_validation(L):
    R = L.moe_router_topk
    assert R(FAKE, 0, FAKE, 4, 256, 8, 0, FAKE, FAKE, None, None, 0, None) == 1    # k = 0
    assert R(FAKE, 0, FAKE, 4, 256, 8, 9, FAKE, FAKE, None, None, 0, None) == 1    # k > E
    assert R(FAKE, 0, FAKE, 4, 200, 8, 2, FAKE, FAKE, None, None, 0, None) == 2    # d % 256
    assert R(FAKE, 0, FAKE, 4, 256, 8, 2, FAKE, FAKE, None, None, 0, None) == 4    # no workspace
    assert R(FAKE, 2, FAKE, 4, 256, 8, 2, FAKE, FAKE, None, None, 0, None) == 1    # bad dtype


def _desc(**kw):
    base = dict(d=256, f=512, E=8, k=2, act=0, wfmt=0, path=0, router_w=FAKE, w_gate_up=FAKE, w_down=FAKE,
                gate_up_tscale=None, down_tscale=None)
    base.update(kw)
    return native.LayerDesc(**base)


def test_layer_validation(L):
    F = L.moe_layer_forward
    ok = _desc()
    need = L.moe_layer_workspace_bytes(ctypes.byref(ok), 16)
    assert need > 0
    assert L.moe_layer_workspace_bytes(ctypes.byref(_desc(k=0)), 16) == 0
    cases = [
        (_desc(k=0), 1), (_desc(k=9), 1), (_desc(k=33, E=64), 1), (_desc(act=5), 1), (_desc(wfmt=3), 1),
        (_desc(d=200), 2), (_desc(f=500), 2), (_desc(E=6), 2), (_desc(E=2048), 2), (_desc(router_w=None), 1),
        (_desc(wfmt=1), 1),                       # NVFP4 needs tensor scales
        (_desc(w_down=FAKE + 8), 3),
        (_desc(act_quant=2), 1),                  # unknown activation quantiser
        (_desc(flags=4), 1),                      # unknown flag
        (_desc(flags=1, path=2), 5),              # host-resident weights cannot take the TMA path
        (_desc(flags=1), 1),                      # not host allocations the device can address
        (_desc(act_quant=1, wfmt=1, gate_up_tscale=FAKE, down_tscale=FAKE), 5),   # Q8_0 activations need Q8_0 weights
    ]
    for desc, want in cases:
        assert F(ctypes.byref(desc), FAKE, 0, 16, None, None, FAKE, FAKE, need, None, None) == want
    # routing supplied half-way, bad dtype, misaligned x
    assert F(ctypes.byref(ok), FAKE, 0, 16, FAKE, None, FAKE, FAKE, need, None, None) == 1
    assert F(ctypes.byref(ok), FAKE, 0, 16, None, FAKE, FAKE, FAKE, need, None, None) == 1
    # supplied routing must be 16-byte aligned, at one token (the one-kernel layer) and more
    for T in (1, 16):
        assert F(ctypes.byref(ok), FAKE, 0, T, FAKE + 4, FAKE, FAKE, FAKE, need, None, None) == 3
        assert F(ctypes.byref(ok), FAKE, 0, T, FAKE, FAKE + 8, FAKE, FAKE, need, None, None) == 3
    assert F(ctypes.byref(ok), FAKE, 3, 16, None, None, FAKE, FAKE, need, None, None) == 1
    assert F(ctypes.byref(ok), FAKE + 2, 0, 16, None, None, FAKE, FAKE, need, None, None) == 3
    # workspace: missing, misaligned, too small
    assert F(ctypes.byref(ok), FAKE, 0, 16, None, None, FAKE, None, need, None, None) == 4
    assert F(ctypes.byref(ok), FAKE, 0, 16, None, None, FAKE, FAKE + 16, need, None, None) == 3
    need1 = L.moe_layer_workspace_bytes(ctypes.byref(ok), 1)   # the exact need of one token
    assert F(ctypes.byref(ok), FAKE, 0, 1, None, None, FAKE, FAKE, need1 - 1, None, None) == 4
    # an empty batch returns OK without touching anything
    assert F(ctypes.byref(ok), FAKE, 0, 0, None, None, FAKE, None, 0, None, None) == 0


def test_workspace_grows_with_tokens(L):
    d = _desc()
    sizes = [L.moe_layer_workspace_bytes(ctypes.byref(d), T) for T in (1, 2, 8, 32, 33, 100, 4096)]
    assert sizes == sorted(sizes)


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "quantized_routed_expert_softmax_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "moe_oracle" not in text and "liboracle" not in text, fn


def test_stack_validation(L):
    two = (native.LayerDesc * 2)(_desc(), _desc())
    mixed = (native.LayerDesc * 2)(_desc(), _desc(f=256))
    need1 = L.moe_layer_workspace_bytes(ctypes.byref(_desc()), 1)
    eps = ctypes.c_float(1e-6)
    def call(descs, n, x=FAKE, xt=0, outs=FAKE, idx=None, w=None, ws=FAKE, nbytes=need1):
        return L.moe_stack_forward(descs, n, x or None, xt, eps, outs, None, idx, w, ws or None, nbytes, None)
    assert call(two, 0) == 1                       # no layers
    assert call(mixed, 2) == 2                     # layers of different shapes
    assert call(two, 2, x=0) == 1                  # NULL x
    assert call(two, 2, idx=FAKE) == 1             # idx without w
    assert call(two, 2, xt=3) == 1                 # bad dtype
    assert call(two, 2, x=FAKE + 2) == 3           # misaligned x
    assert call(two, 2, ws=0) == 4                 # no workspace
    assert call(two, 2, nbytes=need1 - 1) == 4     # workspace too small


def test_stack_launch_count_sums_its_layers(L):
    # without a GPU no layer takes the one-kernel path: the stack runs layer by layer, each
    # layer's own launches and a norm after each; a coded layer (two coding launches more) and
    # a plain one count their own launches
    one = L.moe_layer_forward_launches(ctypes.byref(_desc()), 1, 0)
    coded = L.moe_layer_forward_launches(ctypes.byref(_desc(act_quant=1)), 1, 0)
    assert one > 1 and coded == one + 2
    mixed = (native.LayerDesc * 3)(_desc(act_quant=1), _desc(), _desc())
    assert L.moe_stack_forward_launches(mixed, 3, 1) == (coded + 1) + 2 * (one + 1)
    assert L.moe_stack_forward_launches(mixed, 3, 0) == (coded + 1) + 2 * (one + 1) - 1
    same = (native.LayerDesc * 3)(_desc(), _desc(), _desc())
    assert L.moe_stack_forward_launches(same, 3, 1) == 3 * (one + 1)
