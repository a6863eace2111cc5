"""CPU oracle for the routed quantized-expert MoE layer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product path (the CUDA library and its Python binding)
never does, and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain scalar C, fp64 accumulation); this
module compiles it with gcc on first use and wraps it for numpy arrays.  Each wrapper
names the C function it calls; the C file cites the page passages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

ACT_SWIGLU = 0
ACT_RELU2 = 1
W_Q8_0 = 0
W_NVFP4 = 1
W_INT8PC = 2    # per-channel int8: codes row-major, then one fp32 scale per row


def build_oracle(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so (gcc, -O2 -ffp-contract=off, OpenMP when
    available).  The library is written to a temporary name and renamed into place, so
    concurrent builders never see a half-written file."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    fd, tmp = tempfile.mkstemp(prefix=".liboracle.", suffix=".so", dir=_HERE)
    os.close(fd)
    try:
        try:
            subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
        os.replace(tmp, _LIB)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build_oracle())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


def _declare(L: ctypes.CDLL) -> None:
    sig = {
        "orc_num_threads": (_I, []),
        "orc_set_num_threads": (None, [_I]),
        "orc_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
        "orc_f16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
        "orc_f32_to_e4m3": (ctypes.c_uint8, [ctypes.c_float]),
        "orc_e4m3_to_f64": (ctypes.c_double, [ctypes.c_uint8]),
        "orc_f32_to_e2m1": (ctypes.c_uint8, [ctypes.c_float]),
        "orc_e2m1_to_f64": (ctypes.c_double, [ctypes.c_uint8]),
        "orc_q8_0_bytes": (_I64, [_I64, _I64]),
        "orc_nvfp4_bytes": (_I64, [_I64, _I64]),
        "orc_int8pc_bytes": (_I64, [_I64, _I64]),
        "orc_int8pc_quantize": (None, [_P, _I64, _I64, _P]),
        "orc_int8pc_dequant": (None, [_P, _I64, _I64, _P]),
        "orc_q8_0_quantize": (None, [_P, _I64, _I64, _P]),
        "orc_q8_0_dequant": (None, [_P, _I64, _I64, _P]),
        "orc_q8_0_vec_dot": (ctypes.c_double, [_P, _P, _I64]),
        "orc_q8_0_permute": (None, [_P, _I64, _I64, _I, _P]),
        "orc_int8pc_permute": (None, [_P, _I64, _I64, _I, _P]),
        "orc_nvfp4_tensor_scale": (ctypes.c_float, [_P, _I64, _I64]),
        "orc_nvfp4_quantize": (None, [_P, _I64, _I64, _P, _P]),
        "orc_nvfp4_dequant": (None, [_P, _I64, _I64, ctypes.c_float, _P]),
        "orc_nvfp4_permute_panels": (None, [_P, _I64, _I64, _I, _P]),
        "orc_nvfp4_permute_neuron": (None, [_P, _I64, _I64, _I, _P]),
        "orc_router_logits": (None, [_P, _I, _P, _I64, _I64, _I64, _P]),
        "orc_topk_softmax": (None, [_P, _I64, _I64, _I, _P, _P]),
        "orc_permute": (None, [_P, _I64, _I, _I64, _P, _P, _P]),
        "orc_mul_mat_id": (None, [_P, _I64, _I64, _I64, _I64, _P, _I64, _I, _P, _P]),
        "orc_silu": (ctypes.c_double, [ctypes.c_double]),
        "orc_fused_mul_silu": (None, [_P, _P, _I64, _P]),
        "orc_layer_forward": (_I, [_P, _P, _I, _I64, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
        "orc_layer_forward_ex": (_I, [_P, _P, _I, _I64, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
        "orc_layer_forward_dense_experts": (None, [_P, _P, _I, _I64, _P, _P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on."""
    lib().orc_set_num_threads(int(n))


# ----------------------------------------------------------------------------- codecs
def f32_to_f16_bits(v: float) -> int:
    return int(lib().orc_f32_to_f16(float(v)))


def f16_bits_to_f64(h: int) -> float:
    return float(lib().orc_f16_to_f64(int(h)))


def f32_to_e4m3(v: float) -> int:
    return int(lib().orc_f32_to_e4m3(float(v)))


def e4m3_to_f64(b: int) -> float:
    return float(lib().orc_e4m3_to_f64(int(b)))


def f32_to_e2m1(v: float) -> int:
    return int(lib().orc_f32_to_e2m1(float(v)))


def e2m1_to_f64(c: int) -> float:
    return float(lib().orc_e2m1_to_f64(int(c)))


# ----------------------------------------------------------------------------- sizes
def q8_0_bytes(rows: int, cols: int) -> int:
    return int(lib().orc_q8_0_bytes(rows, cols))


def int8pc_bytes(rows: int, cols: int) -> int:
    return int(lib().orc_int8pc_bytes(rows, cols))


def int8pc_quantize(src: np.ndarray) -> np.ndarray:
    """orc_int8pc_quantize of one fp32 matrix [rows][cols]: per-channel int8 bytes."""
    src = np.ascontiguousarray(src, dtype=np.float32)
    rows, cols = src.shape
    out = np.empty(int8pc_bytes(rows, cols), dtype=np.uint8)
    lib().orc_int8pc_quantize(_ptr(src), rows, cols, _ptr(out))
    return out


def int8pc_dequant(q: np.ndarray, rows: int, cols: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.empty((rows, cols), dtype=np.float64)
    lib().orc_int8pc_dequant(_ptr(q), rows, cols, _ptr(out))
    return out


def int8pc_to_device(canon: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """orc_int8pc_permute(+1): canonical per-channel int8 bytes -> the device layout (the row
    scales first, then panels of 32 columns)."""
    canon = np.ascontiguousarray(canon, dtype=np.uint8)
    out = np.empty_like(canon)
    lib().orc_int8pc_permute(_ptr(canon), rows, cols, 1, _ptr(out))
    return out


def int8pc_from_device(dev: np.ndarray, rows: int, cols: int) -> np.ndarray:
    dev = np.ascontiguousarray(dev, dtype=np.uint8)
    out = np.empty_like(dev)
    lib().orc_int8pc_permute(_ptr(dev), rows, cols, -1, _ptr(out))
    return out


def nvfp4_bytes(rows: int, cols: int) -> int:
    return int(lib().orc_nvfp4_bytes(rows, cols))


# ----------------------------------------------------------------------------- Q8_0
def q8_0_quantize(src: np.ndarray) -> np.ndarray:
    """orc_q8_0_quantize on the last two dims of src (fp32); canonical blocks."""
    src = np.ascontiguousarray(src, dtype=np.float32)
    rows, cols = src.shape[-2], src.shape[-1]
    lead = src.shape[:-2]
    n = int(np.prod(lead)) if lead else 1
    per = q8_0_bytes(rows, cols)
    out = np.empty((n, per), dtype=np.uint8)
    flat = src.reshape(n, rows, cols)
    for i in range(n):
        m = np.ascontiguousarray(flat[i])
        lib().orc_q8_0_quantize(_ptr(m), rows, cols, _ptr(out[i]))
    return out.reshape(*lead, per) if lead else out[0]


def q8_0_dequant(q: np.ndarray, rows: int, cols: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.empty((rows, cols), dtype=np.float64)
    lib().orc_q8_0_dequant(_ptr(q), rows, cols, _ptr(out))
    return out


def q8_0_vec_dot(a: np.ndarray, b: np.ndarray) -> float:
    """orc_q8_0_vec_dot: the activation-quantised dot product of two rows given as canonical
    Q8_0 bytes (the same number of blocks each)."""
    a = np.ascontiguousarray(a, dtype=np.uint8).ravel()
    b = np.ascontiguousarray(b, dtype=np.uint8).ravel()
    if a.size != b.size or a.size % 34:
        raise ValueError("q8_0_vec_dot: two rows of whole Q8_0 blocks of equal length")
    return float(lib().orc_q8_0_vec_dot(_ptr(a), _ptr(b), a.size // 34))


def q8_0_to_device(canon: np.ndarray, rows: int, cols: int) -> np.ndarray:
    canon = np.ascontiguousarray(canon, dtype=np.uint8)
    out = np.empty_like(canon)
    lib().orc_q8_0_permute(_ptr(canon), rows, cols, 1, _ptr(out))
    return out


def q8_0_from_device(dev: np.ndarray, rows: int, cols: int) -> np.ndarray:
    dev = np.ascontiguousarray(dev, dtype=np.uint8)
    out = np.empty_like(dev)
    lib().orc_q8_0_permute(_ptr(dev), rows, cols, -1, _ptr(out))
    return out


# ----------------------------------------------------------------------------- NVFP4
def nvfp4_quantize(src: np.ndarray) -> tuple[np.ndarray, float]:
    """orc_nvfp4_quantize on one matrix: (canonical bytes, tensor scale)."""
    src = np.ascontiguousarray(src, dtype=np.float32)
    rows, cols = src.shape
    out = np.empty(nvfp4_bytes(rows, cols), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    lib().orc_nvfp4_quantize(_ptr(src), rows, cols, _ptr(out), _ptr(ts))
    return out, float(ts[0])


def nvfp4_dequant(q: np.ndarray, rows: int, cols: int, tscale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.empty((rows, cols), dtype=np.float64)
    lib().orc_nvfp4_dequant(_ptr(q), rows, cols, float(np.float32(tscale)), _ptr(out))
    return out


def nvfp4_to_panels(canon: np.ndarray, rows: int, cols: int) -> np.ndarray:
    canon = np.ascontiguousarray(canon, dtype=np.uint8)
    out = np.empty_like(canon)
    lib().orc_nvfp4_permute_panels(_ptr(canon), rows, cols, 1, _ptr(out))
    return out


def nvfp4_from_panels(dev: np.ndarray, rows: int, cols: int) -> np.ndarray:
    dev = np.ascontiguousarray(dev, dtype=np.uint8)
    out = np.empty_like(dev)
    lib().orc_nvfp4_permute_panels(_ptr(dev), rows, cols, -1, _ptr(out))
    return out


def nvfp4_to_neuron(canon: np.ndarray, rows: int, cols: int) -> np.ndarray:
    canon = np.ascontiguousarray(canon, dtype=np.uint8)
    out = np.empty_like(canon)
    lib().orc_nvfp4_permute_neuron(_ptr(canon), rows, cols, 1, _ptr(out))
    return out


def nvfp4_from_neuron(dev: np.ndarray, rows: int, cols: int) -> np.ndarray:
    dev = np.ascontiguousarray(dev, dtype=np.uint8)
    out = np.empty_like(dev)
    lib().orc_nvfp4_permute_neuron(_ptr(dev), rows, cols, -1, _ptr(out))
    return out


# ----------------------------------------------------------------------------- routing
def _x_arg(x: np.ndarray) -> tuple[np.ndarray, int]:
    """fp32 arrays pass as-is (xt=0); bf16 inputs are passed as their uint16 bits (xt=1)."""
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), 0
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), 1
    raise TypeError("x must be float32 or uint16 (bf16 bits)")


def router_logits(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    xa, xt = _x_arg(x)
    W = np.ascontiguousarray(W, dtype=np.float32)
    T, d = xa.shape
    E = W.shape[1]
    out = np.empty((T, E), dtype=np.float32)
    lib().orc_router_logits(_ptr(xa), xt, _ptr(W), T, d, E, _ptr(out))
    return out


def topk_softmax(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    lib().orc_topk_softmax(_ptr(logits), T, E, k, _ptr(idx), _ptr(w))
    return idx, w


def permute(idx: np.ndarray, E: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    pos = np.empty(T * k, dtype=np.int32)
    lib().orc_permute(_ptr(idx), T, k, E, _ptr(offsets), _ptr(perm), _ptr(pos))
    return offsets, perm, pos


# ----------------------------------------------------------------------------- experts
def mul_mat_id(W: list[np.ndarray], row0: int, nrows: int, x: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """orc_mul_mat_id: W is a list of E dequantised fp64 matrices [ld_rows][cols];
    returns [T, k, nrows] for the row view row0..row0+nrows-1."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    mats = [np.ascontiguousarray(m, dtype=np.float64) for m in W]
    ld_rows, cols = mats[0].shape
    table = (ctypes.c_void_p * len(mats))(*[m.ctypes.data for m in mats])
    out = np.empty((T, k, nrows), dtype=np.float64)
    lib().orc_mul_mat_id(ctypes.cast(table, ctypes.c_void_p), ld_rows, cols, row0, nrows, _ptr(x), T, k,
                         _ptr(ids), _ptr(out))
    return out


def fused_mul_silu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    gate = np.ascontiguousarray(gate, dtype=np.float64)
    up = np.ascontiguousarray(up, dtype=np.float64)
    out = np.empty_like(gate)
    lib().orc_fused_mul_silu(_ptr(gate), _ptr(up), gate.size, _ptr(out))
    return out


class _OrcLayer(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int64), ("f", ctypes.c_int64), ("E", ctypes.c_int64),
        ("k", ctypes.c_int), ("act", ctypes.c_int), ("wfmt", ctypes.c_int),
        ("router_w", ctypes.c_void_p), ("gate_up", ctypes.c_void_p), ("down", ctypes.c_void_p),
        ("gate_up_tscale", ctypes.c_void_p), ("down_tscale", ctypes.c_void_p),
    ]


class Layer:
    """Weights of one layer for the oracle, in canonical quantised bytes.

    gate_up[e] / down[e] may be None for experts the routing never selects (a
    sampled full-size check only quantises the experts it needs)."""

    def __init__(self, d, f, E, k, act, wfmt, router_w, gate_up, down, gate_up_tscale=None, down_tscale=None):
        self.d, self.f, self.E, self.k, self.act, self.wfmt = d, f, E, k, act, wfmt
        self.router_w = np.ascontiguousarray(router_w, dtype=np.float32)
        self.gate_up = [None if g is None else np.ascontiguousarray(g, dtype=np.uint8) for g in gate_up]
        self.down = [None if g is None else np.ascontiguousarray(g, dtype=np.uint8) for g in down]
        self.gate_up_tscale = None if gate_up_tscale is None else np.ascontiguousarray(gate_up_tscale, np.float32)
        self.down_tscale = None if down_tscale is None else np.ascontiguousarray(down_tscale, np.float32)

    def _struct(self):
        gu = (ctypes.c_void_p * self.E)(*[0 if g is None else g.ctypes.data for g in self.gate_up])
        dn = (ctypes.c_void_p * self.E)(*[0 if g is None else g.ctypes.data for g in self.down])
        s = _OrcLayer(self.d, self.f, self.E, self.k, self.act, self.wfmt, self.router_w.ctypes.data,
                      ctypes.cast(gu, ctypes.c_void_p), ctypes.cast(dn, ctypes.c_void_p),
                      _ptr(self.gate_up_tscale), _ptr(self.down_tscale))
        return s, (gu, dn)

    def forward(self, x: np.ndarray, idx_in=None, w_in=None, sparse_down: bool = True, act_q8: bool = False) -> dict:
        """orc_layer_forward_ex: returns logits (when routed here), idx, w, offsets, perm, pos,
        h [T*k, f] and y [T*k, d] in pair order, and out [T, d] (fp64).  act_q8: the
        activation-quantised expert path (each expert input quantised to Q8_0 blocks, then
        Q8_0 x Q8_0 block dots; Q8_0 weights and f a multiple of 32 only)."""
        xa, xt = _x_arg(x)
        T = xa.shape[0]
        k, E, d, f = self.k, self.E, self.d, self.f
        P = T * k
        res = {
            "logits": None if idx_in is not None else np.empty((T, E), np.float32),
            "idx": np.empty((T, k), np.int32), "w": np.empty((T, k), np.float64),
            "offsets": np.empty(E + 1, np.int32), "perm": np.empty(P, np.int32), "pos": np.empty(P, np.int32),
            "h": np.empty((P, f), np.float64), "y": np.empty((P, d), np.float64),
            "out": np.empty((T, d), np.float64),
        }
        ii = None if idx_in is None else np.ascontiguousarray(idx_in, np.int32)
        ww = None if w_in is None else np.ascontiguousarray(w_in, np.float32)
        s, keep = self._struct()
        rc = lib().orc_layer_forward_ex(ctypes.byref(s), _ptr(xa), xt, T, _ptr(ii), _ptr(ww), int(sparse_down),
                                        int(act_q8), _ptr(res["logits"]), _ptr(res["idx"]), _ptr(res["w"]),
                                        _ptr(res["offsets"]), _ptr(res["perm"]), _ptr(res["pos"]), _ptr(res["h"]),
                                        _ptr(res["y"]), _ptr(res["out"]))
        del keep
        if rc == -2:
            raise ValueError("oracle: the activation-quantised path needs Q8_0 weights and f a multiple of 32")
        if rc != 0:
            raise ValueError("oracle: routing selected an expert whose weights were not supplied")
        return res

    def forward_dense_experts(self, x: np.ndarray, wfull: np.ndarray) -> np.ndarray:
        xa, xt = _x_arg(x)
        T = xa.shape[0]
        wfull = np.ascontiguousarray(wfull, np.float64)
        out = np.empty((T, self.d), np.float64)
        s, keep = self._struct()
        lib().orc_layer_forward_dense_experts(ctypes.byref(s), _ptr(xa), xt, T, _ptr(wfull), _ptr(out))
        del keep
        return out
