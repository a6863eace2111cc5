"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function here turns torch tensors into pointers and sizes, calls the C entry point
of the same name, and raises on a non-OK status.  All arithmetic runs in libmoe's CUDA
kernels; there is no fallback of any kind: if libmoe.so is missing or cannot load, the
import of the functions below fails loudly.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_SHAPE", 3: "MOE_ERR_ALIGNMENT",
                4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_UNSUPPORTED", 6: "MOE_ERR_CUDA", 7: "MOE_ERR_DEVICE_CHECK"}
ACT = {"swiglu": 0, "relu2": 1}
WFMT = {"q8_0": 0, "nvfp4": 1, "int8pc": 2}
DTYPE_F32, DTYPE_BF16 = 0, 1
LAYOUT = {"canonical": 0, "device": 1, "neuron": 2}
PATH = {"auto": 0, "gemv": 1, "gemm": 2}
ACT_QUANT = {"none": 0, "q8_0": 1}
FLAG_HOST_GATE_UP, FLAG_HOST_DOWN = 1, 2

# Every symbol include/moe.h declares.
EXPORTS = ["moe_q8_0_bytes", "moe_nvfp4_bytes", "moe_int8pc_bytes", "moe_quantize_q8_0", "moe_pack_nvfp4",
           "moe_quantize_int8pc", "moe_quantize_act_q8_0",
           "moe_router_workspace_bytes",
           "moe_router_topk", "moe_layer_workspace_bytes", "moe_layer_forward", "moe_rmsnorm_bf16",
           "moe_get_device_status", "moe_status_string", "moe_abi_version", "moe_layer_forward_launches",
           "moe_layer_forward_noalloc", "moe_layer_forward_noalloc_status", "moe_stack_forward",
           "moe_stack_forward_launches"]


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


class LayerDesc(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int64), ("f", ctypes.c_int64), ("E", ctypes.c_int64),
        ("k", ctypes.c_int32), ("act", ctypes.c_int32), ("wfmt", ctypes.c_int32), ("path", ctypes.c_int32),
        ("router_w", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
        ("gate_up_tscale", ctypes.c_void_p), ("down_tscale", ctypes.c_void_p),
        ("l2_prefetch", ctypes.c_void_p), ("l2_prefetch_bytes", ctypes.c_int64),
        ("act_quant", ctypes.c_int32), ("flags", ctypes.c_int32),
    ]


class Trace(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("logits", "idx", "w", "offsets", "perm", "pos", "h")] + [
        ("stage_events", ctypes.c_void_p * 5)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with quantized_routed_expert_softmax_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        sig = {
            "moe_q8_0_bytes": (SZ, [I64, I64]),
            "moe_nvfp4_bytes": (SZ, [I64, I64]),
            "moe_int8pc_bytes": (SZ, [I64, I64]),
            "moe_quantize_int8pc": (I32, [P, I64, I64, I64, I32, P, P]),
            "moe_quantize_q8_0": (I32, [P, I64, I64, I64, I32, P, P]),
            "moe_pack_nvfp4": (I32, [P, I64, I64, I64, I32, P, P, P]),
            "moe_quantize_act_q8_0": (I32, [P, I32, I64, I64, P, P]),
            "moe_router_workspace_bytes": (SZ, [I64, I64]),
            "moe_router_topk": (I32, [P, I32, P, I64, I64, I64, I32, P, P, P, P, SZ, P]),
            "moe_layer_workspace_bytes": (SZ, [ctypes.POINTER(LayerDesc), I64]),
            "moe_layer_forward": (I32, [ctypes.POINTER(LayerDesc), P, I32, I64, P, P, P, P, SZ,
                                        ctypes.POINTER(Trace), P]),
            "moe_rmsnorm_bf16": (I32, [P, I64, I64, ctypes.c_float, P, P]),
            "moe_get_device_status": (I32, [P, P, ctypes.POINTER(I32)]),
            "moe_status_string": (ctypes.c_char_p, [I32]),
            "moe_abi_version": (I32, []),
            "moe_layer_forward_launches": (I32, [ctypes.POINTER(LayerDesc), I64, I32]),
            "moe_layer_forward_noalloc": (I32, [ctypes.POINTER(LayerDesc), P, I32, I64, P, P, P, P]),
            "moe_layer_forward_noalloc_status": (I32, [P, ctypes.POINTER(I32)]),
            "moe_stack_forward": (I32, [ctypes.POINTER(LayerDesc), I32, P, I32, ctypes.c_float, P, P, P, P, P, SZ, P]),
            "moe_stack_forward_launches": (I32, [ctypes.POINTER(LayerDesc), I32, I32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise MoeError(fn, status)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def q8_0_bytes(rows: int, cols: int) -> int:
    return int(lib().moe_q8_0_bytes(rows, cols))


def nvfp4_bytes(rows: int, cols: int) -> int:
    return int(lib().moe_nvfp4_bytes(rows, cols))


def quantize_q8_0(src, layout: str = "device", out=None, stream=None):
    """moe_quantize_q8_0 on a device fp32 tensor [..., rows, cols] -> uint8 [n_mat, bytes]."""
    import torch
    rows, cols = src.shape[-2], src.shape[-1]
    n = src.numel() // (rows * cols)
    per = q8_0_bytes(rows, cols)
    if out is None:
        out = torch.empty((n, per), dtype=torch.uint8, device=src.device)
    _check("moe_quantize_q8_0", lib().moe_quantize_q8_0(_ptr(src), n, rows, cols, LAYOUT[layout], _ptr(out),
                                                         _stream(stream)))
    return out


def pack_nvfp4(src, layout: str = "device", out=None, tscale=None, stream=None):
    """moe_pack_nvfp4 on a device fp32 tensor [..., rows, cols] -> (uint8 [n_mat, bytes], fp32 [n_mat])."""
    import torch
    rows, cols = src.shape[-2], src.shape[-1]
    n = src.numel() // (rows * cols)
    per = nvfp4_bytes(rows, cols)
    if out is None:
        out = torch.empty((n, per), dtype=torch.uint8, device=src.device)
    if tscale is None:
        tscale = torch.empty(n, dtype=torch.float32, device=src.device)
    _check("moe_pack_nvfp4", lib().moe_pack_nvfp4(_ptr(src), n, rows, cols, LAYOUT[layout], _ptr(out),
                                                   _ptr(tscale), _stream(stream)))
    return out, tscale


def int8pc_bytes(rows: int, cols: int) -> int:
    return int(lib().moe_int8pc_bytes(rows, cols))


def quantize_int8pc(src, layout: str = "device", out=None, stream=None):
    """moe_quantize_int8pc: src fp32 [n, rows, cols] (or [rows, cols]) -> uint8 [n, bytes]."""
    import torch
    s3 = src if src.dim() == 3 else src.unsqueeze(0)
    n, rows, cols = s3.shape
    if out is None:
        out = torch.empty((n, int8pc_bytes(rows, cols)), dtype=torch.uint8, device=src.device)
    _check("moe_quantize_int8pc", lib().moe_quantize_int8pc(_ptr(s3), n, rows, cols, LAYOUT[layout], _ptr(out),
                                                             _stream(stream)))
    return out


def quantize_act_q8_0(x, out=None, stream=None):
    """moe_quantize_act_q8_0: x [rows, cols] fp32 or bf16 -> the Q8_0-coded values, fp32."""
    import torch
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    _check("moe_quantize_act_q8_0", lib().moe_quantize_act_q8_0(_ptr(x), _x_dtype(x), x.shape[0], x.shape[1],
                                                                 _ptr(out), _stream(stream)))
    return out


def _x_dtype(x) -> int:
    import torch
    if x.dtype == torch.float32:
        return DTYPE_F32
    if x.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError("x must be float32 or bfloat16")


def router_topk(x, W, k: int, return_logits: bool = False, stream=None):
    """moe_router_topk: (idx int32 [T,k], w fp32 [T,k][, logits fp32 [T,E]])."""
    import torch
    T, d = x.shape
    E = W.shape[1]
    idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    _check("moe_router_topk", lib().moe_router_topk(_ptr(x), _x_dtype(x), _ptr(W), T, d, E, k, _ptr(idx), _ptr(w),
                                                     _ptr(logits), None, 0, _stream(stream)))
    return (idx, w, logits) if return_logits else (idx, w)


def rmsnorm_bf16(x, eps: float = 1e-6, out=None, stream=None):
    import torch
    T, d = x.shape
    if out is None:
        out = torch.empty((T, d), dtype=torch.bfloat16, device=x.device)
    _check("moe_rmsnorm_bf16", lib().moe_rmsnorm_bf16(_ptr(x), T, d, ctypes.c_float(eps), _ptr(out), _stream(stream)))
    return out


def device_status(workspace, stream=None) -> int:
    """moe_get_device_status: the device error code a workspace holds (0 if none); reading
    clears it."""
    code = ctypes.c_int32(0)
    st = lib().moe_get_device_status(_ptr(workspace), _stream(stream), ctypes.byref(code))
    if st not in (MOE_OK, 7):
        raise MoeError("moe_get_device_status", st)
    return int(code.value)


class MoELayer:
    """Device weights of one layer plus its descriptor; calls moe_layer_forward.

    gate_up: uint8 [E, bytes] in the device layout (SwiGLU: rows 0..f-1 gate, f..2f-1 up)
    down:    uint8 [E, bytes] (Q8_0 device layout / NVFP4 neuron layout)
    router_w: fp32 [d, E]; tscales: fp32 [E] each (NVFP4).
    """

    def __init__(self, d, f, E, k, act, wfmt, router_w, gate_up, down, gate_up_tscale=None, down_tscale=None,
                 path: str = "auto", act_quant: str = "none", host_weights: str = "none"):
        self.d, self.f, self.E, self.k, self.act, self.wfmt = d, f, E, k, act, wfmt
        self.router_w, self.gate_up, self.down = router_w, gate_up, down
        self.gate_up_tscale, self.down_tscale = gate_up_tscale, down_tscale
        self.desc = LayerDesc(d, f, E, k, ACT[act], WFMT[wfmt], PATH[path], _ptr(router_w), _ptr(gate_up), _ptr(down),
                              _ptr(gate_up_tscale), _ptr(down_tscale))
        self.desc.act_quant = ACT_QUANT[act_quant]
        # host_weights: "none", "down" (the down stack in page-locked host memory) or "all"
        self.desc.flags = {"none": 0, "down": FLAG_HOST_DOWN, "all": FLAG_HOST_GATE_UP | FLAG_HOST_DOWN}[host_weights]
        self.host_resident = host_weights
        self._ws = None
        self._ws_tokens = 0

    def set_l2_prefetch(self, t) -> None:
        """Bytes (a device tensor, or None) that this layer pulls into L2 while its experts
        stream: in a stack, the next layer's router weights."""
        self._l2_prefetch = t
        self.desc.l2_prefetch = _ptr(t) if t is not None else None
        self.desc.l2_prefetch_bytes = 0 if t is None else t.numel() * t.element_size()

    def set_path(self, path: str) -> None:
        self.desc.path = PATH[path]

    def workspace_bytes(self, T_max: int) -> int:
        n = int(lib().moe_layer_workspace_bytes(ctypes.byref(self.desc), T_max))
        if n == 0:
            raise MoeError("moe_layer_workspace_bytes", 1)
        return n

    def workspace(self, T: int):
        """A zero-filled workspace for up to T tokens with the current descriptor (kept, and
        replaced by a larger one when T or the descriptor needs more)."""
        import torch
        need = self.workspace_bytes(T)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(need, dtype=torch.uint8, device=self.router_w.device)
            self._ws_tokens = T
        return self._ws

    def launches(self, T: int, routing_supplied: bool = False) -> int:
        """Kernels one forward launches (moe_layer_forward_launches)."""
        return int(lib().moe_layer_forward_launches(ctypes.byref(self.desc), T, int(routing_supplied)))

    def forward(self, x, idx_in=None, w_in=None, out=None, trace: dict | None = None, workspace=None, stream=None,
                stage_events=None):
        """moe_layer_forward.  trace: a dict filled with device copies of the intermediates.
        stage_events: up to 5 torch.cuda.Event (timing enabled, already recorded once so
        that the handle exists) recorded at the stage boundaries."""
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.d), dtype=torch.float32, device=x.device)
        if workspace is not None:
            ws = workspace
        elif T == 0:
            ws = None      # an empty batch launches nothing and needs no workspace
        else:
            ws = self.workspace(T)
        tr = None
        if trace is not None:
            P = T * self.k
            dev = x.device
            trace.update(
                logits=torch.empty((T, self.E), dtype=torch.float32, device=dev) if idx_in is None else None,
                idx=torch.empty((T, self.k), dtype=torch.int32, device=dev),
                w=torch.empty((T, self.k), dtype=torch.float32, device=dev),
                offsets=torch.empty(self.E + 1, dtype=torch.int32, device=dev),
                perm=torch.empty(P, dtype=torch.int32, device=dev),
                pos=torch.empty(P, dtype=torch.int32, device=dev),
                h=torch.empty((P, self.f), dtype=torch.float32, device=dev))
            tr = Trace(*[_ptr(trace[n]) for n in ("logits", "idx", "w", "offsets", "perm", "pos", "h")])
        if stage_events is not None:
            if tr is None:
                tr = Trace()
            for i, ev in enumerate(stage_events):
                tr.stage_events[i] = None if ev is None else ev.cuda_event
        st = lib().moe_layer_forward(ctypes.byref(self.desc), _ptr(x), _x_dtype(x), T, _ptr(idx_in), _ptr(w_in),
                                     _ptr(out), _ptr(ws), 0 if ws is None else ws.numel(),
                                     ctypes.byref(tr) if tr is not None else None,
                                     _stream(stream))
        _check("moe_layer_forward", st)
        return out

    def forward_noalloc(self, x, idx_in=None, w_in=None, out=None, stream=None):
        """moe_layer_forward_noalloc: the same forward with the library's fixed scratch
        instead of a workspace (for callers that cannot allocate device memory)."""
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.d), dtype=torch.float32, device=x.device)
        _check("moe_layer_forward_noalloc",
               lib().moe_layer_forward_noalloc(ctypes.byref(self.desc), _ptr(x), _x_dtype(x), T, _ptr(idx_in),
                                               _ptr(w_in), _ptr(out), _stream(stream)))
        return out

    @staticmethod
    def noalloc_status(stream=None) -> int:
        """moe_layer_forward_noalloc_status: the device error code the last no-allocation
        call on this device left (0 if none); reading clears it."""
        code = ctypes.c_int32(0)
        st = lib().moe_layer_forward_noalloc_status(_stream(stream), ctypes.byref(code))
        if st not in (MOE_OK, 7):
            raise MoeError("moe_layer_forward_noalloc_status", st)
        return int(code.value)

    def device_status(self, stream=None, workspace=None) -> int:
        """moe_get_device_status on this layer's workspace (or `workspace`): 0 or the device
        error code."""
        return device_status(self._ws if workspace is None else workspace, stream)


class MoEStack:
    """Layers of one shape called as a stack for one token (moe_stack_forward): each layer's
    input is the RMS-normalised (bf16) output of the previous one."""

    def __init__(self, layers, eps: float = 1e-6):
        self.layers = list(layers)
        self.eps = eps
        self.descs = (LayerDesc * len(self.layers))(*[l.desc for l in self.layers])
        self._ws = None

    def refresh(self) -> None:
        """Copy the layers' descriptors again (after set_path / set_l2_prefetch)."""
        self.descs = (LayerDesc * len(self.layers))(*[l.desc for l in self.layers])

    def workspace(self):
        import torch
        if self._ws is None:
            self._ws = torch.zeros(self.layers[0].workspace_bytes(1), dtype=torch.uint8,
                                   device=self.layers[0].router_w.device)
        return self._ws

    def launches(self, with_x_next: bool = False) -> int:
        return int(lib().moe_stack_forward_launches(self.descs, len(self.layers), int(with_x_next)))

    def forward(self, x, outs=None, x_next=None, routing: dict | None = None, workspace=None, stream=None):
        """x: [1, d] fp32 or bf16 on the device.  Returns outs fp32 [n_layers, d]; x_next
        (bf16 [n_layers, d]) and routing (dict with idx int32 / w fp32 [n_layers, k]) are
        filled when given."""
        import torch
        n, l0 = len(self.layers), self.layers[0]
        if outs is None:
            outs = torch.empty((n, l0.d), dtype=torch.float32, device=x.device)
        idx = w = None
        if routing is not None:
            idx = torch.empty((n, l0.k), dtype=torch.int32, device=x.device)
            w = torch.empty((n, l0.k), dtype=torch.float32, device=x.device)
            routing.update(idx=idx, w=w)
        ws = workspace if workspace is not None else self.workspace()
        _check("moe_stack_forward",
               lib().moe_stack_forward(self.descs, n, _ptr(x), _x_dtype(x), ctypes.c_float(self.eps), _ptr(outs),
                                       _ptr(x_next), _ptr(idx), _ptr(w), _ptr(ws), ws.numel(), _stream(stream)))
        return outs
