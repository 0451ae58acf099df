"""ctypes binding of libbgq.so (the C ABI in include/bgq.h).

Argument marshalling only: torch tensors supply device memory and the current
CUDA stream; every step of the computation runs in the library's kernels.
Function names follow the C entry points. Loading fails loudly if the
library has not been built (``__graft_entry__.build()`` or
``python -m bit_group_quantized_gb300.build``); there is no fallback.
"""

from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbgq.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(6)
DQ_INT, DQ_STANDARD, DQ_REORDERED, DQ_HOISTED = range(4)
GROUP = 64


class BGQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class bgq_qmatrix(C.Structure):
    _fields_ = [("q", C.c_void_p), ("sb", C.c_void_p), ("rows", C.c_int32), ("cols", C.c_int32),
                ("bits", C.c_int32), ("group", C.c_int32)]


class bgq_expert(C.Structure):
    _fields_ = [("gate", bgq_qmatrix), ("up", bgq_qmatrix), ("down", bgq_qmatrix)]


class bgq_moe_layer(C.Structure):
    _fields_ = [("d_model", C.c_int32), ("d_ff", C.c_int32), ("n_experts", C.c_int32), ("top_k", C.c_int32),
                ("bits", C.c_int32), ("group", C.c_int32), ("router", C.c_void_p), ("shared_gate", C.c_void_p),
                ("expert_q", C.c_void_p), ("expert_sb", C.c_void_p), ("expert_q_stride", C.c_int64),
                ("expert_sb_stride", C.c_int64), ("shared_q", C.c_void_p), ("shared_sb", C.c_void_p)]


_lib = None
_P = C.c_void_p
_I = C.c_int32
_S = C.c_size_t

_SIGS = {
    "bgq_status_string": (C.c_char_p, [_I]),
    "bgq_abi_version": (_I, []),
    "q4_gemv": (_I, [C.POINTER(bgq_qmatrix), _P, _P, _I, _P]),
    "q2_gemv": (_I, [C.POINTER(bgq_qmatrix), _P, _P, _I, _P]),
    "bgq_qgemv_variant": (_I, [C.POINTER(bgq_qmatrix), _P, _P, _I, _I, _P]),
    "q8_gemv": (_I, [C.POINTER(bgq_qmatrix), _P, _P, _I, _P]),
    "moe_route_workspace_bytes": (_S, [_I, _I]),
    "moe_route_topk": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _S, _P]),
    "moe_expert_workspace_bytes": (_S, [C.POINTER(bgq_expert), _I]),
    "moe_expert_swiglu": (_I, [C.POINTER(bgq_expert), _P, _I, _P, _P, _P, _S, _P]),
    "moe_layer_workspace_bytes": (_S, [C.POINTER(bgq_moe_layer), _I]),
    "moe_layer_forward": (_I, [C.POINTER(bgq_moe_layer), _P, _I, _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_layer_forward_noalloc": (_I, [C.POINTER(bgq_moe_layer), _P, _I, _P, _P, _P, _P, _P, _P]),
    "moe_stream_slots_bytes": (_S, [C.POINTER(bgq_moe_layer), _I]),
    "moe_layer_forward_streamed": (_I, [C.POINTER(bgq_moe_layer), _P, _I, _P, _P, _P, _P, _P, _P, _S, _P, _S,
                                        _P]),
    "bgq_rmsnorm": (_I, [_P, _P, _I, _I, C.c_float, _P, _P]),
    "bgq_residual_add": (_I, [_P, _P, C.c_int64, _P]),
    "bgq_gemv_chain_workspace_bytes": (_S, [C.POINTER(bgq_qmatrix), _I, _I]),
    "bgq_gemv_chain": (_I, [C.POINTER(bgq_qmatrix), _I, _P, _I, _I, _P, C.c_float, _I, _P, _P, _P, _S, _P]),
    "moe_stack_workspace_bytes": (_S, [C.POINTER(bgq_moe_layer), _I]),
    "moe_stack_decode": (_I, [C.POINTER(bgq_moe_layer), C.POINTER(_P), _I, C.c_float, _P, _P, _P, _P, _P, _S,
                              _P]),
    "moe_stack_trace_entries": (_S, [C.POINTER(bgq_moe_layer), _I]),
    "moe_stack_decode_traced": (_I, [C.POINTER(bgq_moe_layer), C.POINTER(_P), _I, C.c_float, _P, _P, _P, _P, _P,
                                     _S, _P, _P]),
    "bgq_wait_selftest": (_I, [_P, _S, C.c_int64, _P]),
    "bgq_read_device_status": (_I, [_P, _P]),
}


def load():
    """Load libbgq.so once and declare every entry point's argtypes/restype."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(the CUDA library is required; there is no fallback)")
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(s: int) -> str:
    return load().bgq_status_string(s).decode()


def _check(status: int, where: str):
    if status != OK:
        raise BGQError(status, where)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


_alloc = None


def set_allocator(fn) -> None:
    """Route the buffers this binding creates (outputs not passed in, and
    workspaces) through fn(shape, dtype, device, zero) -> tensor, e.g. a
    caller's pool; None restores plain torch allocation. fn must return a
    contiguous tensor of that shape and dtype, 256-byte aligned, zero-filled
    when zero is True."""
    global _alloc
    _alloc = fn


def alloc(shape, dtype, device, zero=False) -> torch.Tensor:
    """A buffer from the installed allocator (see set_allocator), else torch."""
    if _alloc is not None:
        return _alloc(tuple(shape), dtype, device, zero)
    return (torch.zeros if zero else torch.empty)(tuple(shape), dtype=dtype, device=device)


def workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled workspace (torch allocations are at least 256-byte aligned)."""
    return alloc((max(int(nbytes), 256),), torch.uint8, device, zero=True)


# ------------------------------------------------------------------ matrices
class QMatrix:
    """A packed matrix: q int32 [rows][cols*bits/32], sb bf16 [rows][cols/group][2].

    group is 64, or cols for the per-row 8-bit format (one (scale, bias) per row).
    """

    def __init__(self, q: torch.Tensor, sb: torch.Tensor, rows: int, cols: int, bits: int, group: int = GROUP):
        self.q, self.sb, self.rows, self.cols, self.bits, self.group = q, sb, rows, cols, bits, group

    def struct(self) -> bgq_qmatrix:
        return bgq_qmatrix(self.q.data_ptr(), self.sb.data_ptr(), self.rows, self.cols, self.bits, self.group)


def _gemv(fn, W: QMatrix, x, y, stream, *extra):
    x2 = x.reshape(-1, W.cols)
    if y is None:
        y = alloc((x2.shape[0], W.rows), torch.bfloat16, x.device)
    s = W.struct()
    _check(fn(C.byref(s), _ptr(x2), _ptr(y), x2.shape[0], *extra, _stream(stream)), fn.__name__)
    return y


def q4_gemv(W: QMatrix, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    return _gemv(load().q4_gemv, W, x, y, stream)


def q2_gemv(W: QMatrix, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    return _gemv(load().q2_gemv, W, x, y, stream)


def q8_gemv(W: QMatrix, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """8-bit GEMV (int8 MLP / QKV weights; per-group or, with W.group == W.cols, per-row scale/bias)."""
    return _gemv(load().q8_gemv, W, x, y, stream)


def qgemv_variant(W: QMatrix, x: torch.Tensor, variant: int, y=None, stream=None) -> torch.Tensor:
    lib = load()
    x2 = x.reshape(-1, W.cols)
    if y is None:
        y = alloc((x2.shape[0], W.rows), torch.bfloat16, x.device)
    s = W.struct()
    _check(lib.bgq_qgemv_variant(C.byref(s), _ptr(x2), _ptr(y), x2.shape[0], variant, _stream(stream)),
           "bgq_qgemv_variant")
    return y


# ------------------------------------------------------------------ routing
def moe_route_topk(router, shared_gate, x, top_k, ws=None, want_logits=False, stream=None):
    lib = load()
    B, d = x.shape
    E = router.shape[0]
    dev = x.device
    idx = alloc((B, top_k), torch.int32, dev)
    w = alloc((B, top_k), torch.float32, dev)
    gamma = alloc((B,), torch.float32, dev)
    logits = alloc((B, E), torch.float32, dev) if want_logits else None
    need = lib.moe_route_workspace_bytes(B, E)
    if ws is None:
        ws = workspace(need, dev)
    _check(lib.moe_route_topk(_ptr(router), _ptr(shared_gate), _ptr(x), B, d, E, top_k, _ptr(idx), _ptr(w),
                              _ptr(gamma), _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)), "moe_route_topk")
    return idx, w, gamma, logits


# ------------------------------------------------------------------ experts
class Expert:
    """gate [f][d], up [f][d], down [d][f], each a QMatrix."""

    def __init__(self, gate: QMatrix, up: QMatrix, down: QMatrix):
        self.gate, self.up, self.down = gate, up, down

    def struct(self) -> bgq_expert:
        return bgq_expert(self.gate.struct(), self.up.struct(), self.down.struct())


def expert_workspace_bytes(e: Expert, batch: int) -> int:
    s = e.struct()
    return int(load().moe_expert_workspace_bytes(C.byref(s), batch))


def moe_expert_swiglu(e: Expert, x: torch.Tensor, ws=None, want_f32=False, stream=None):
    lib = load()
    B = x.shape[0]
    d = e.gate.cols
    s = e.struct()
    y = alloc((B, d), torch.bfloat16, x.device)
    yf = alloc((B, d), torch.float32, x.device) if want_f32 else None
    need = lib.moe_expert_workspace_bytes(C.byref(s), B)
    if ws is None:
        ws = workspace(need, x.device)
    _check(lib.moe_expert_swiglu(C.byref(s), _ptr(x), B, _ptr(y), _ptr(yf), _ptr(ws), ws.numel(),
                                 _stream(stream)), "moe_expert_swiglu")
    return y, yf


# ------------------------------------------------------------------ layers
class MoELayer:
    """One layer's tensors: router bf16 [E][d], shared_gate bf16 [d] or None,
    pool_q int32 [E(+1)][q_stride], pool_sb bf16 [E(+1)][sb_stride] (routed
    experts 0..E-1), shared_q / shared_sb (one expert, same internal layout)."""

    def __init__(self, d_model, d_ff, n_experts, top_k, bits, router, shared_gate, pool_q, pool_sb, shared_q,
                 shared_sb):
        self.d_model, self.d_ff, self.n_experts, self.top_k, self.bits = d_model, d_ff, n_experts, top_k, bits
        self.router, self.shared_gate = router, shared_gate
        self.pool_q, self.pool_sb, self.shared_q, self.shared_sb = pool_q, pool_sb, shared_q, shared_sb

    def struct(self) -> bgq_moe_layer:
        return bgq_moe_layer(self.d_model, self.d_ff, self.n_experts, self.top_k, self.bits, GROUP,
                             self.router.data_ptr(),
                             None if self.shared_gate is None else self.shared_gate.data_ptr(),
                             self.pool_q.data_ptr(), self.pool_sb.data_ptr(), self.pool_q.stride(0),
                             self.pool_sb.stride(0), self.shared_q.data_ptr(), self.shared_sb.data_ptr())


def moe_layer_workspace_bytes(layer: MoELayer, batch: int) -> int:
    s = layer.struct()
    return load().moe_layer_workspace_bytes(C.byref(s), batch)


def moe_layer_forward(layer: MoELayer, x: torch.Tensor, ws=None, out=None, out_f32=None, want_out=True,
                      want_f32=False, want_route=False, stream=None):
    lib = load()
    B, d = x.shape
    dev = x.device
    s = layer.struct()
    if out is None and want_out:
        out = alloc((B, d), torch.bfloat16, dev)
    if out_f32 is None and want_f32:
        out_f32 = alloc((B, d), torch.float32, dev)
    idx = w = gamma = None
    if want_route:
        idx = alloc((B, layer.top_k), torch.int32, dev)
        w = alloc((B, layer.top_k), torch.float32, dev)
        gamma = alloc((B,), torch.float32, dev)
    if ws is None:
        ws = workspace(lib.moe_layer_workspace_bytes(C.byref(s), B), dev)
    _check(lib.moe_layer_forward(C.byref(s), _ptr(x), B, _ptr(out), _ptr(out_f32), _ptr(idx), _ptr(w),
                                 _ptr(gamma), _ptr(ws), ws.numel(), _stream(stream)), "moe_layer_forward")
    return out, out_f32, idx, w, gamma


def moe_layer_forward_noalloc(layer: MoELayer, x: torch.Tensor, out=None, out_f32=None, idx=None, w=None,
                              gamma=None, stream=None):
    """moe_layer_forward with the library's fixed scratch array instead of a
    workspace: for callers that cannot allocate device memory at call time.
    Output buffers given as None are not written (pass tensors to receive them)."""
    B = x.shape[0]
    s = layer.struct()
    _check(load().moe_layer_forward_noalloc(C.byref(s), _ptr(x), B, _ptr(out), _ptr(out_f32), _ptr(idx), _ptr(w),
                                            _ptr(gamma), _stream(stream)), "moe_layer_forward_noalloc")
    return out, out_f32, idx, w, gamma


def moe_stream_slots_bytes(layer: MoELayer, batch: int) -> int:
    s = layer.struct()
    return load().moe_stream_slots_bytes(C.byref(s), batch)


def moe_layer_forward_streamed(layer: MoELayer, x: torch.Tensor, slots=None, ws=None, out=None, out_f32=None,
                               want_out=True, want_f32=False, want_route=False, stream=None):
    """moe_layer_forward with the selected experts copied into device `slots`
    first (a uint8 tensor of moe_stream_slots_bytes(layer, batch) bytes), then
    computed there."""
    lib = load()
    B, d = x.shape
    dev = x.device
    s = layer.struct()
    if out is None and want_out:
        out = alloc((B, d), torch.bfloat16, dev)
    if out_f32 is None and want_f32:
        out_f32 = alloc((B, d), torch.float32, dev)
    idx = w = gamma = None
    if want_route:
        idx = alloc((B, layer.top_k), torch.int32, dev)
        w = alloc((B, layer.top_k), torch.float32, dev)
        gamma = alloc((B,), torch.float32, dev)
    if ws is None:
        ws = workspace(lib.moe_layer_workspace_bytes(C.byref(s), B), dev)
    if slots is None:
        slots = alloc((lib.moe_stream_slots_bytes(C.byref(s), B),), torch.uint8, dev)
    _check(lib.moe_layer_forward_streamed(C.byref(s), _ptr(x), B, _ptr(out), _ptr(out_f32), _ptr(idx), _ptr(w),
                                          _ptr(gamma), _ptr(slots), slots.numel(), _ptr(ws), ws.numel(),
                                          _stream(stream)), "moe_layer_forward_streamed")
    return out, out_f32, idx, w, gamma


def bgq_rmsnorm(h: torch.Tensor, rho, eps: float, a=None, stream=None):
    B, d = h.shape
    if a is None:
        a = alloc((B, d), torch.bfloat16, h.device)
    _check(load().bgq_rmsnorm(_ptr(h), _ptr(rho), B, d, eps, _ptr(a), _stream(stream)), "bgq_rmsnorm")
    return a


def bgq_residual_add(h: torch.Tensor, delta: torch.Tensor, stream=None):
    _check(load().bgq_residual_add(_ptr(h), _ptr(delta), h.numel(), _stream(stream)), "bgq_residual_add")
    return h


def _chain_structs(mats: list):
    arr = (bgq_qmatrix * len(mats))()
    for i, m in enumerate(mats):
        arr[i] = m.struct()
    return arr


def gemv_chain_workspace_bytes(mats: list, batch: int) -> int:
    return load().bgq_gemv_chain_workspace_bytes(_chain_structs(mats), len(mats), batch)


def gemv_chain(mats: list, x: torch.Tensor, norm: bool = False, rho=None, eps: float = 1e-6, residual: bool = False,
               want_out: bool = True, want_f32: bool = False, ws=None, out=None, out_f32=None, stream=None):
    """bgq_gemv_chain: v_0 = rmsnorm(x)*rho (norm) or x, v_i = bf16(W_i v_{i-1}), out = W_n v (+ x).

    Returns (out bf16 or None, out_f32 or None), each [batch][mats[-1].rows]."""
    lib = load()
    arr = _chain_structs(mats)
    x2 = x.reshape(-1, mats[0].cols)
    B = x2.shape[0]
    rows = mats[-1].rows
    if want_out and out is None:
        out = alloc((B, rows), torch.bfloat16, x.device)
    if want_f32 and out_f32 is None:
        out_f32 = alloc((B, rows), torch.float32, x.device)
    if ws is None:
        ws = workspace(lib.bgq_gemv_chain_workspace_bytes(arr, len(mats), B), x.device)
    _check(lib.bgq_gemv_chain(arr, len(mats), _ptr(x2), B, int(norm), _ptr(rho), eps, int(residual), _ptr(out),
                              _ptr(out_f32), _ptr(ws), ws.numel(), _stream(stream)), "bgq_gemv_chain")
    return out, out_f32


class Stack:
    """Marshalled arguments of moe_stack_decode for a list of layers and RMSNorm weights."""

    def __init__(self, layers: list, rhos: list):
        self.layers, self.rhos = layers, rhos
        n = len(layers)
        self.c_layers = (bgq_moe_layer * n)(*[L.struct() for L in layers])
        self.c_rho = (C.c_void_p * n)(*[r.data_ptr() for r in rhos])
        self.ws_bytes = load().moe_stack_workspace_bytes(self.c_layers, n)


def moe_stack_decode(stack: Stack, x: torch.Tensor, eps: float = 1e-6, ws=None, x_next=None, h_out=None,
                     idx_out=None, stream=None):
    lib = load()
    n = len(stack.layers)
    if ws is None:
        ws = workspace(stack.ws_bytes, x.device)
    _check(lib.moe_stack_decode(stack.c_layers, stack.c_rho, n, eps, _ptr(x), _ptr(x_next), _ptr(h_out),
                                _ptr(idx_out), _ptr(ws), ws.numel(), _stream(stream)), "moe_stack_decode")
    return x_next, h_out, idx_out


def wait_selftest(ws: torch.Tensor, timeout_ns: int, stream=None) -> None:
    _check(load().bgq_wait_selftest(_ptr(ws), ws.numel(), timeout_ns, _stream(stream)), "bgq_wait_selftest")


TRACE_EVENTS = ("layer_start", "prev_layer_done", "input_normalised", "router_done", "shared_gateup_done",
                "logits_visible", "selected_gateup_done", "swiglu_visible", "down_combine_done", "down_rows_landed",
                "down_dots_done", "selected", "input_staged", "swiglu_staged", "first_chunk_landed", "last_chunk_landed")


def moe_stack_decode_traced(stack: Stack, x: torch.Tensor, eps: float = 1e-6, ws=None, x_next=None, h_out=None,
                            idx_out=None, stream=None):
    """moe_stack_decode plus per-SM phase timestamps; returns the trace as an
    int64 tensor [n_layers][n_sm][10] of %globaltimer nanoseconds."""
    lib = load()
    n = len(stack.layers)
    ent = lib.moe_stack_trace_entries(stack.c_layers, n)
    if ent == 0:
        raise BGQError(ERR_UNSUPPORTED, "moe_stack_trace_entries")
    trace = alloc((ent,), torch.int64, x.device, zero=True)
    if ws is None:
        ws = workspace(stack.ws_bytes, x.device)
    _check(lib.moe_stack_decode_traced(stack.c_layers, stack.c_rho, n, eps, _ptr(x), _ptr(x_next), _ptr(h_out),
                                       _ptr(idx_out), _ptr(ws), ws.numel(), _ptr(trace), _stream(stream)),
           "moe_stack_decode_traced")
    return trace.view(n, -1, len(TRACE_EVENTS))


def read_device_status(ws: torch.Tensor, stream=None) -> int:
    return load().bgq_read_device_status(_ptr(ws), _stream(stream))
