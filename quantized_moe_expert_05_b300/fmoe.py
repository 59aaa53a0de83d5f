"""ctypes binding of libfmoe.so (argument marshalling only).

Every step of the MoE block runs in the library's CUDA kernels; this module
turns torch tensors into device pointers, passes the current CUDA stream and
raises on a non-OK status.  There is no CPU fallback: if the library cannot
be loaded, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfmoe.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_RANGE = 0, 1, 2, 3, 4, 5
MAX_TOKENS, MAX_TOPK, MAX_EXPERTS, MAX_LAYERS = 16, 16, 1024, 1024


class FmoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


class fmoe_layer(ctypes.Structure):
    _fields_ = [
        ("bits", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("inter", ctypes.c_int32),
        ("n_experts", ctypes.c_int32),
        ("has_shared", ctypes.c_int32),
        ("experts", ctypes.c_void_p),
        ("shared", ctypes.c_void_p),
        ("shared_gate_w", ctypes.c_void_p),
    ]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m quantized_moe_expert_05_b300.build` "
            "(the library has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    LP = ctypes.POINTER(fmoe_layer)
    sig = {
        "fmoe_expert_bytes": (Z, [I, I, I, I]),
        "fmoe_workspace_bytes": (Z, [LP, I, I, I]),
        "fmoe_workspace_init": (I, [P, Z, P]),
        "fmoe_route": (I, [P, I, I, I, P, P, P]),
        "fmoe_router_logits": (I, [P, P, I, I, I, P, P]),
        "fmoe_route_from_x": (I, [P, P, I, I, I, I, P, P, P, P, P, P]),
        "fmoe_expert_ffn": (I, [LP, P, I, I, P, P, P, P]),
        "fmoe_moe_block": (I, [LP, P, P, P, P, I, I, P, P]),
        "fmoe_stack_decode": (I, [LP, I, P, P, I, F, P, P]),
        "fmoe_ws_routing": (I, [P, LP, I, I, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P),
                                ctypes.POINTER(P)]),
        "fmoe_ws_batch_plan": (I, [P, LP, I, I, ctypes.POINTER(P)]),
        "fmoe_status_string": (ctypes.c_char_p, [I]),
        "fmoe_last_device_error": (I, [P, P]),
        "fmoe_debug_wait_test": (I, [P, I, I, I, P]),
        "fmoe_moe_block_noalloc": (I, [LP, P, P, P, P, I, P, P]),
        "fmoe_debug_launch_geometry": (I, [I, I, I, I, I, I, I, ctypes.POINTER(ctypes.c_int64), I]),
        "fmoe_debug_block_pieces": (I, [I, I, I, I, I, I, I, ctypes.POINTER(ctypes.c_int64), I]),
        "fmoe_dense_row_bytes": (Z, [I, I]),
        "fmoe_dense_gemv": (I, [P, I, I, I, P, I, P, P, P]),
        "fmoe_rmsnorm": (I, [P, P, I, I, F, P, P]),
        "fmoe_pool_state_bytes": (Z, [I, I]),
        "fmoe_pool_init": (I, [P, Z, I, I, Z, P, P]),
        "fmoe_pool_plan": (I, [P, P, I, I, P, P, ctypes.POINTER(I)]),
        "fmoe_pool_load": (I, [P, P, I, P]),
        "fmoe_pool_slot_logits": (I, [P, P, P, P, I, I, P]),
        "fmoe_pool_stats": (I, [P, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64),
                                ctypes.POINTER(ctypes.c_uint64)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.fmoe_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise FmoeError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def expert_bytes(bits: int, hidden: int, inter: int, group: int = 64) -> int:
    return int(lib.fmoe_expert_bytes(bits, hidden, inter, group))


@dataclass
class Layer:
    """One MoE layer: packed routed experts, optional shared expert and gate."""

    bits: int
    hidden: int
    inter: int
    n_experts: int
    experts: torch.Tensor                      # flat int32/uint8 device tensor, E blobs
    shared: Optional[torch.Tensor] = None      # one blob
    shared_gate_w: Optional[torch.Tensor] = None  # int16/bfloat16 [H]

    def c(self) -> fmoe_layer:
        s = fmoe_layer()
        s.bits, s.group, s.hidden, s.inter = self.bits, 64, self.hidden, self.inter
        s.n_experts = self.n_experts
        s.has_shared = 1 if self.shared is not None else 0
        s.experts = _ptr(self.experts)
        s.shared = _ptr(self.shared)
        s.shared_gate_w = _ptr(self.shared_gate_w)
        return s


def workspace_bytes(layer: Layer, T: int, K: int, L: int = 1) -> int:
    n = int(lib.fmoe_workspace_bytes(ctypes.byref(layer.c()), T, K, L))
    if n == 0:
        raise FmoeError(ERR_INVALID_ARG, "fmoe_workspace_bytes")
    return n


def new_workspace(layer: Layer, T: int, K: int, L: int = 1, device=None, stream=None) -> torch.Tensor:
    """Allocate (through torch) and zero a workspace for the given sizes."""
    n = workspace_bytes(layer, T, K, L)
    ws = torch.empty(n, dtype=torch.uint8, device=device or layer.experts.device)
    _check(lib.fmoe_workspace_init(_ptr(ws), n, _stream(stream)), "fmoe_workspace_init")
    return ws


def route(logits: torch.Tensor, K: int, ids: Optional[torch.Tensor] = None,
          weights: Optional[torch.Tensor] = None, stream=None):
    T, E = logits.shape
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    if ids is None:
        ids = torch.empty((T, K), dtype=torch.int32, device=logits.device)
    if weights is None:
        weights = torch.empty((T, K), dtype=torch.float32, device=logits.device)
    _check(lib.fmoe_route(_ptr(logits), T, E, K, _ptr(ids), _ptr(weights), _stream(stream)), "fmoe_route")
    return ids, weights


def dense_row_bytes(bits: int, hidden: int) -> int:
    return int(lib.fmoe_dense_row_bytes(bits, hidden))


def dense_gemv(w: torch.Tensor, bits: int, n_rows: int, x: torch.Tensor, residual: Optional[torch.Tensor] = None,
               y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y[t] = W x[t] (+ residual[t]) for a dense quantised matrix of n_rows row records."""
    T, H = x.shape
    if y is None:
        y = torch.empty((T, n_rows), dtype=torch.float32, device=x.device)
    _check(lib.fmoe_dense_gemv(_ptr(w), bits, n_rows, H, _ptr(x), T, _ptr(residual), _ptr(y), _stream(stream)),
           "fmoe_dense_gemv")
    return y


def rmsnorm(h: torch.Tensor, eps: float, weight: Optional[torch.Tensor] = None, x: Optional[torch.Tensor] = None,
            stream=None) -> torch.Tensor:
    """x[t] = h[t] / sqrt(mean(h[t]^2) + eps) (* weight)."""
    T, H = h.shape
    if x is None:
        x = torch.empty_like(h)
    _check(lib.fmoe_rmsnorm(_ptr(h), _ptr(weight), T, H, eps, _ptr(x), _stream(stream)), "fmoe_rmsnorm")
    return x


def router_logits(w_router: torch.Tensor, x: torch.Tensor, logits: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """logits[t] = W_r x[t]; w_router int16/bfloat16 [E][H], x fp32 [T][H]."""
    E, H = w_router.shape
    T = x.shape[0]
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    _check(lib.fmoe_router_logits(_ptr(w_router), _ptr(x), T, H, E, _ptr(logits), _stream(stream)),
           "fmoe_router_logits")
    return logits


def route_from_x(w_router: torch.Tensor, x: torch.Tensor, K: int, shared_gate_w: Optional[torch.Tensor] = None,
                 stream=None):
    """(logits, ids, weights, gate or None): the router projection, then top-K + softmax."""
    E, H = w_router.shape
    T = x.shape[0]
    dev = x.device
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    weights = torch.empty((T, K), dtype=torch.float32, device=dev)
    gate = torch.empty((T,), dtype=torch.float32, device=dev) if shared_gate_w is not None else None
    _check(lib.fmoe_route_from_x(_ptr(w_router), _ptr(x), T, H, E, K, _ptr(shared_gate_w), _ptr(logits), _ptr(ids),
                                 _ptr(weights), _ptr(gate), _stream(stream)), "fmoe_route_from_x")
    return logits, ids, weights, gate


def expert_ffn(layer: Layer, ids: torch.Tensor, x: torch.Tensor, ws: torch.Tensor,
               y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    T, K = ids.shape
    S = 1 if layer.shared is not None else 0
    if y is None:
        y = torch.empty((T, K + S, layer.hidden), dtype=torch.float32, device=x.device)
    _check(lib.fmoe_expert_ffn(ctypes.byref(layer.c()), _ptr(ids), T, K, _ptr(x), _ptr(y), _ptr(ws),
                               _stream(stream)), "fmoe_expert_ffn")
    return y


def moe_block(layer: Layer, x: torch.Tensor, logits: torch.Tensor, residual: torch.Tensor, K: int,
              ws: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    T = x.shape[0]
    if x.shape != (T, layer.hidden) or logits.shape != (T, layer.n_experts) or residual.shape != x.shape:
        raise ValueError("x, residual must be [T][H] and logits [T][E]")
    if out is None:
        out = torch.empty_like(residual)
    _check(lib.fmoe_moe_block(ctypes.byref(layer.c()), _ptr(x), _ptr(logits), _ptr(residual), _ptr(out), T, K,
                              _ptr(ws), _stream(stream)), "fmoe_moe_block")
    return out


def stack_decode(layers: Sequence[Layer], logits: torch.Tensor, h: torch.Tensor, K: int, eps: float,
                 ws: torch.Tensor, stream=None) -> torch.Tensor:
    """In place: h <- h + MoE_l(RMSNorm(h)) for every layer."""
    if logits.numel() != len(layers) * layers[0].n_experts or h.numel() != layers[0].hidden:
        raise ValueError("logits must be [L][E] and h [H]")
    arr = (fmoe_layer * len(layers))(*[l.c() for l in layers])
    _check(lib.fmoe_stack_decode(arr, len(layers), _ptr(logits), _ptr(h), K, float(eps), _ptr(ws),
                                 _stream(stream)), "fmoe_stack_decode")
    return h


def ws_routing(ws: torch.Tensor, layer: Layer, T: int, K: int) -> dict:
    """Views of the routing result and h left in a workspace by moe_block."""
    P = ctypes.c_void_p
    ids, w, g, h = P(), P(), P(), P()
    _check(lib.fmoe_ws_routing(_ptr(ws), ctypes.byref(layer.c()), T, K, ctypes.byref(ids), ctypes.byref(w),
                               ctypes.byref(g), ctypes.byref(h)), "fmoe_ws_routing")
    base = ws.data_ptr()
    S = 1 if layer.shared is not None else 0

    def view(p, dtype, n):
        off = p.value - base
        return ws[off: off + 4 * n].view(dtype)

    return {
        "ids": view(ids, torch.int32, T * K).view(T, K),
        "weights": view(w, torch.float32, T * K).view(T, K),
        "gate": view(g, torch.float32, T),
        "h": view(h, torch.float32, T * (K + S) * layer.inter).view(T, K + S, layer.inter),
    }


def ws_batch_plan(ws: torch.Tensor, layer: Layer, T: int, K: int) -> dict:
    """The batch plan left in a workspace by expert_ffn or a batched moe_block
    (copied to the host; synchronises): item count, distinct experts read, and
    per item (expert id or -1 for the shared expert, [(t, slot), ...])."""
    p = ctypes.c_void_p()
    _check(lib.fmoe_ws_batch_plan(_ptr(ws), ctypes.byref(layer.c()), T, K, ctypes.byref(p)),
           "fmoe_ws_batch_plan")
    off = p.value - ws.data_ptr()
    head = ws[off: off + 32].view(torch.int32).cpu().tolist()
    n = head[0]
    body = ws[off + 32: off + 32 + 32 * n].view(torch.int32).view(n, 8).cpu().tolist()
    items = [(r[0], [(v >> 8, v & 255) for v in r[2: 2 + r[1]]]) for r in body]
    return {"n_items": n, "n_unique": head[1], "items": items}


def last_device_error(ws: torch.Tensor, stream=None) -> int:
    return int(lib.fmoe_last_device_error(_ptr(ws), _stream(stream)))


def debug_wait_test(ws: torch.Tensor, n_blocks: int, expected: int, timeout_us: int, stream=None) -> None:
    _check(lib.fmoe_debug_wait_test(_ptr(ws), n_blocks, expected, timeout_us, _stream(stream)),
           "fmoe_debug_wait_test")


NOALLOC_SCRATCH_BYTES = 128 * 1024


def moe_block_noalloc(layer: Layer, x: torch.Tensor, logits: torch.Tensor, residual: torch.Tensor, K: int,
                      out: Optional[torch.Tensor] = None, device_error: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """One token through fmoe_moe_block_noalloc (no workspace; the library's own
    fixed device scratch).  For callers that cannot allocate device memory the
    output (and the optional int32 error word) must be preallocated."""
    if x.shape != (1, layer.hidden) or logits.shape != (1, layer.n_experts) or residual.shape != x.shape:
        raise ValueError("x, residual must be [1][H] and logits [1][E]")
    if out is None:
        out = torch.empty_like(residual)
    _check(lib.fmoe_moe_block_noalloc(ctypes.byref(layer.c()), _ptr(x), _ptr(logits), _ptr(residual), _ptr(out),
                                      K, _ptr(device_error), _stream(stream)), "fmoe_moe_block_noalloc")
    return out


class SlotPool:
    """HBM slot pool over a copy of every expert blob in pinned host memory.

    ``slots`` (device, n_slots * blob bytes) and ``host_blobs`` (pinned host,
    n_experts * blob bytes) are owned by the caller; this object holds the
    pool's host bookkeeping.  ``plan`` decides slots and loads for a request
    (host only), ``load`` issues the copies, ``slot_logits`` maps router
    logits onto the slots."""

    def __init__(self, n_slots: int, n_experts: int, blob_bytes: int, slots_ptr: int, host_ptr: int):
        n = int(lib.fmoe_pool_state_bytes(n_slots, n_experts))
        if n == 0:
            raise FmoeError(ERR_INVALID_ARG, "fmoe_pool_state_bytes")
        self.n_slots, self.n_experts = n_slots, n_experts
        self._state = (ctypes.c_uint64 * ((n + 7) // 8))()
        _check(lib.fmoe_pool_init(ctypes.addressof(self._state), n, n_slots, n_experts, blob_bytes, slots_ptr,
                                  host_ptr), "fmoe_pool_init")

    @property
    def state(self) -> int:
        return ctypes.addressof(self._state)

    def plan(self, ids, keep: int = 0):
        """(slots, loads) for a request: ids a sequence of expert ids; loads a list of (expert, slot)."""
        ids = [int(i) for i in ids]
        n = len(ids)
        a_ids = (ctypes.c_int32 * n)(*ids)
        a_slots = (ctypes.c_int32 * n)()
        a_loads = (ctypes.c_int32 * (2 * n))()
        nl = ctypes.c_int(0)
        _check(lib.fmoe_pool_plan(self.state, ctypes.addressof(a_ids), n, keep, ctypes.addressof(a_slots),
                                  ctypes.addressof(a_loads), ctypes.byref(nl)), "fmoe_pool_plan")
        loads = [(a_loads[2 * i], a_loads[2 * i + 1]) for i in range(nl.value)]
        return list(a_slots), loads

    def load(self, loads, stream=None) -> None:
        flat = [v for pair in loads for v in pair]
        arr = (ctypes.c_int32 * max(1, len(flat)))(*flat)
        _check(lib.fmoe_pool_load(self.state, ctypes.addressof(arr), len(loads), _stream(stream)), "fmoe_pool_load")

    def slot_logits(self, logits, ids, slots):
        """logits [T][E] (host, fp32 numpy), ids and slots [T][K] -> slot logits [T][n_slots] (numpy)."""
        import numpy as np
        lg = np.ascontiguousarray(logits, dtype=np.float32)
        i = np.ascontiguousarray(ids, dtype=np.int32)
        sl = np.ascontiguousarray(slots, dtype=np.int32)
        T, K = i.shape
        out = np.empty((T, self.n_slots), dtype=np.float32)
        _check(lib.fmoe_pool_slot_logits(self.state, lg.ctypes.data, i.ctypes.data, sl.ctypes.data, T, K,
                                         out.ctypes.data), "fmoe_pool_slot_logits")
        return out

    def stats(self):
        h, m, r = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
        _check(lib.fmoe_pool_stats(self.state, ctypes.byref(h), ctypes.byref(m), ctypes.byref(r)), "fmoe_pool_stats")
        return {"hits": h.value, "misses": m.value, "requests": r.value}
