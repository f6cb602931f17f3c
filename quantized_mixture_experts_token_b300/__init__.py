"""quantized_mixture_experts_token_b300 -- a routed MoE expert-FFN layer on 2/3-bit
block-quantised weights for NVIDIA B300 (sm_103a).

This module is a thin ctypes binding over ``libmoeq.so`` (C ABI in
``include/moeq.h``).  It only marshals torch tensors (device pointers, the
current CUDA stream) into the library calls; every step of the layer runs in
the library's CUDA kernels.  There is no CPU fallback: importing works on any
machine, but each call needs the built library and CUDA tensors and raises if
either is missing.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoeq.so")

MODE_AUTO, MODE_GEMV, MODE_GEMM, MODE_GEMM_S8 = 0, 1, 2, 3
STATUS_WAIT_TIMEOUT, STATUS_BAD_INDEX = 0x1, 0x2

# Function names of the C ABI (include/moeq.h).
ABI_FUNCTIONS = (
    "moe_route_topk", "moe_permute", "moe_permute_noalloc", "moe_quantize_act", "moe_expert_ffn_q2",
    "moe_shared_expert_q2", "moe_combine",
    "moe_layer_forward", "moe_workspace_bytes", "moe_get_device_status", "moe_last_error_string",
    "moe_trace_events", "moe_version", "moe_set_wait_limit",
)


class MoeqError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libmoeq error {code}: {msg}")
        self.code = code


class QWeights(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int), ("E", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("codes", ctypes.c_void_p * 3), ("scales", ctypes.c_void_p * 3)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run __graft_entry__.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        P, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.moe_route_topk.argtypes = [P, i, i, P, P, i, i, P, P, P, sz, P]
        L.moe_permute.argtypes = [P, i, i, i, P, P, P, P, P, P, sz, P]
        L.moe_permute_noalloc.argtypes = [P, i, i, i, P, P, P, P, P, P]
        L.moe_quantize_act.argtypes = [P, i, i, P, P, P]
        L.moe_expert_ffn_q2.argtypes = [P, i, ctypes.POINTER(QWeights), i, P, P, P, P, P, P, i, i, P, P, P, sz, P]
        L.moe_combine.argtypes = [P, P, P, i, i, i, P, P, P]
        L.moe_shared_expert_q2.argtypes = [P, i, ctypes.POINTER(QWeights), P, i, i, P, sz, P]
        L.moe_layer_forward.argtypes = [P, i, P, P, ctypes.POINTER(QWeights), i, i, P, P, P, i, P, sz, P]
        L.moe_workspace_bytes.argtypes = [i, i, i, i, i, i]
        L.moe_workspace_bytes.restype = sz
        L.moe_get_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
        L.moe_last_error_string.restype = ctypes.c_char_p
        L.moe_version.restype = ctypes.c_char_p
        L.moe_trace_events.argtypes = [P, i]
        L.moe_set_wait_limit.argtypes = [ctypes.c_uint64]
        for name in ABI_FUNCTIONS:
            if name not in ("moe_workspace_bytes", "moe_last_error_string", "moe_version"):
                getattr(L, name).restype = i
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        raise MoeqError(rc, lib().moe_last_error_string().decode())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoeq takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libmoeq takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def version() -> str:
    return lib().moe_version().decode()


def workspace_bytes(T: int, H: int, I: int, E: int, k: int, bits: int = 2) -> int:
    n = lib().moe_workspace_bytes(T, H, I, E, k, bits)
    if n == 0:
        raise MoeqError(-2, "unsupported shape")
    return int(n)


def workspace(T: int, H: int, I: int, E: int, k: int, bits: int = 2, device="cuda") -> torch.Tensor:
    """A zeroed workspace buffer (torch allocations are 512-byte aligned)."""
    return torch.zeros(workspace_bytes(T, H, I, E, k, bits), dtype=torch.uint8, device=device)


@dataclass
class ExpertWeights:
    """Quantised expert matrices of one layer, resident on the device.

    codes[m]: uint8 [E, K/32, N, 4*bits], scales[m]: fp16 [E, K/32, N] for
    m = gate, up (N=I, K=H) and down (N=H, K=I).
    """
    bits: int
    E: int
    H: int
    I: int
    codes: list
    scales: list

    @classmethod
    def from_layer(cls, layer) -> "ExpertWeights":
        s = layer.shape
        return cls(s.bits, s.E, s.H, s.I, list(layer.codes), list(layer.scales))

    def struct(self) -> QWeights:
        q = QWeights()
        q.bits, q.E, q.H, q.I = self.bits, self.E, self.H, self.I
        for m in range(3):
            q.codes[m] = self.codes[m].data_ptr()
            q.scales[m] = self.scales[m].data_ptr()
            if not (self.codes[m].is_cuda and self.scales[m].is_cuda):
                raise ValueError("expert weights must be on the device")
        return q


def route_topk(x, Wr, bias, k, ws):
    T, H = x.shape
    E = Wr.shape[0]
    idx = torch.empty(T, k, dtype=torch.int32, device=x.device)
    w = torch.empty(T, k, dtype=torch.float32, device=x.device)
    _check(lib().moe_route_topk(_ptr(x), T, H, _ptr(Wr), _ptr(bias), E, k, _ptr(idx), _ptr(w), _ptr(ws),
                                ws.numel(), _stream(x.device)))
    return idx, w


def permute(idx, E, ws):
    T, k = idx.shape
    dev = idx.device
    out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               perm_tok=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
               perm_slot=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
               inv=torch.empty(max(T, 1), k, dtype=torch.int32, device=dev))
    _check(lib().moe_permute(_ptr(idx), T, k, E, _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm_tok"]),
                             _ptr(out["perm_slot"]), _ptr(out["inv"]), _ptr(ws), ws.numel(), _stream(dev)))
    out["perm_tok"] = out["perm_tok"][: T * k]
    out["perm_slot"] = out["perm_slot"][: T * k]
    out["inv"] = out["inv"][:T]
    return out


def permute_noalloc(idx, E):
    """moe_permute without a workspace: its scratch is a fixed array inside the
    library, for callers that cannot allocate device memory (outputs are
    allocated here only because this wrapper returns torch tensors)."""
    T, k = idx.shape
    dev = idx.device
    out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               perm_tok=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
               perm_slot=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
               inv=torch.empty(max(T, 1), k, dtype=torch.int32, device=dev))
    _check(lib().moe_permute_noalloc(_ptr(idx), T, k, E, _ptr(out["counts"]), _ptr(out["offsets"]),
                                     _ptr(out["perm_tok"]), _ptr(out["perm_slot"]), _ptr(out["inv"]), _stream(dev)))
    out["perm_tok"] = out["perm_tok"][: T * k]
    out["perm_slot"] = out["perm_slot"][: T * k]
    out["inv"] = out["inv"][:T]
    return out


def quantize_act(x):
    T, H = x.shape
    q = torch.empty(T, H, dtype=torch.int8, device=x.device)
    s = torch.empty(T, H // 32, dtype=torch.float32, device=x.device)
    _check(lib().moe_quantize_act(_ptr(x), T, H, _ptr(q), _ptr(s), _stream(x.device)))
    return q, s


def expert_ffn(x, weights: ExpertWeights, k, perm, w=None, *, want_y=True, want_sorted=False, residual=False,
               mode=MODE_AUTO, want_h=False, ws=None):
    T = x.shape[0]
    dev = x.device
    P = T * k
    y = torch.empty(T, weights.H, dtype=torch.float32, device=dev) if want_y else None
    D = torch.empty(max(P, 1), weights.H, dtype=torch.float32, device=dev) if want_sorted else None
    qh = torch.empty(max(P, 1), weights.I, dtype=torch.int8, device=dev) if want_h else None
    sh = torch.empty(max(P, 1), weights.I // 32, dtype=torch.float32, device=dev) if want_h else None
    q = weights.struct()
    _check(lib().moe_expert_ffn_q2(_ptr(x), T, ctypes.byref(q), k, _ptr(perm["offsets"]), _ptr(perm["perm_tok"]),
                                   _ptr(perm["perm_slot"]), _ptr(w), _ptr(D), _ptr(y), int(residual), mode,
                                   _ptr(qh), _ptr(sh), _ptr(ws), ws.numel(), _stream(dev)))
    out = dict(y=y)
    if want_sorted:
        out["out_sorted"] = D[:P]
    if want_h:
        out["qh"], out["sh"] = qh[:P], sh[:P]
    return out


def shared_expert(x, weights: ExpertWeights, y=None, *, accumulate=False, mode=MODE_AUTO, ws=None):
    """y = (y if accumulate else 0) + the shared (E = 1) expert's SwiGLU FFN of every token."""
    T = x.shape[0]
    if y is None:
        if accumulate:
            raise ValueError("accumulate needs y")
        y = torch.empty(T, weights.H, dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(T, weights.H, weights.I, 1, 1, weights.bits, device=x.device)
    q = weights.struct()
    _check(lib().moe_shared_expert_q2(_ptr(x), T, ctypes.byref(q), _ptr(y), int(accumulate), mode, _ptr(ws),
                                      ws.numel(), _stream(x.device)))
    return y


def combine(out_sorted, inv, w, residual_x=None):
    T, k = inv.shape
    H = out_sorted.shape[1]
    y = torch.empty(T, H, dtype=torch.float32, device=out_sorted.device)
    _check(lib().moe_combine(_ptr(out_sorted), _ptr(inv), _ptr(w), T, k, H, _ptr(residual_x), _ptr(y),
                             _stream(out_sorted.device)))
    return y


def layer_forward(x, weights: ExpertWeights, Wr, bias, k, ws, *, residual=False, mode=MODE_AUTO, y=None,
                  want_routing=False):
    T = x.shape[0]
    dev = x.device
    if y is None:
        y = torch.empty(T, weights.H, dtype=torch.float32, device=dev)
    idx = torch.empty(max(T, 1), k, dtype=torch.int32, device=dev) if want_routing else None
    w = torch.empty(max(T, 1), k, dtype=torch.float32, device=dev) if want_routing else None
    q = weights.struct()
    _check(lib().moe_layer_forward(_ptr(x), T, _ptr(Wr), _ptr(bias), ctypes.byref(q), k, int(residual), _ptr(y),
                                   _ptr(idx), _ptr(w), mode, _ptr(ws), ws.numel(), _stream(dev)))
    if want_routing:
        return y, idx[:T], w[:T]
    return y


def trace_events(events) -> None:
    """Bracket every expert-kernel launch of this thread with the given
    torch.cuda.Event objects, pairwise in order (None switches tracing off)."""
    if not events:
        _check(lib().moe_trace_events(None, 0))
        return
    for e in events:
        e.record()  # materialise the underlying cudaEvent_t
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().moe_trace_events(arr, len(events)))


def set_wait_limit(ns: int = 0) -> None:
    """Bound of the device-side pipeline waits in ns (0: the default, 2 s)."""
    _check(lib().moe_set_wait_limit(int(ns)))


def device_status() -> int:
    st = ctypes.c_int(0)
    rc = lib().moe_get_device_status(_stream(), ctypes.byref(st))
    if rc not in (0, -6):
        _check(rc)
    return st.value
