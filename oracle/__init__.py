"""CPU oracle of the routed expert-FFN layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
use this module.  The product path never imports it and it imports nothing
from the product.  The arithmetic lives in ``moe_oracle.c`` (plain C, fp64);
this file only marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(_build.build())
        P = ctypes.c_void_p
        i = ctypes.c_int
        _lib.oracle_layer.argtypes = [P, i, i, i, i, i, i, P, P, P, P, P, P, P, P, i, P, i, i, P, P, P, P, P, P, P, P]
        _lib.oracle_layer.restype = i
        _lib.oracle_router_logits.argtypes = [P, i, i, P, P, i, P, i]
        _lib.oracle_topk_softmax.argtypes = [P, i, i, i, P, P]
        _lib.oracle_topk_softmax.restype = i
        _lib.oracle_permute.argtypes = [P, i, i, i, P, P, P, P, P]
        _lib.oracle_quantize_block32.argtypes = [P, i, P, P]
        _lib.oracle_expert_token.argtypes = [P, P, i, i, i, P, P, P, P, P, P, P, P, P, P, P, P, P]
        _lib.oracle_weight_code.argtypes = [P, i, i, i, i]
        _lib.oracle_weight_code.restype = i
        _lib.oracle_weight_value.argtypes = [P, P, i, i, i, i]
        _lib.oracle_weight_value.restype = ctypes.c_double
        _lib.oracle_weight_column.argtypes = [P, P, i, i, i, P]
        _lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        _lib.oracle_half_to_double.restype = ctypes.c_double
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def quantize_block32(v):
    v = _c(v, np.float32)
    n = v.shape[-1]
    flat = v.reshape(-1, n)
    q = np.empty(flat.shape, np.int8)
    s = np.empty((flat.shape[0], n // 32), np.float32)
    for r in range(flat.shape[0]):
        lib().oracle_quantize_block32(_p(flat[r]), n, _p(q[r]), _p(s[r]))
    return q.reshape(v.shape), s.reshape(*v.shape[:-1], n // 32)


def router_logits(x, Wr, bias=None, nthreads=None):
    x = _c(x, np.float32)
    Wr = _c(Wr, np.float32)
    T, H = x.shape
    E = Wr.shape[0]
    L = np.empty((T, E), np.float64)
    b = None if bias is None else _c(bias, np.float32)
    lib().oracle_router_logits(_p(x), T, H, _p(Wr), _p(b), E, _p(L), nthreads or default_threads())
    return L


def topk_softmax(L, k):
    L = _c(L, np.float64)
    T, E = L.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    if lib().oracle_topk_softmax(_p(L), T, E, k, _p(idx), _p(w)) != 0:
        raise ValueError("bad top-k arguments")
    return idx, w


def permute(idx, E):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm_tok = np.empty(T * k, np.int32)
    perm_slot = np.empty(T * k, np.int32)
    inv = np.empty((T, k), np.int32)
    lib().oracle_permute(_p(idx), T, k, E, _p(counts), _p(offsets), _p(perm_tok), _p(perm_slot), _p(inv))
    return dict(counts=counts, offsets=offsets, perm_tok=perm_tok, perm_slot=perm_slot, inv=inv)


def weight_code(codes_e, bits, N, n, kk):
    return lib().oracle_weight_code(_p(_c(codes_e, np.uint8)), bits, N, n, kk)


def dequantize_matrix(codes_e, scales_e, bits, N, K):
    """Dense fp64 [N, K] matrix of one expert, element by element (slow; tiny shapes only)."""
    c = _c(codes_e, np.uint8)
    s = _c(scales_e, np.uint16)
    out = np.empty((N, K), np.float64)
    f = lib().oracle_weight_value
    for n in range(N):
        for kk in range(K):
            out[n, kk] = f(_p(c), _p(s), bits, N, n, kk)
    return out


def weight_column(codes_e, scales_e, bits, N, kk):
    """Column kk (an input index) of one expert's dequantised [N, K] matrix, fp64."""
    out = np.empty(N, np.float64)
    lib().oracle_weight_column(_p(_c(codes_e, np.uint8)), _p(_c(scales_e, np.uint16)), bits, N, kk, _p(out))
    return out


def half_to_double(bits16: int) -> float:
    return lib().oracle_half_to_double(bits16)


def expert_token(qx, sx, codes3, scales3, bits, H, I):
    """One token through one expert; returns a dict of every intermediate."""
    qx = _c(qx, np.int8)
    sx = _c(sx, np.float32)
    c = [_c(a, np.uint8) for a in codes3]
    s = [_c(a, np.uint16) for a in scales3]
    out = dict(G=np.empty(I), U=np.empty(I), h=np.empty(I, np.float32), qh=np.empty(I, np.int8),
               sh=np.empty(I // 32, np.float32), hdist=np.empty(I), D=np.empty(H))
    lib().oracle_expert_token(_p(qx), _p(sx), H, I, bits, _p(c[0]), _p(s[0]), _p(c[1]), _p(s[1]), _p(c[2]), _p(s[2]),
                              _p(out["G"]), _p(out["U"]), _p(out["h"]), _p(out["qh"]), _p(out["sh"]),
                              _p(out["hdist"]), _p(out["D"]))
    return out


def layer(x, Wr, bias, codes, scales, bits, k, residual=False, tokens=None, nthreads=None, detail=False):
    """The whole layer for the given token rows (all rows by default).

    codes/scales: per matrix (gate, up, down) arrays of the whole layer in the
    storage layout; scales as uint16 fp16 bits.
    Returns dict(idx, w, y[, qh, sh, hdist, D]) for the selected rows.
    """
    x = _c(x, np.float32)
    T, H = x.shape
    Wr = _c(Wr, np.float32)
    E = Wr.shape[0]
    I = codes[0].shape[2]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    n = int(tokens.shape[0])
    c = [_c(a, np.uint8) for a in codes]
    s = [_c(a, np.uint16) for a in scales]
    b = None if bias is None else _c(bias, np.float32)
    out = dict(idx=np.empty((n, k), np.int32), w=np.empty((n, k), np.float32), y=np.empty((n, H), np.float32))
    if detail:
        out.update(h=np.empty((n, k, I), np.float32), qh=np.empty((n, k, I), np.int8), sh=np.empty((n, k, I // 32), np.float32),
                   hdist=np.empty((n, k, I)), D=np.empty((n, k, H)))
    rc = lib().oracle_layer(_p(x), T, H, I, E, k, bits, _p(Wr), _p(b), _p(c[0]), _p(s[0]), _p(c[1]), _p(s[1]),
                            _p(c[2]), _p(s[2]), int(bool(residual)), _p(tokens), n, nthreads or default_threads(),
                            _p(out["idx"]), _p(out["w"]), _p(out["y"]), _p(out.get("h")), _p(out.get("qh")), _p(out.get("sh")),
                            _p(out.get("hdist")), _p(out.get("D")))
    if rc != 0:
        raise ValueError("oracle_layer rejected its arguments")
    return out
