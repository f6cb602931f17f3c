"""The C ABI library loads, exports every declared entry point, and validates
arguments on the host (no kernel is launched by these tests)."""
import ctypes
import os
import re

import pytest

import quantized_mixture_experts_token_b300 as moeq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__

    __graft_entry__.build()
    return moeq.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moeq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_names():
    assert set(declared_functions()) == set(moeq.ABI_FUNCTIONS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.moe_version().decode().startswith("moeq")


def test_peaks_library_exports_its_header():
    import ctypes as C

    src = open(os.path.join(ROOT, "include", "moeq_peaks.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))
    assert names == ["moe_peak_mma_s8", "moe_peak_umma_issue"]
    import __graft_entry__

    __graft_entry__.build()
    lib = C.CDLL(os.path.join(ROOT, "quantized_mixture_experts_token_b300", "libmoeq_peaks.so"))
    for n in names:
        assert hasattr(lib, n), n
    lib.moe_peak_mma_s8.argtypes = [C.c_int, C.c_int, C.c_void_p]
    assert lib.moe_peak_mma_s8(0, 1, None) == -1  # argument checks, nothing launched
    lib.moe_peak_umma_issue.argtypes = [C.c_int, C.c_int, C.c_int, C.c_void_p]
    assert lib.moe_peak_umma_issue(24, 8, 1, None) == -1


def test_workspace_bytes_host_logic(L):
    n1 = moeq.workspace_bytes(1, 2048, 512, 512, 10)
    n8 = moeq.workspace_bytes(8, 2048, 512, 512, 10)
    n4k = moeq.workspace_bytes(4096, 2048, 512, 512, 10)
    assert 0 < n1 < n8 < n4k
    assert n4k % 256 == 0
    # unsupported shapes report 0
    assert L.moe_workspace_bytes(4, 100, 512, 512, 10, 2) == 0
    assert L.moe_workspace_bytes(4, 2048, 512, 512, 40, 2) == 0
    assert L.moe_workspace_bytes(4, 2048, 512, 2048, 10, 2) == 0
    assert L.moe_workspace_bytes(4, 2048, 512, 512, 10, 4) == 0


def test_argument_errors_are_reported_before_launch(L):
    P = ctypes.c_void_p
    # NULL x -> bad argument
    rc = L.moe_route_topk(None, 4, 2048, P(256), None, 512, 10, P(256), P(256), P(256), 1 << 30, None)
    assert rc == -1 and b"x is NULL" in L.moe_last_error_string()
    # misaligned pointer
    rc = L.moe_route_topk(P(258), 4, 2048, P(256), None, 512, 10, P(256), P(256), P(256), 1 << 30, None)
    assert rc == -3
    # unsupported shape
    rc = L.moe_route_topk(P(256), 4, 2000, P(256), None, 512, 10, P(256), P(256), P(256), 1 << 30, None)
    assert rc == -2
    # workspace too small
    q = moeq.QWeights()
    q.bits, q.E, q.H, q.I = 2, 512, 2048, 512
    for m in range(3):
        q.codes[m] = 256
        q.scales[m] = 256
    rc = L.moe_layer_forward(P(256), 4, P(256), None, ctypes.byref(q), 10, 0, P(256), None, None, 0, P(256), 16, None)
    assert rc == -4
    # inconsistent weight descriptor
    q.bits = 5
    rc = L.moe_layer_forward(P(256), 4, P(256), None, ctypes.byref(q), 10, 0, P(256), None, None, 0, P(256), 1 << 40,
                             None)
    assert rc == -2
    # expert call without any output
    q.bits = 2
    rc = L.moe_expert_ffn_q2(P(256), 4, ctypes.byref(q), 10, P(256), P(256), P(256), P(256), None, None, 0, 0, None,
                             None, P(256), 1 << 40, None)
    assert rc == -1
    # bad mode
    rc = L.moe_layer_forward(P(256), 4, P(256), None, ctypes.byref(q), 10, 0, P(256), None, None, 7, P(256), 1 << 40,
                             None)
    assert rc == -1
    assert L.moe_get_device_status(None, None) == -1
    # shared expert: routed (E != 1) weights, NULL y, bad mode, small workspace
    rc = L.moe_shared_expert_q2(P(256), 4, ctypes.byref(q), P(256), 0, 0, P(256), 1 << 40, None)
    assert rc == -1 and b"one expert" in L.moe_last_error_string()
    q.E = 1
    rc = L.moe_shared_expert_q2(P(256), 4, ctypes.byref(q), None, 0, 0, P(256), 1 << 40, None)
    assert rc == -1 and b"y is NULL" in L.moe_last_error_string()
    rc = L.moe_shared_expert_q2(P(256), 4, ctypes.byref(q), P(256), 1, 4, P(256), 1 << 40, None)
    assert rc == -1
    rc = L.moe_shared_expert_q2(P(256), 4, ctypes.byref(q), P(256), 1, 0, P(256), 16, None)
    assert rc == -4
    need = L.moe_workspace_bytes(4, 2048, 512, 1, 1, 2)
    assert 0 < need < moeq.workspace_bytes(4, 2048, 512, 512, 10)


def test_binding_refuses_host_tensors():
    import torch

    x = torch.zeros(4, 128)
    with pytest.raises(ValueError):
        moeq.quantize_act(x)
