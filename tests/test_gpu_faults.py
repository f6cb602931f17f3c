"""Failure detection on the GPU without a GPU fault.

* A forced wait timeout: moe_set_wait_limit shortens the bound of every
  pipeline wait to 1 ns, so waits that are not already satisfied give up at
  once.  Nothing is broken: every copy the kernels issue still lands, and each
  kernel drains its own copies and tensor-core work (under a separate, fixed
  bound) before it returns.  The device status must report
  MOEQ_STATUS_WAIT_TIMEOUT, and the next calls with the default bound on the
  same workspace must give the results of a clean run.
* Bad indices: an expert index out of range or repeated in a row, and a
  corrupted permutation handed to the expert kernels, are skipped by the
  kernels' own bounds checks and reported as MOEQ_STATUS_BAD_INDEX.
"""
import numpy as np
import pytest
import torch

import synth
from test_gpu_parity import LayerCase, _ws

pytestmark = pytest.mark.gpu


def _dev():
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def full(cuda_lib):
    return LayerCase(synth.FULL, seed=0, device="cuda")


@pytest.fixture(scope="module")
def tiny(cuda_lib):
    return LayerCase(synth.TINY, seed=0, device="cpu")


def _layer(cuda_lib, case, x, ws, mode):
    return cuda_lib.layer_forward(x, case.W, case.dev.Wr, case.dev.bias, case.shape.k, ws, residual=True, mode=mode)


@pytest.mark.parametrize("T,mode", [(1, 0), (8, 0), (2048, 2)])
def test_forced_wait_timeout_is_reported_and_recovered(full, cuda_lib, T, mode):
    x = full.x(T, seed=900 + T).to(_dev())
    ws = _ws(cuda_lib, T, full.shape)
    y_clean = _layer(cuda_lib, full, x, ws, mode).clone()
    assert cuda_lib.device_status() == 0
    try:
        cuda_lib.set_wait_limit(1)
        for _ in range(2):
            _layer(cuda_lib, full, x, ws, mode)
        st = cuda_lib.device_status()
    finally:
        cuda_lib.set_wait_limit(0)
    assert st & cuda_lib.STATUS_WAIT_TIMEOUT, f"status 0x{st:x}"
    assert cuda_lib.device_status() == 0  # read-and-clear
    for _ in range(2):
        y = _layer(cuda_lib, full, x, ws, mode)
        torch.cuda.synchronize()
        assert cuda_lib.device_status() == 0
        scale = float(y_clean.abs().max())
        assert float((y - y_clean).abs().max()) <= 1e-5 * scale


def test_set_wait_limit_rejects_long_limits(cuda_lib):
    with pytest.raises(cuda_lib.MoeqError):
        cuda_lib.set_wait_limit(61 * 10**9)


def test_bad_expert_index_through_permute_and_combine(cuda_lib):
    T, k, E, H = 40, 3, 16, 128
    rng = np.random.default_rng(0)
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[3, 1] = E + 5          # out of range
    idx[7, 2] = -1             # out of range
    idx[9, 2] = idx[9, 0]      # the same expert twice in one row
    for noalloc in (False, True):
        d = torch.from_numpy(idx).to(_dev())
        if noalloc:
            perm = cuda_lib.permute_noalloc(d, E)
        else:
            perm = cuda_lib.permute(d, E, cuda_lib.workspace(T, 128, 128, E, k, device=_dev()))
        st = cuda_lib.device_status()
        assert st & cuda_lib.STATUS_BAD_INDEX
        inv = perm["inv"].cpu().numpy()
        assert inv[3, 1] == -1 and inv[7, 2] == -1
        # combine skips the rejected pairs (and reports them) instead of reading out of bounds
        D = torch.randn(T * k, H, device=_dev())
        w = torch.full((T, k), 1.0 / k, device=_dev())
        y = cuda_lib.combine(D, perm["inv"], w)
        torch.cuda.synchronize()
        assert torch.isfinite(y).all()
        assert cuda_lib.device_status() & cuda_lib.STATUS_BAD_INDEX
        yh = y.cpu().numpy().astype(np.float64)
        Dh = D.cpu().numpy().astype(np.float64)
        want = np.zeros(H)
        for j in range(k):
            if inv[3, j] >= 0:
                want += Dh[inv[3, j]] / k
        assert np.allclose(yh[3], want, rtol=1e-5, atol=1e-6)
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_corrupted_permutation_into_the_experts(tiny, cuda_lib, mode):
    T = 64
    x = tiny.x(T, seed=950).to(_dev())
    ws = _ws(cuda_lib, T, tiny.shape)
    idx, w = cuda_lib.route_topk(x, tiny.dev.Wr, None, tiny.shape.k, ws)
    perm = cuda_lib.permute(idx, tiny.shape.E, ws)
    clean = cuda_lib.expert_ffn(x, tiny.W, tiny.shape.k, perm, w, want_sorted=True, mode=mode, ws=ws)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    bad = {key: v.clone() for key, v in perm.items()}
    bad["perm_tok"][5] = T + 100
    bad["perm_tok"][11] = -7
    bad["perm_slot"][20] = tiny.shape.k + 3
    if mode != 1:
        # the grouped GEMMs' scratch (operand images included) poisoned with NaN bit patterns:
        # the rejected pairs' rows are never written, and nothing of them may reach y
        ws.fill_(0xFF)
    out = cuda_lib.expert_ffn(x, tiny.W, tiny.shape.k, bad, w, want_sorted=True, mode=mode, ws=ws)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() & cuda_lib.STATUS_BAD_INDEX
    assert torch.isfinite(out["y"]).all()
    # offsets that are not a prefix sum: no expert work at all, y = 0
    bad2 = {key: v.clone() for key, v in perm.items()}
    bad2["offsets"][3] = 10**6
    out2 = cuda_lib.expert_ffn(x, tiny.W, tiny.shape.k, bad2, w, mode=mode, ws=ws)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() & cuda_lib.STATUS_BAD_INDEX
    assert not out2["y"].any()
    # and the next clean call is unaffected
    again = cuda_lib.expert_ffn(x, tiny.W, tiny.shape.k, perm, w, want_sorted=True, mode=mode, ws=ws)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    # (the GEMV path sums its I-blocks into out_sorted with fp32 atomics: order may vary)
    scale = float(clean["out_sorted"].abs().max())
    assert float((again["out_sorted"] - clean["out_sorted"]).abs().max()) <= 1e-6 * scale
