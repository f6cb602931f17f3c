"""moe_permute_noalloc: the permutation for callers that cannot allocate device
memory (a host framework that owns every allocation, or a hot path that must
not reach the CUDA allocator).  It uses a fixed scratch array inside the
library instead of a caller workspace; its results must equal moe_permute's,
call after call, since every call reuses (and clears) the same array.

This file is collected last on purpose: a failure here leaves every other
test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

KEYS = ("counts", "offsets", "perm_tok", "perm_slot", "inv")


def _idx(T, E, k, seed):
    rng = np.random.default_rng(seed)
    p = rng.zipf(1.3, size=E).astype(np.float64)
    p[rng.random(E) < 0.1] = 0
    p /= p.sum()
    use_p = p if (p > 0).sum() >= k else None
    return np.stack([rng.choice(E, k, replace=False, p=use_p) for _ in range(T)]).astype(np.int32)


# (2048, 1024, 32): E * ceil(T/32) = 65,536 words, the whole scratch array
@pytest.mark.parametrize("T,E,k", [(4096, 512, 10), (64, 16, 2), (1, 512, 10), (2048, 1024, 32)])
def test_noalloc_permute_matches_workspace_permute_twice(cuda_lib, T, E, k):
    dev = torch.device("cuda:0")
    ws = cuda_lib.workspace(T, 128, 128, E, k, device=dev)
    for call in range(2):  # two calls in a row: the shared scratch must not carry state over
        idx = torch.from_numpy(_idx(T, E, k, seed=1000 * call + T)).to(dev)
        ref = cuda_lib.permute(idx, E, ws)
        got = cuda_lib.permute_noalloc(idx, E)
        torch.cuda.synchronize()
        for key in KEYS:
            assert torch.equal(got[key], ref[key]), (call, key)


def test_noalloc_permute_rejects_sizes_beyond_its_scratch(cuda_lib):
    L = cuda_lib.lib()
    P = ctypes.c_void_p
    # E * ceil(T/32) = 1024 * 128 > 65536 words
    rc = L.moe_permute_noalloc(P(256), 4096, 10, 1024, P(256), P(256), P(256), P(256), P(256), None)
    assert rc == -2
    assert b"fixed scratch" in L.moe_last_error_string()


def test_noalloc_permute_zero_tokens_zeroes_counts_and_offsets(cuda_lib):
    dev = torch.device("cuda:0")
    E, k = 512, 10
    # fill the outputs with garbage first: a T = 0 call must write zeros
    idx = torch.zeros(0, k, dtype=torch.int32, device=dev)
    for _ in range(2):
        got = cuda_lib.permute_noalloc(idx, E)
        got["counts"].fill_(7)
        got["offsets"].fill_(7)
        L = cuda_lib.lib()
        P = ctypes.c_void_p
        rc = L.moe_permute_noalloc(None, 0, k, E, P(got["counts"].data_ptr()), P(got["offsets"].data_ptr()),
                                   None, None, None, P(torch.cuda.current_stream().cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()
        assert not got["counts"].any() and not got["offsets"].any()
