"""GPU parity of the paths the headline measurements run: the 3-bit verify
window through the fused decode tail, the 3-bit 16,384-token prefill chunk, a
stack of decode layers chained by programmatic dependent launch inside one CUDA
graph over one shared workspace, in-CTA routing at two tokens, and the
standalone gather-combine against the oracle's per-pair outputs.

Tolerances are those of test_gpu_parity (see its docstring).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle.checks import small_gap_tokens
from test_gpu_parity import DELTA, DELTA3, LayerCase, _w_close, _ws

pytestmark = pytest.mark.gpu


def _dev():
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def full(cuda_lib):
    return LayerCase(synth.FULL, seed=0, device="cuda")


@pytest.fixture(scope="module")
def full3(cuda_lib):
    return LayerCase(synth.FULL3, seed=1, device="cuda")


@pytest.fixture(scope="module")
def tiny(cuda_lib):
    return LayerCase(synth.TINY, seed=0, device="cpu")


# ------------------------------------------------- 3-bit: verify window, prefill


def test_layer_forward_3bit_verify_window(full3, cuda_lib):
    """64 tokens (4 drafts x 16 sequences) in one call: the fused decode tail
    (router kernel quantises x in natural order for 3-bit) and the GEMV experts."""
    T = 64
    x = full3.x(T, seed=500)
    ws = _ws(cuda_lib, T, full3.shape)
    y, idx, w = cuda_lib.layer_forward(x.to(_dev()), full3.W, full3.dev.Wr, None, full3.shape.k, ws,
                                       want_routing=True)
    torch.cuda.synchronize()
    ref = full3.oracle(x)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert _w_close(w.cpu().numpy(), ref["w"])
    full3.check_y(y.cpu().numpy(), ref, delta=DELTA3[1])
    assert cuda_lib.device_status() == 0


def test_layer_forward_3bit_prefill_16k(full3, cuda_lib):
    """The 16,384-token 3-bit chunk with uniform routing (163,840 pairs), on
    48 sampled tokens."""
    T = 16384
    x = full3.x(T, seed=501)
    ws = _ws(cuda_lib, T, full3.shape)
    y, idx, w = cuda_lib.layer_forward(x.to(_dev()), full3.W, full3.dev.Wr, None, full3.shape.k, ws,
                                       want_routing=True)
    torch.cuda.synchronize()
    tokens = np.random.default_rng(5).choice(T, 48, replace=False).astype(np.int32)
    ref = full3.oracle(x, tokens=tokens)
    assert np.array_equal(idx.cpu().numpy()[tokens], ref["idx"])
    full3.check_y(y.cpu().numpy()[tokens], ref, delta=DELTA3[2])
    assert cuda_lib.device_status() == 0


# ------------------------------------------------ in-CTA routing at two tokens


@pytest.mark.parametrize("same", [False, True])
def test_layer_forward_two_tokens(full, cuda_lib, same):
    """T = 2 ranks the router logits inside every expert CTA.  With two equal
    tokens only 10 of the 20 launched units have an expert: the other CTAs leave
    early while their activation copy is in flight."""
    T = 2
    x = full.x(T, seed=600)
    if same:
        x[1] = x[0]
    ws = _ws(cuda_lib, T, full.shape)
    for _ in range(2):
        y, idx, w = cuda_lib.layer_forward(x.to(_dev()), full.W, full.dev.Wr, None, full.shape.k, ws,
                                           want_routing=True)
        torch.cuda.synchronize()
        ref = full.oracle(x)
        assert np.array_equal(idx.cpu().numpy(), ref["idx"])
        assert _w_close(w.cpu().numpy(), ref["w"])
        full.check_y(y.cpu().numpy(), ref, delta=DELTA[1])
    if same:
        assert np.array_equal(ref["idx"][0], ref["idx"][1])
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("T", [1, 2])
def test_layer_forward_without_routing_outputs(full, cuda_lib, T):
    """The routing outputs of moe_layer_forward are optional: with none asked
    for, the in-CTA routing (T <= 2) writes nothing for any token and y is the
    same as with them."""
    x = full.x(T, seed=610).to(_dev())
    ws = _ws(cuda_lib, T, full.shape)
    y_with, _, _ = cuda_lib.layer_forward(x, full.W, full.dev.Wr, None, full.shape.k, ws, want_routing=True)
    y_without = cuda_lib.layer_forward(x, full.W, full.dev.Wr, None, full.shape.k, ws)
    torch.cuda.synchronize()
    ref = full.oracle(x.cpu())
    full.check_y(y_without.cpu().numpy(), ref, delta=DELTA[1])
    # the same kernels on the same inputs; only the fp32 atomics' order may differ
    assert np.allclose(y_with.cpu().numpy(), y_without.cpu().numpy(), rtol=1e-5, atol=1e-6)
    assert cuda_lib.device_status() == 0


# ------------------------------------------- a decode stack inside a CUDA graph


@pytest.fixture(scope="module")
def stack(cuda_lib):
    shape = synth.FULL
    layers = [synth.make_layer(shape, seed=0, layer=l, device=_dev()) for l in range(4)]
    torch.cuda.synchronize()
    return shape, layers


@pytest.mark.parametrize("T", [1, 8])
def test_decode_stack_in_cuda_graph(stack, cuda_lib, T):
    """x_{l+1} = x_l + moe_l(x_l) through 4 layers, captured once in a CUDA
    graph (programmatic dependent launch between the kernels, one workspace,
    the router's arrival counter re-armed by every call) and replayed twice.
    Each layer is checked against the oracle on the device's own input x_l;
    a token whose fp64 routing margin at that layer is below 1e-3 is only
    checked where its routing matches."""
    shape, layers = stack
    Ws = [cuda_lib.ExpertWeights.from_layer(l) for l in layers]
    nl = len(layers)
    ws = _ws(cuda_lib, T, shape)
    xs = [torch.empty(T, shape.H, device=_dev()) for _ in range(nl + 1)]
    x0 = synth.make_x(T, shape.H, seed=700 + T)
    xs[0].copy_(x0)

    def run():
        for l in range(nl):
            # want_routing=False keeps the graph free of allocations; routing is read
            # back through a second, eager pass below
            cuda_lib.layer_forward(xs[l], Ws[l], layers[l].Wr, None, shape.k, ws, residual=True, y=xs[l + 1])

    run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    skipped = 0
    for rep in range(2):
        for t in xs[1:]:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        # (replays need not agree bit for bit: the experts add into y with fp32
        # atomics, and the residual chain carries those roundings on; each
        # replay is checked against the oracle on its own inputs)
        skipped += _check_stack(cuda_lib, shape, layers, Ws, ws, [t.cpu().numpy().copy() for t in xs], T)
    print(f"decode stack T={T}: {skipped} token-layers skipped for a routing margin below 1e-3")
    assert skipped <= 2 * nl * T // 4
    assert cuda_lib.device_status() == 0


def _check_stack(cuda_lib, shape, layers, Ws, ws, xh, T):
    from oracle.checks import compare_layer_output

    skipped = 0
    for l in range(len(layers)):
        lnp = layers[l].numpy()
        ref = oracle.layer(xh[l], lnp[0], None, lnp[2], lnp[3], shape.bits, shape.k, detail=True)
        _, idx_dev, _ = cuda_lib.layer_forward(torch.from_numpy(xh[l]).to(_dev()), Ws[l], layers[l].Wr, None, shape.k,
                                               ws, residual=True, y=torch.empty(T, shape.H, device=_dev()),
                                               want_routing=True)
        idx_dev = idx_dev.cpu().numpy()
        L = oracle.router_logits(xh[l], lnp[0], None)
        near = set(small_gap_tokens(L, shape.k, 1e-3).tolist())
        keep = [t for t in range(T) if t not in near or np.array_equal(idx_dev[t], ref["idx"][t])]
        skipped += T - len(keep)
        for t in range(T):
            if t not in near:
                assert np.array_equal(idx_dev[t], ref["idx"][t]), (l, t)
        dy = xh[l + 1].astype(np.float64) - xh[l].astype(np.float64)
        sub = {key: v[keep] for key, v in ref.items()}
        rms = float(np.sqrt(np.mean(ref["y"].astype(np.float64) ** 2)))
        compare_layer_output(dy[keep], sub, lnp[2][2], lnp[3][2], shape.bits, rms=rms, delta=DELTA[1])
    return skipped


# --------------------------------------------------- combine against the oracle


@pytest.mark.parametrize("case_name,T", [("tiny", 64), ("full", 8)])
@pytest.mark.parametrize("residual", [False, True])
def test_combine_against_oracle(request, cuda_lib, case_name, T, residual):
    """moe_combine on the oracle's own per-pair outputs D and weights reproduces
    the oracle's y (fp32 sums of k products, j ascending)."""
    case = request.getfixturevalue(case_name)
    x = case.x(T, seed=800 + T)
    ref = case.oracle(x, residual=residual)
    k, H = case.shape.k, case.shape.H
    perm = oracle.permute(ref["idx"], case.shape.E)
    D = np.zeros((T * k, H), np.float32)
    D[perm["inv"].reshape(-1)] = ref["D"].reshape(T * k, H).astype(np.float32)
    y = cuda_lib.combine(torch.from_numpy(D).to(_dev()), torch.from_numpy(perm["inv"]).to(_dev()),
                         torch.from_numpy(ref["w"]).to(_dev()),
                         residual_x=x.to(_dev()) if residual else None)
    torch.cuda.synchronize()
    yd = y.cpu().numpy().astype(np.float64)
    # bound: fp32 rounding of D, of each product and of each of the k + 1 additions
    mag = np.einsum("tj,tjh->th", np.abs(ref["w"].astype(np.float64)), np.abs(ref["D"]))
    if residual:
        mag += np.abs(x.numpy().astype(np.float64))
    bound = (k + 3) * 2.0**-24 * mag + 1e-30
    assert (np.abs(yd - ref["y"].astype(np.float64)) <= bound + 2.0**-24 * np.abs(ref["y"])).all()
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("H,T,mode", [(384, 37, 1), (256, 3, 1), (384, 600, 2), (384, 600, 3)])
def test_other_hidden_sizes(cuda_lib, H, T, mode):
    """The expert kernels at hidden sizes other than the model's (12 and 8
    K-blocks): the decode kernel with more tokens than one pass holds (T = 37),
    and the grouped GEMMs with H an odd multiple of 128 (the tcgen05 down GEMM's
    last item then holds one 128-row block instead of two)."""
    shape = synth.LayerShape(H=H, I=128, E=8, k=2)
    case = LayerCase(shape, seed=31, device="cpu")
    x = case.x(T, seed=900 + H)
    ws = _ws(cuda_lib, T, shape)
    y, idx, w = cuda_lib.layer_forward(x.to(_dev()), case.W, case.dev.Wr, None, shape.k, ws, mode=mode,
                                       want_routing=True)
    torch.cuda.synchronize()
    ref = case.oracle(x)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    case.check_y(y.cpu().numpy(), ref, delta=DELTA[mode])
    assert cuda_lib.device_status() == 0
