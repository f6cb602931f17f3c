"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: activation quantisation, routing indices, the permutation.
Routing weights within W_REL relative: w_j = exp(L_j - L_0) / sum, so an error
dL in every fp32 logit moves w_j by at most about 2 * max|dL| * w_j; fp32
sums of H = 2048 products of N(0,1) x N(0,0.02) values carry |dL| of a few
1e-6, hence W_REL = 1e-5.  Layer outputs within 2e-3 x RMS(output) (max
abs error), allowing only the alternative int8 roundings of SwiGLU values that
the oracle itself reports as lying within DELTA of a rounding boundary (in
units of the quantisation step).  DELTA follows from each path's arithmetic:
the GEMV path forms G and U from exact integer block dots with fp32 FMAs
(relative error ~1e-7, so |dh/s| <= 127 * 1e-7 * few << 1e-3); the tensor-core
path accumulates 2 * H / 16 = 256 MMAs of K = 16 in the fp32 TMEM accumulator,
which rounds toward zero at each step: relative error up to 256 * 2^-24 per
accumulator (~1.5e-5, measured 2.7e-5 on G*U), i.e. |dh/s| up to 127 * 3e-5
~ 4e-3.  With 3-bit weights the tensor-core path splits the weight panel into
fp16 hi + lo as well and spends 3 MMAs per product (384 per accumulator), so
its bound grows by 3/2 to ~6e-3.  The warp-level int8 path (mode 3) forms the
same exact integer block dots as the GEMV path and scales them with fp32 FMAs,
so it shares the GEMV bound for either bit width.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle.checks import compare_layer_output, margin_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3
W_REL = 1e-5
DELTA = {1: 1e-3, 2: 4e-3, 3: 1e-3}  # GEMV, tcgen05 GEMM, warp-level int8 GEMM
DELTA3 = {1: 1e-3, 2: 6e-3, 3: 1e-3}  # the same with 3-bit weights


def _w_close(w_dev, w_ref):
    w_dev = np.asarray(w_dev, np.float64)
    w_ref = np.asarray(w_ref, np.float64)
    return bool((np.abs(w_dev - w_ref) <= W_REL * w_ref + 1e-7).all())


def _dev():
    return torch.device("cuda:0")


class LayerCase:
    """A layer on the device plus host copies for the oracle."""

    def __init__(self, shape, seed=0, skew=False, device="cuda"):
        self.shape = shape
        self.layer = synth.make_layer(shape, seed=seed, device=device, skew=skew)
        self.np = self.layer.numpy()
        self.dev = self.layer.to(_dev())
        torch.cuda.synchronize()  # weights complete before any call reads them
        import quantized_mixture_experts_token_b300 as moeq

        self.W = moeq.ExpertWeights.from_layer(self.dev)

    def x(self, T, seed=1, stream=0, margin=True):
        x = synth.make_x(T, self.shape.H, seed=seed, stream=stream)
        if margin and T > 0:
            x = margin_inputs(x, self.np[0], self.np[1], self.shape.k, seed)
        return x

    def oracle(self, x, tokens=None, residual=False):
        Wr, b, c, s = self.np
        return oracle.layer(x.numpy(), Wr, b, c, s, self.shape.bits, self.shape.k, residual=residual,
                            tokens=tokens, detail=True)

    def check_y(self, y_dev, ref, rms=None, delta=DELTA[2]):
        c, s = self.np[2][2], self.np[3][2]
        return compare_layer_output(y_dev, ref, c, s, self.shape.bits, tol=TOL, rms=rms, delta=delta)


@pytest.fixture(scope="module")
def tiny(cuda_lib):
    return LayerCase(synth.TINY, seed=0, device="cpu")


@pytest.fixture(scope="module")
def full(cuda_lib):
    return LayerCase(synth.FULL, seed=0, device="cuda")


@pytest.fixture(scope="module")
def full_skew(cuda_lib):
    return LayerCase(synth.FULL, seed=2, skew=True, device="cuda")


@pytest.fixture(scope="module")
def tiny3(cuda_lib):
    return LayerCase(synth.LayerShape(H=256, I=128, E=16, k=2, bits=3), seed=3, device="cpu")


@pytest.fixture(scope="module")
def full3(cuda_lib):
    return LayerCase(synth.FULL3, seed=1, device="cuda")


@pytest.fixture(scope="module")
def shared_tiny(cuda_lib):
    return LayerCase(synth.LayerShape(H=256, I=128, E=1, k=1), seed=6, device="cpu")


@pytest.fixture(scope="module")
def shared_full(cuda_lib):
    return LayerCase(synth.LayerShape(H=2048, I=512, E=1, k=1), seed=8, device="cuda")


def _ws(moeq, T, shape):
    return moeq.workspace(T, shape.H, shape.I, shape.E, shape.k, shape.bits, device=_dev())


# ------------------------------------------------------------ quantiser


@pytest.mark.parametrize("T,H", [(3, 128), (64, 256), (4096, 2048)])
def test_quantize_act_bit_exact(cuda_lib, T, H):
    x = synth.make_x(T, H, seed=T) * 3
    x[0, :32] = torch.tensor([127, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -127] + [0.0] * 24)  # exact ties
    x[0, 32:64] = 0.0  # a zero block
    if T > 1:
        x[1] *= 1e-30  # tiny scales
    q, s = cuda_lib.quantize_act(x.to(_dev()))
    qo, so = oracle.quantize_block32(x.numpy())
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


# ---------------------------------------------------------------- routing


def _check_routing(case, x, idx, w):
    L = oracle.router_logits(x.numpy(), case.np[0], case.np[1])
    io, wo = oracle.topk_softmax(L, case.shape.k)
    assert np.array_equal(idx.cpu().numpy(), io)
    assert _w_close(w.cpu().numpy(), wo)
    return io


@pytest.mark.parametrize("T", [1, 8, 64, 200])
def test_route_topk_tiny(tiny, cuda_lib, T):
    x = tiny.x(T, seed=T)
    ws = _ws(cuda_lib, T, tiny.shape)
    idx, w = cuda_lib.route_topk(x.to(_dev()), tiny.dev.Wr, None, tiny.shape.k, ws)
    _check_routing(tiny, x, idx, w)


@pytest.mark.parametrize("T", [1, 8, 64, 4096])
def test_route_topk_full(full, full_skew, cuda_lib, T):
    for case in (full, full_skew):
        x = case.x(T, seed=10 + T)
        ws = _ws(cuda_lib, T, case.shape)
        idx, w = cuda_lib.route_topk(x.to(_dev()), case.dev.Wr, case.dev.bias, case.shape.k, ws)
        _check_routing(case, x, idx, w)


@pytest.mark.parametrize("n_tied", [512, 40])
@pytest.mark.parametrize("T,fused", [(1, True), (2, True), (8, False)])
def test_routing_heavy_ties_full(full, cuda_lib, n_tied, T, fused):
    """Exact ties among more than 32 logits at the top take the warp top-k's
    rare paths (more candidates than lanes).  x = 0 gives logits equal to the
    bias: all 512 tied, or the first 40 at +1 and the rest at 0.  Ties go to the
    lower expert index; the oracle's stable sort says the same."""
    shape = full.shape
    x = torch.zeros(T, shape.H)
    bias = torch.zeros(shape.E)
    if n_tied < shape.E:
        bias[:n_tied] = 1.0
    L = oracle.router_logits(x.numpy(), full.dev.Wr.cpu().numpy(), bias.numpy())
    ref_idx, ref_w = oracle.topk_softmax(L, shape.k)
    ws = _ws(cuda_lib, T, shape)
    if fused:  # through the fused decode tail (in-CTA ranking for T <= 2)
        _, idx, w = cuda_lib.layer_forward(x.to(_dev()), full.W, full.dev.Wr, bias.to(_dev()), shape.k, ws,
                                           want_routing=True)
    else:
        idx, w = cuda_lib.route_topk(x.to(_dev()), full.dev.Wr, bias.to(_dev()), shape.k, ws)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.allclose(w.cpu().numpy(), ref_w, rtol=1e-6, atol=0)
    assert cuda_lib.device_status() == 0


# ------------------------------------------------------------- permutation


@pytest.mark.parametrize("T,E,k", [(1, 512, 10), (8, 512, 10), (64, 16, 2), (1000, 7, 3), (4096, 512, 10),
                                   (33, 1024, 32), (4096, 16, 2)])
def test_permute_bit_exact(cuda_lib, T, E, k):
    rng = np.random.default_rng(T * 31 + E)
    # skewed expert popularity with some experts never chosen
    p = rng.zipf(1.3, size=E).astype(np.float64)
    p[rng.random(E) < 0.1] = 0
    p /= p.sum()
    idx = np.stack([rng.choice(E, k, replace=False, p=p if (p > 0).sum() >= k else None) for _ in range(T)])
    idx = idx.astype(np.int32)
    ws = cuda_lib.workspace(T, 128, 128, E, k, device=_dev())
    out = cuda_lib.permute(torch.from_numpy(idx).to(_dev()), E, ws)
    ref = oracle.permute(idx, E)
    for key in ("counts", "offsets", "perm_tok", "perm_slot", "inv"):
        assert np.array_equal(out[key].cpu().numpy().reshape(ref[key].shape), ref[key]), key


# ------------------------------------------------------------------ experts


def _expert_case(case, cuda_lib, T, mode, residual=False, seed=5):
    x = case.x(T, seed=seed)
    xd = x.to(_dev())
    ws = _ws(cuda_lib, T, case.shape)
    idx, w = cuda_lib.route_topk(xd, case.dev.Wr, case.dev.bias, case.shape.k, ws)
    perm = cuda_lib.permute(idx, case.shape.E, ws)
    out = cuda_lib.expert_ffn(xd, case.W, case.shape.k, perm, w, want_y=True, want_sorted=True,
                              residual=residual, mode=mode, want_h=True, ws=ws)
    torch.cuda.synchronize()
    return x, idx, w, perm, out


def _check_h_codes(ref, qh_dev, sh_dev, inv, delta):
    """Device int8 SwiGLU codes equal the oracle's except at oracle-reported near-ties (by one step)."""
    n, k, I = ref["qh"].shape
    q = qh_dev[inv.reshape(-1)].reshape(n, k, I).astype(np.int32)
    s = sh_dev[inv.reshape(-1)].reshape(n, k, I // 32)
    diff = q - ref["qh"].astype(np.int32)
    bad = diff != 0
    assert (np.abs(diff) <= 1).all()
    assert (ref["hdist"][bad] < delta).all(), "a code differs away from a rounding boundary"
    assert np.allclose(s, ref["sh"], rtol=delta / 64, atol=0)
    return int(bad.sum())


@pytest.mark.parametrize("mode", [1, 2, 3])
@pytest.mark.parametrize("T", [64, 600])
def test_expert_ffn_tiny(tiny, cuda_lib, mode, T):
    x, idx, w, perm, out = _expert_case(tiny, cuda_lib, T, mode)
    ref = tiny.oracle(x)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    _check_h_codes(ref, out["qh"].cpu().numpy(), out["sh"].cpu().numpy(), perm["inv"].cpu().numpy(), DELTA[mode])
    tiny.check_y(out["y"].cpu().numpy(), ref, delta=DELTA[mode])
    # the per-pair outputs combined on the device reproduce y
    y2 = cuda_lib.combine(out["out_sorted"], perm["inv"], w)
    assert np.abs(y2.cpu().numpy() - out["y"].cpu().numpy()).max() <= 1e-5 * float(out["y"].abs().max())


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_expert_ffn_full_sampled(full_skew, cuda_lib, mode):
    T = 256 if mode == 1 else 4096
    x, idx, w, perm, out = _expert_case(full_skew, cuda_lib, T, mode, seed=7)
    counts = perm["counts"].cpu().numpy()
    assert (counts == 0).any(), "the skewed router must leave some experts without tokens"
    tokens = np.random.default_rng(0).choice(T, 96, replace=False).astype(np.int32)
    ref = full_skew.oracle(x, tokens=tokens)
    assert np.array_equal(idx.cpu().numpy()[tokens], ref["idx"])
    inv = perm["inv"].cpu().numpy()[tokens]
    _check_h_codes(ref, out["qh"].cpu().numpy(), out["sh"].cpu().numpy(), inv, DELTA[mode])
    full_skew.check_y(out["y"].cpu().numpy()[tokens], ref, delta=DELTA[mode])


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_expert_ffn_tiny_3bit(tiny3, cuda_lib, mode):
    T = 600
    x, idx, w, perm, out = _expert_case(tiny3, cuda_lib, T, mode)
    ref = tiny3.oracle(x)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    _check_h_codes(ref, out["qh"].cpu().numpy(), out["sh"].cpu().numpy(), perm["inv"].cpu().numpy(), DELTA3[mode])
    tiny3.check_y(out["y"].cpu().numpy(), ref, delta=DELTA3[mode])


@pytest.mark.parametrize("T,mode", [(8, 1), (1024, 2), (1024, 3)])
def test_expert_ffn_full_3bit(full3, cuda_lib, T, mode):
    x, idx, w, perm, out = _expert_case(full3, cuda_lib, T, mode, seed=11)
    tokens = np.arange(T, dtype=np.int32) if T <= 8 else \
        np.random.default_rng(2).choice(T, 48, replace=False).astype(np.int32)
    ref = full3.oracle(x, tokens=tokens)
    assert np.array_equal(idx.cpu().numpy()[tokens], ref["idx"])
    inv = perm["inv"].cpu().numpy()[tokens]
    _check_h_codes(ref, out["qh"].cpu().numpy(), out["sh"].cpu().numpy(), inv, DELTA3[mode])
    full3.check_y(out["y"].cpu().numpy()[tokens], ref, delta=DELTA3[mode])


def _shared_case(case, cuda_lib, T, mode, tokens=None):
    """The shared expert through moe_shared_expert_q2, fresh and accumulated onto y0,
    against the oracle's single-expert layer (E = 1, k = 1: weight 1 for every token)."""
    x = case.x(T, seed=40 + T, margin=False)
    xd = x.to(_dev())
    y = cuda_lib.shared_expert(xd, case.W, mode=mode)
    y0 = synth.make_x(T, case.shape.H, seed=50 + T).to(_dev())
    y_acc = cuda_lib.shared_expert(xd, case.W, y=y0.clone(), accumulate=True, mode=mode)
    torch.cuda.synchronize()
    ref = case.oracle(x, tokens=tokens)
    rows = slice(None) if tokens is None else tokens
    yh = y.cpu().numpy()
    case.check_y(yh[rows], ref, delta=DELTA[mode])
    # accumulate adds the same values onto y0 (fp32 atomics: one rounding per addition)
    added = (y_acc - y0).cpu().numpy()
    scale = float(np.abs(y0.cpu().numpy()).max() + np.abs(yh).max())
    assert np.abs(added - yh).max() <= 1e-5 * scale
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("T,mode", [(5, 1), (64, 1), (600, 2), (600, 3)])
def test_shared_expert_tiny(shared_tiny, cuda_lib, T, mode):
    _shared_case(shared_tiny, cuda_lib, T, mode)


@pytest.mark.parametrize("T,mode", [(8, 1), (1024, 2)])
def test_shared_expert_full(shared_full, cuda_lib, T, mode):
    tokens = None if T <= 8 else np.random.default_rng(3).choice(T, 48, replace=False).astype(np.int32)
    _shared_case(shared_full, cuda_lib, T, mode, tokens)


def test_shared_expert_rejects_routed_weights(full, cuda_lib):
    with pytest.raises(cuda_lib.MoeqError):
        cuda_lib.shared_expert(torch.zeros(4, 2048, device=_dev()), full.W)


def test_prefill_experts_repeatable(full_skew, cuda_lib):
    """Repeated prefill expert calls on the same inputs give bit-identical SwiGLU
    codes, scales and per-pair outputs (y itself sums the k pairs of a token with
    fp32 atomics, whose order may vary)."""
    T = 4096
    x = full_skew.x(T, seed=7).to(_dev())
    ws = _ws(cuda_lib, T, full_skew.shape)
    idx, w = cuda_lib.route_topk(x, full_skew.dev.Wr, full_skew.dev.bias, full_skew.shape.k, ws)
    perm = cuda_lib.permute(idx, full_skew.shape.E, ws)
    first = None
    for _ in range(4):
        out = cuda_lib.expert_ffn(x, full_skew.W, full_skew.shape.k, perm, w, want_y=True, want_sorted=True,
                                  mode=2, want_h=True, ws=ws)
        torch.cuda.synchronize()
        cur = [out[n].cpu().numpy() for n in ("qh", "sh", "out_sorted")]
        if first is None:
            first = cur
            continue
        for a, b in zip(first, cur):
            assert np.array_equal(a, b)
    assert cuda_lib.device_status() == 0


# -------------------------------------------------------------- whole layer


@pytest.mark.parametrize("T", [1, 8, 16, 64])
def test_layer_forward_decode_full(full, cuda_lib, T):
    x = full.x(T, seed=100 + T)
    ws = _ws(cuda_lib, T, full.shape)
    y, idx, w = cuda_lib.layer_forward(x.to(_dev()), full.W, full.dev.Wr, None, full.shape.k, ws, want_routing=True)
    torch.cuda.synchronize()
    ref = full.oracle(x)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert _w_close(w.cpu().numpy(), ref["w"])
    full.check_y(y.cpu().numpy(), ref, delta=DELTA[1])
    # a second call on the same workspace (re-armed counters) gives the same result
    y2 = cuda_lib.layer_forward(x.to(_dev()), full.W, full.dev.Wr, None, full.shape.k, ws)
    torch.cuda.synchronize()
    assert np.abs(y2.cpu().numpy() - y.cpu().numpy()).max() <= 1e-6 * float(y.abs().max())


def test_layer_forward_auto_mid_size(full, cuda_lib):
    """A 200-token call in auto mode (the GEMV expert path above the fused decode range)."""
    T = 200
    x = full.x(T, seed=300)
    ws = _ws(cuda_lib, T, full.shape)
    y, idx, w = cuda_lib.layer_forward(x.to(_dev()), full.W, full.dev.Wr, None, full.shape.k, ws, want_routing=True)
    torch.cuda.synchronize()
    tokens = np.random.default_rng(4).choice(T, 48, replace=False).astype(np.int32)
    ref = full.oracle(x, tokens=tokens)
    assert np.array_equal(idx.cpu().numpy()[tokens], ref["idx"])
    full.check_y(y.cpu().numpy()[tokens], ref, delta=DELTA[1])
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("residual", [False, True])
def test_layer_forward_prefill_full(full_skew, cuda_lib, residual):
    T = 4096
    x = full_skew.x(T, seed=200)
    ws = _ws(cuda_lib, T, full_skew.shape)
    y, idx, w = cuda_lib.layer_forward(x.to(_dev()), full_skew.W, full_skew.dev.Wr, full_skew.dev.bias,
                                       full_skew.shape.k, ws, residual=residual, want_routing=True)
    torch.cuda.synchronize()
    tokens = np.random.default_rng(1).choice(T, 64, replace=False).astype(np.int32)
    ref = full_skew.oracle(x, tokens=tokens, residual=residual)
    assert np.array_equal(idx.cpu().numpy()[tokens], ref["idx"])
    full_skew.check_y(y.cpu().numpy()[tokens], ref)
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_layer_forward_tiny_modes(tiny, cuda_lib, mode):
    T = 256 if mode == 1 else 4096
    x = tiny.x(T, seed=300)
    ws = _ws(cuda_lib, T, tiny.shape)
    y, idx, w = cuda_lib.layer_forward(x.to(_dev()), tiny.W, tiny.dev.Wr, None, tiny.shape.k, ws, mode=mode,
                                       want_routing=True)
    torch.cuda.synchronize()
    ref = tiny.oracle(x)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    tiny.check_y(y.cpu().numpy(), ref, delta=DELTA[mode])


def test_zero_tokens(tiny, cuda_lib):
    ws = _ws(cuda_lib, 0, tiny.shape)
    x = torch.zeros(0, tiny.shape.H, device=_dev())
    y = cuda_lib.layer_forward(x, tiny.W, tiny.dev.Wr, None, tiny.shape.k, ws)
    assert y.shape == (0, tiny.shape.H)


def test_zero_input_gives_zero_output(tiny, cuda_lib):
    T = 32
    x = torch.zeros(T, tiny.shape.H)
    ws = _ws(cuda_lib, T, tiny.shape)
    for mode in (1, 2, 3):
        y, idx, w = cuda_lib.layer_forward(x.to(_dev()), tiny.W, tiny.dev.Wr, None, tiny.shape.k, ws, mode=mode,
                                           want_routing=True)
        torch.cuda.synchronize()
        assert not y.cpu().numpy().any()
        assert idx.cpu().numpy().tolist() == [[0, 1]] * T
        assert np.allclose(w.cpu().numpy(), 0.5)


def test_device_status_clean(cuda_lib):
    assert cuda_lib.device_status() == 0
