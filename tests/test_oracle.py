"""Pins for the CPU oracle: closed forms, brute force, library routines, invariants.

None of these checks re-types the oracle's own formulas: each compares it with
a value fixed by exact arithmetic (golden files), a different computation of
the same quantity (dense numpy fp64 matmuls, Python's stable sort, Python
big-integer bit packing), or a library routine (scipy's softmax / expit).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------- quantiser


def test_quantizer_golden():
    for case in _golden("quant_block32.json")["cases"]:
        q, s = oracle.quantize_block32(np.array(case["x"], np.float32))
        assert s.tolist() == [case["s"]], case["name"]
        assert q.tolist() == case["q"], case["name"]


def test_quantizer_roundtrip_on_grid():
    rng = np.random.default_rng(1)
    for scale in (2.0**-9, 0.25, 1.0, 3.0**-1):
        qs = rng.integers(-127, 128, size=(50, 32))
        qs[:, 0] = 127 * np.where(rng.random(50) < 0.5, 1, -1)  # the block maximum
        s = np.float32(scale)
        x = (qs.astype(np.float32) * s).astype(np.float32)
        q, s_out = oracle.quantize_block32(x.reshape(-1))
        # the amax element maps to +-127 exactly and every grid point back to its integer
        assert np.array_equal(q.reshape(50, 32), qs)


def test_quantizer_bounds_and_half_even_random():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(32 * 200).astype(np.float32) * 3
    q, s = oracle.quantize_block32(x)
    qb = q.reshape(200, 32).astype(np.int64)
    assert np.abs(qb).max() <= 127
    assert (np.abs(qb).max(axis=1) == 127).all()
    # every code is within half a step of the value (exact rational check in fp64)
    err = np.abs(x.reshape(200, 32).astype(np.float64) / s.astype(np.float64)[:, None] - qb)
    assert err.max() <= 0.5 + 1e-6


# ------------------------------------------------------------ fp16 decode


@pytest.mark.parametrize("bits,val", [(0x3C00, 1.0), (0xC000, -2.0), (0x3555, 0.333251953125), (0x7BFF, 65504.0),
                                      (0x0001, 2.0**-24), (0x0400, 2.0**-14), (0x8000, -0.0), (0x3800, 0.5)])
def test_half_decode(bits, val):
    assert oracle.half_to_double(bits) == val
    assert float(np.array([bits], np.uint16).view(np.float16)[0]) == val


# --------------------------------------------------------- weight layout


def test_weight_layout_two_bit_golden():
    g = _golden("weight_layout.json")["two_bit"]
    N, K = g["N"], g["K"]
    codes = np.frombuffer(bytes.fromhex("".join(g["codes_hex"])), np.uint8)
    scales = np.array([int(h, 16) for h in g["scales_fp16_hex"]], np.uint16)
    dense = oracle.dequantize_matrix(codes, scales, 2, N, K)
    for n in range(N):
        lv = np.array(g[f"expected_levels_row{n}"], np.float64)
        sc = np.repeat(np.array(g[f"expected_scale_row{n}"]), 32)
        assert np.array_equal(dense[n], lv * sc)


def test_weight_layout_three_bit_bigint():
    # codes c_i = (5*i + n + 3*kb) % 8 packed as a 96-bit little-endian integer
    N, K = 3, 64
    blocks = []
    want = np.zeros((N, K))
    for kb in range(K // 32):
        for n in range(N):
            word = 0
            for i in range(32):
                c = (5 * i + n + 3 * kb) % 8
                word |= c << (3 * i)
                want[n, 32 * kb + i] = c - 4
            blocks.append(word.to_bytes(12, "little"))
    codes = np.frombuffer(b"".join(blocks), np.uint8)
    scales = np.full(N * (K // 32), 0x3C00, np.uint16)
    assert np.array_equal(oracle.dequantize_matrix(codes, scales, 3, N, K), want)


def test_generator_codes_decode_to_quantised_weights():
    # the synthetic generator's packing and the oracle's accessor agree
    shape = synth.LayerShape(H=64, I=32, E=2, k=1, bits=2)
    for bits in (2, 3):
        shape = synth.LayerShape(H=64, I=32, E=2, k=1, bits=bits)
        g = torch.Generator().manual_seed(5)
        w = torch.randn(1, 32, 64, generator=g) * 0.02
        codes, scales = synth._quantise_weights(w, bits)
        c = codes[0].numpy()
        s = scales[0].view(torch.int16).numpy().view(np.uint16)
        dense = oracle.dequantize_matrix(c, s, bits, 32, 64)
        # each dequantised value is within half a step of the fp32 weight, except clipping at the top level
        s_rows = np.repeat(scales[0].float().numpy().T, 32, axis=1)  # [N, K]
        diff = np.abs(dense - w[0].double().numpy())
        top = (1 if bits == 2 else 3) * s_rows
        ok = (diff <= 0.5 * s_rows + 1e-12) | (w[0].double().numpy() > top)
        assert ok.all()


# ---------------------------------------------------------------- routing


def _route_inputs(L_rows):
    """Router inputs whose logits are exactly the given rows: x = e_0, Wr[:,0] = logits."""
    L_rows = np.asarray(L_rows, np.float32)
    T, E = L_rows.shape
    x = np.zeros((T, 32), np.float32)
    x[:, 0] = 1.0
    Wr = np.zeros((E, 32), np.float32)
    return x, Wr, L_rows


def test_topk_softmax_closed_forms():
    ln2, ln3 = math.log(2.0), math.log(3.0)
    L = np.array([[0.0, ln3, ln2, -5.0, -1.0, -7.0]])
    idx, w = oracle.topk_softmax(L, 3)
    assert idx.tolist() == [[1, 2, 0]]
    assert np.allclose(w, [[0.5, 1 / 3, 1 / 6]], rtol=0, atol=1e-7)
    idx, w = oracle.topk_softmax(np.array([[0.0, ln3, -9.0, -9.0]]), 2)
    assert idx.tolist() == [[1, 0]] and np.allclose(w, [[0.75, 0.25]], atol=1e-7)
    # exact ties go to the lower expert index and share the weight
    idx, w = oracle.topk_softmax(np.array([[0.5, 2.0, 2.0, 2.0, 0.5]]), 2)
    assert idx.tolist() == [[1, 2]] and w.tolist() == [[0.5, 0.5]]
    # one expert: weight exactly one
    idx, w = oracle.topk_softmax(np.array([[3.0]]), 1)
    assert idx.tolist() == [[0]] and w.tolist() == [[1.0]]


def test_router_logits_match_dense_matmul():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 96)).astype(np.float32)
    Wr = (rng.standard_normal((11, 96)) * 0.02).astype(np.float32)
    b = rng.standard_normal(11).astype(np.float32)
    L = oracle.router_logits(x, Wr, b)
    ref = x.astype(np.float64) @ Wr.astype(np.float64).T + b.astype(np.float64)
    assert np.allclose(L, ref, rtol=1e-13, atol=1e-13)


def test_topk_matches_stable_sort_and_full_softmax():
    rng = np.random.default_rng(4)
    L = rng.standard_normal((50, 24))
    L[:, 5] = L[:, 6]  # some exact ties
    for k in (1, 3, 24):
        idx, w = oracle.topk_softmax(L, k)
        for t in range(50):
            order = sorted(range(24), key=lambda e: (-L[t, e], e))[:k]
            assert idx[t].tolist() == order
        assert np.allclose(w.sum(1), 1.0, atol=1e-6)
        assert (np.diff(w, axis=1) <= 0).all()
    # k = E: the full softmax in descending order
    idx, w = oracle.topk_softmax(L, 24)
    full = softmax(L, axis=1)
    assert np.allclose(w, np.take_along_axis(full, idx, 1), rtol=0, atol=1e-7)


# ------------------------------------------------------------ permutation


def test_permute_matches_stable_sort():
    rng = np.random.default_rng(5)
    T, k, E = 37, 4, 9
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    P = oracle.permute(idx, E)
    flat = idx.reshape(-1)
    order = sorted(range(T * k), key=lambda p: (flat[p], p))
    assert P["perm_tok"].tolist() == [p // k for p in order]
    assert P["perm_slot"].tolist() == [p % k for p in order]
    assert np.array_equal(P["counts"], np.bincount(flat, minlength=E))
    assert np.array_equal(P["offsets"], np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    # inv is the inverse permutation
    pos = np.empty(T * k, np.int64)
    pos[np.array(order)] = np.arange(T * k)
    assert np.array_equal(P["inv"].reshape(-1), pos)
    # every token appears exactly k times
    assert np.array_equal(np.bincount(P["perm_tok"], minlength=T), np.full(T, k))


# ----------------------------------------------------- expert and layer


def _dense_expert(layer_np, e, I, H, bits):
    Wr, b, c, s = layer_np
    Wg = oracle.dequantize_matrix(c[0][e], s[0][e], bits, I, H)
    Wu = oracle.dequantize_matrix(c[1][e], s[1][e], bits, I, H)
    Wd = oracle.dequantize_matrix(c[2][e], s[2][e], bits, H, I)
    return Wg, Wu, Wd


def _dense_token_expert(xq_deq, Wg, Wu, Wd):
    G = Wg @ xq_deq
    U = Wu @ xq_deq
    h = (G * expit(G) * U).astype(np.float32)
    qh, sh = oracle.quantize_block32(h)
    hdeq = qh.astype(np.float64) * np.repeat(sh.astype(np.float64), 32)
    return G, U, h, Wd @ hdeq


@pytest.mark.parametrize("bits", [2, 3])
def test_expert_block_dots_equal_dense_fp64(bits):
    H, I = 64, 64
    shape = synth.LayerShape(H=H, I=I, E=3, k=2, bits=bits)
    lay = synth.make_layer(shape, seed=11)
    ln = lay.numpy()
    x = synth.make_x(4, H, seed=11).numpy()
    for e in range(3):
        Wg, Wu, Wd = _dense_expert(ln, e, I, H, bits)
        for t in range(4):
            qx, sx = oracle.quantize_block32(x[t])
            xdeq = qx.astype(np.float64) * np.repeat(sx.astype(np.float64), 32)
            out = oracle.expert_token(qx, sx, [ln[2][m][e] for m in range(3)], [ln[3][m][e] for m in range(3)], bits, H, I)
            G, U, h, D = _dense_token_expert(xdeq, Wg, Wu, Wd)
            assert np.allclose(out["G"], G, rtol=1e-12, atol=1e-14)
            assert np.allclose(out["U"], U, rtol=1e-12, atol=1e-14)
            # h agrees to the fp32 rounding of two fp64 evaluations of the same value
            assert np.allclose(out["h"], h, rtol=2e-7, atol=1e-30)
            if np.array_equal(out["h"], h):
                assert np.allclose(out["D"], D, rtol=1e-12, atol=1e-14)


def _numpy_layer(x, ln, k, bits, residual):
    """An independent dense implementation of the whole layer (brute force)."""
    Wr, b, c, s = ln
    T, H = x.shape
    E = Wr.shape[0]
    I = c[0].shape[2]
    L = x.astype(np.float64) @ Wr.astype(np.float64).T + (0 if b is None else b.astype(np.float64))
    dense = [_dense_expert(ln, e, I, H, bits) for e in range(E)]
    y = np.zeros((T, H))
    idx_all, w_all = [], []
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-L[t, e], e))[:k]
        w = softmax(L[t, order]).astype(np.float32)
        qx, sx = oracle.quantize_block32(x[t])
        xdeq = qx.astype(np.float64) * np.repeat(sx.astype(np.float64), 32)
        for j, e in enumerate(order):
            y[t] += float(w[j]) * _dense_token_expert(xdeq, *dense[e])[3]
        if residual:
            y[t] += x[t]
        idx_all.append(order)
        w_all.append(w)
    return np.array(idx_all), np.array(w_all), y.astype(np.float32)


@pytest.mark.parametrize("residual", [False, True])
def test_layer_matches_dense_bruteforce(residual):
    shape = synth.LayerShape(H=64, I=64, E=6, k=2)
    lay = synth.make_layer(shape, seed=3)
    ln = lay.numpy()
    x = synth.make_x(6, 64, seed=3).numpy() * 3
    out = oracle.layer(x, ln[0], ln[1], ln[2], ln[3], 2, 2, residual=residual)
    idx, w, y = _numpy_layer(x, ln, 2, 2, residual)
    assert np.array_equal(out["idx"], idx)
    assert np.allclose(out["w"], w, atol=1e-7)
    rms = np.sqrt(np.mean(y.astype(np.float64) ** 2))
    assert np.abs(out["y"] - y).max() <= 1e-6 * rms


def test_layer_zero_input_and_one_expert():
    shape = synth.LayerShape(H=64, I=32, E=5, k=3)
    ln = synth.make_layer(shape, seed=7).numpy()
    x = np.zeros((3, 64), np.float32)
    out = oracle.layer(x, ln[0], None, ln[2], ln[3], 2, 3)
    # all logits tie at zero: the lowest k experts, equal weights, and silu(0)*0 = 0
    assert out["idx"].tolist() == [[0, 1, 2]] * 3
    assert np.allclose(out["w"], 1 / 3, atol=1e-7)
    assert not out["y"].any()
    # k = 1: weight exactly one and y is that expert's down projection
    x = synth.make_x(2, 64, seed=7).numpy()
    out = oracle.layer(x, ln[0], None, ln[2], ln[3], 2, 1, detail=True)
    assert (out["w"] == 1.0).all()
    assert np.array_equal(out["y"], out["D"][:, 0, :].astype(np.float32))


def test_layer_single_expert_is_a_dense_expert():
    # E = 1, k = 1 (the form a shared expert takes): every token goes to expert 0
    # with weight exactly 1, and y is that expert's down projection, which equals
    # the dense fp64 SwiGLU of the dequantised matrices up to the int8 rounding of h
    shape = synth.LayerShape(H=64, I=32, E=1, k=1)
    ln = synth.make_layer(shape, seed=9).numpy()
    x = synth.make_x(4, 64, seed=9).numpy()
    out = oracle.layer(x, ln[0], None, ln[2], ln[3], 2, 1, detail=True)
    assert (out["idx"] == 0).all() and (out["w"] == 1.0).all()
    assert np.array_equal(out["y"], out["D"][:, 0, :].astype(np.float32))
    Wg, Wu, Wd = (oracle.dequantize_matrix(ln[2][m][0], ln[3][m][0], 2, *dims)
                  for m, dims in enumerate(((32, 64), (32, 64), (64, 32))))
    q, s = oracle.quantize_block32(x)
    xq = q.astype(np.float64) * np.repeat(s.astype(np.float64), 32, axis=1)
    G, U = xq @ Wg.T, xq @ Wu.T
    h = G * expit(G) * U
    dense = h @ Wd.T
    assert np.abs(out["y"] - dense).max() <= 0.02 * np.abs(dense).max()


def test_layer_k_equals_E_is_dense_mixture():
    shape = synth.LayerShape(H=64, I=32, E=4, k=4)
    ln = synth.make_layer(shape, seed=9).numpy()
    x = synth.make_x(3, 64, seed=9).numpy()
    out = oracle.layer(x, ln[0], None, ln[2], ln[3], 2, 4, detail=True)
    L = x.astype(np.float64) @ ln[0].astype(np.float64).T
    p = softmax(L, axis=1)
    for t in range(3):
        # every expert is used, with its full-softmax probability
        assert sorted(out["idx"][t].tolist()) == [0, 1, 2, 3]
        assert np.allclose(out["w"][t], p[t, out["idx"][t]], atol=1e-7)
    y = np.einsum("tj,tjh->th", out["w"].astype(np.float64), out["D"])
    assert np.allclose(out["y"], y, rtol=1e-6, atol=1e-9)


def test_layer_token_subset_is_exact():
    shape = synth.LayerShape(H=64, I=32, E=8, k=2)
    ln = synth.make_layer(shape, seed=13).numpy()
    x = synth.make_x(10, 64, seed=13).numpy()
    full = oracle.layer(x, ln[0], ln[1], ln[2], ln[3], 2, 2, nthreads=3)
    sub = oracle.layer(x, ln[0], ln[1], ln[2], ln[3], 2, 2, tokens=[7, 2, 9], nthreads=2)
    assert np.array_equal(sub["y"], full["y"][[7, 2, 9]])
    assert np.array_equal(sub["idx"], full["idx"][[7, 2, 9]])


def test_hdist_measures_distance_to_rounding_boundary():
    shape = synth.LayerShape(H=64, I=64, E=2, k=1)
    ln = synth.make_layer(shape, seed=17).numpy()
    x = synth.make_x(3, 64, seed=17).numpy()
    out = oracle.layer(x, ln[0], None, ln[2], ln[3], 2, 1, detail=True)
    for t in range(3):
        e = out["idx"][t, 0]
        qx, sx = oracle.quantize_block32(x[t])
        d = oracle.expert_token(qx, sx, [ln[2][m][e] for m in range(3)], [ln[3][m][e] for m in range(3)], 2, 64, 64)
        r = d["h"].astype(np.float64) / np.repeat(d["sh"].astype(np.float64), 32)
        # |r - q| = 0.5 - hdist for every element: the code is the nearest integer
        assert np.allclose(np.abs(r - d["qh"]), 0.5 - d["hdist"], atol=1e-9)
        assert np.array_equal(out["qh"][t, 0], d["qh"])
