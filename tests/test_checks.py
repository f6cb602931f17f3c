"""Pins for the test-side parity helpers in oracle/checks.py and for
oracle.weight_column, which they use.

compare_layer_output decides which over-tolerance rows of a device output are
still correct: only rows explained by moving int8 SwiGLU codes that the oracle
reports as near-ties to their other neighbour.  These tests plant such a flip,
and mistakes of similar size that are not one, in the oracle's own output on
the CPU and check that the helper accepts the first and rejects the others.
The expected effect of a flip is built from an independent numpy unpacking of
the weight layout (not from the oracle's accessors).
"""
import numpy as np
import pytest

import oracle
import synth
from oracle.checks import compare_layer_output


def _unpack_levels(codes_e, bits, N, K):
    """Signed levels [N, K] of one expert matrix, from the storage layout:
    codes [K/32][N][4*bits]; 2-bit element i of a block is byte i/4, bits
    2(i%4), level = code - 2; 3-bit element i is bits 3i..3i+2 of the block's
    96-bit little-endian word, level = code - 4."""
    KB = K // 32
    c = np.asarray(codes_e, np.uint8).reshape(KB, N, 4 * bits)
    bitsarr = np.unpackbits(c, axis=-1, bitorder="little").reshape(KB, N, 32, bits)
    weights = (1 << np.arange(bits)).astype(np.int64)
    code = (bitsarr.astype(np.int64) * weights).sum(-1)  # [KB, N, 32]
    lv = code - (1 << (bits - 1))
    return lv.transpose(1, 0, 2).reshape(N, K)


def _dense(codes_e, scales_e, bits, N, K):
    lv = _unpack_levels(codes_e, bits, N, K).astype(np.float64)
    sc = np.asarray(scales_e, np.uint16).reshape(K // 32, N).view(np.float16).astype(np.float64)
    return lv * np.repeat(sc.T, 32, axis=1)


@pytest.mark.parametrize("bits", [2, 3])
def test_unpacker_matches_golden_three_bit_and_generator(bits):
    # the test's own unpacker against a hand-built block (codes c_i = (3i + 1) % 2^bits)
    N, K = 2, 64
    nlev = 1 << bits
    blocks = []
    want = np.zeros((N, K), np.int64)
    for kb in range(K // 32):
        for n in range(N):
            word = 0
            for i in range(32):
                c = (3 * i + 1 + n + kb) % nlev
                word |= c << (bits * i)
                want[n, 32 * kb + i] = c - nlev // 2
            blocks.append(word.to_bytes(4 * bits, "little"))
    codes = np.frombuffer(b"".join(blocks), np.uint8)
    assert np.array_equal(_unpack_levels(codes, bits, N, K), want)


@pytest.mark.parametrize("bits", [2, 3])
def test_weight_column_matches_independent_unpack(bits):
    shape = synth.LayerShape(H=256, I=128, E=3, k=2, bits=bits)
    _, _, c, s = synth.make_layer(shape, seed=21).numpy()
    for e in range(3):
        dense = _dense(c[2][e], s[2][e], bits, shape.H, shape.I)  # down: [H, I]
        for kk in (0, 1, 31, 32, 77, shape.I - 1):
            col = oracle.weight_column(c[2][e], s[2][e], bits, shape.H, kk)
            assert np.array_equal(col, dense[:, kk])
        # and the whole matrix through the oracle's element accessor
        if e == 0:
            assert np.array_equal(oracle.dequantize_matrix(c[2][e], s[2][e], bits, shape.H, shape.I), dense)


@pytest.fixture(scope="module")
def tiny_ref():
    shape = synth.TINY
    lay = synth.make_layer(shape, seed=0)
    ln = lay.numpy()
    x = synth.make_x(64, shape.H, seed=1).numpy()
    ref = oracle.layer(x, *ln, shape.bits, shape.k, detail=True)
    return shape, ln, ref


def _flip_effect(shape, ln, ref, t, j, i):
    """Change of y[t] when SwiGLU code i of pair (t, j) moves to its other neighbour."""
    e = int(ref["idx"][t, j])
    s = float(ref["sh"][t, j, i // 32])
    r = float(ref["h"][t, j, i]) / s
    q = int(ref["qh"][t, j, i])
    alt = q + (1 if r > q else -1)
    dense = _dense(ln[2][2][e], ln[3][2][e], shape.bits, shape.H, shape.I)
    return float(ref["w"][t, j]) * (alt - q) * s * dense[:, i]


def _rms(ref):
    return float(np.sqrt(np.mean(ref["y"].astype(np.float64) ** 2)))


def test_exact_output_passes(tiny_ref):
    shape, ln, ref = tiny_ref
    err, rows, n_alt = compare_layer_output(ref["y"].copy(), ref, ln[2][2], ln[3][2], shape.bits)
    assert err == 0.0 and rows == 0 and n_alt == 0


def _pick(ref, near: bool):
    hd = ref["hdist"]
    cand = np.argwhere(hd < 5e-4) if near else np.argwhere(hd > 0.45)
    assert len(cand) > 0
    # the candidate with the largest routing weight, so the flip is well above the bound
    wts = np.array([ref["w"][t, j] for t, j, _ in cand])
    return tuple(int(v) for v in cand[int(np.argmax(wts))])


def test_near_tie_flip_is_accepted(tiny_ref):
    shape, ln, ref = tiny_ref
    t, j, i = _pick(ref, near=True)
    d = _flip_effect(shape, ln, ref, t, j, i)
    rms = _rms(ref)
    tol = 0.25 * np.abs(d).max() / rms  # the flip alone is four times the bound
    y = ref["y"].astype(np.float64).copy()
    y[t] += d
    err, rows, n_alt = compare_layer_output(y.astype(np.float32), ref, ln[2][2], ln[3][2], shape.bits, tol=tol,
                                            delta=1e-3)
    assert rows == 1 and n_alt == 1 and err <= tol


def test_flip_far_from_a_boundary_is_rejected(tiny_ref):
    shape, ln, ref = tiny_ref
    t, j, i = _pick(ref, near=False)
    d = _flip_effect(shape, ln, ref, t, j, i)
    tol = 0.25 * np.abs(d).max() / _rms(ref)
    y = ref["y"].astype(np.float64).copy()
    y[t] += d
    with pytest.raises(AssertionError):
        compare_layer_output(y.astype(np.float32), ref, ln[2][2], ln[3][2], shape.bits, tol=tol, delta=1e-3)


def test_near_tie_flip_plus_far_flip_is_rejected(tiny_ref):
    shape, ln, ref = tiny_ref
    tn, jn, i_n = _pick(ref, near=True)
    d_near = _flip_effect(shape, ln, ref, tn, jn, i_n)
    far = [tuple(int(v) for v in c) for c in np.argwhere(ref["hdist"][tn] > 0.45)]
    _, jf, i_f = max(((tn, j, i) for j, i in far), key=lambda c: ref["w"][tn, c[1]])
    d_far = _flip_effect(shape, ln, ref, tn, jf, i_f)
    tol = 0.25 * min(np.abs(d_near).max(), np.abs(d_far).max()) / _rms(ref)
    y = ref["y"].astype(np.float64).copy()
    y[tn] += d_near + d_far
    with pytest.raises(AssertionError):
        compare_layer_output(y.astype(np.float32), ref, ln[2][2], ln[3][2], shape.bits, tol=tol, delta=1e-3)


def test_random_perturbation_is_rejected(tiny_ref):
    shape, ln, ref = tiny_ref
    rms = _rms(ref)
    rng = np.random.default_rng(9)
    for _ in range(5):
        y = ref["y"].astype(np.float64).copy()
        t, n = int(rng.integers(64)), int(rng.integers(shape.H))
        y[t, n] += 3e-3 * rms * (1 if rng.random() < 0.5 else -1)
        with pytest.raises(AssertionError):
            compare_layer_output(y.astype(np.float32), ref, ln[2][2], ln[3][2], shape.bits, tol=2e-3)
