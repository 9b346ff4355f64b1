"""Pins for the oracle's weight formats: the uint4 group quantiser, the packed
layout, the INT8 per-channel quantiser and the linear layers built on them.

The quantisers are pinned by their error bounds, by round trips of inputs
that lie exactly on a quantisation grid, by brute force over all levels and by
numpy's independent fp16 rounding; the linears by numpy's matmul of the
dequantised matrix and by one-hot probes."""
import numpy as np
import pytest

import oracle
from quantized_speculative_decoding_gb300 import synth


def _f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _pack_words(q):
    """Pack q[N][K] (0..15) by the layout's definition: nibble j of word c
    holds k = 8c + j."""
    N, K = q.shape
    q = q.astype(np.uint32).reshape(N, K // 8, 8)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    return np.bitwise_or.reduce(q << shifts, axis=2).astype(np.uint32)


@pytest.mark.parametrize("N,K", [(7, 256), (33, 512), (3, 1024)])
def test_w4_error_bound_and_ranges(N, K):
    rng = np.random.default_rng(N * K)
    w = (rng.standard_normal((N, K)) * rng.choice([1e-3, 0.02, 1.0, 50.0], (N, 1))).astype(np.float32)
    w[0, :128] = 0.0                         # an all-zero group
    w[1, 128:256] = np.abs(w[1, 128:256])    # a one-signed group
    q, s, z = oracle.quantize_w4(w, 128)
    sf, zf = _f16(s), _f16(z)
    assert q.max() <= 15
    assert np.all(zf == np.round(zf)) and zf.min() >= 0 and zf.max() <= 15
    wq = oracle.dequant_w4(q, s, z, 128)
    srep = np.repeat(sf, 128, axis=1)
    err = np.abs(w.astype(np.float64) - wq)
    assert np.all(err <= srep / 2 * (1 + 1e-12))
    assert np.all(wq[0, :128] == 0.0)
    # numpy's fp16 rounding of the exact range / 15, stepped up only if needed
    wg = w.astype(np.float64).reshape(N, K // 128, 128)
    rng_ = np.maximum(wg.max(-1), 0) - np.minimum(wg.min(-1), 0)
    rn = (rng_ / 15).astype(np.float16).astype(np.float64)
    step = (rng_ / 15).astype(np.float16)
    step = np.nextafter(step, np.float16(np.inf)).astype(np.float64)
    expect = np.where(rng_ == 0, 1.0, np.where(15 * rn >= rng_, rn, step))
    assert np.array_equal(sf, expect)


def test_w4_brute_force_levels():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((16, 128)) * 0.02).astype(np.float32)
    q, s, z = oracle.quantize_w4(w, 128)
    sf, zf = _f16(s)[:, 0], _f16(z)[:, 0]
    for n in range(16):
        levels = (np.arange(16) - zf[n]) * sf[n]
        for k in range(128):
            d = np.abs(w[n, k] - levels)
            best = np.flatnonzero(d == d.min())
            # ties (exact halves) are allowed either way; the chosen level is
            # a nearest one
            assert q[n, k] in best


def test_w4_round_trip_of_grid_values():
    # weights that lie exactly on an fp16 grid with levels 0 and 15 present
    rng = np.random.default_rng(10)
    N, K = 24, 512
    s = rng.uniform(1e-3, 2e-2, (N, K // 128)).astype(np.float16)
    z = rng.integers(0, 16, (N, K // 128))
    q = rng.integers(0, 16, (N, K))
    q[:, ::128] = 0
    q[:, 1::128] = 15
    w = ((q.reshape(N, K // 128, 128) - z[..., None]) * s.astype(np.float64)[..., None])
    w = w.reshape(N, K).astype(np.float32)
    q2, s2, z2 = oracle.quantize_w4(w, 128)
    assert np.array_equal(q2, q)
    assert np.array_equal(_f16(s2), s.astype(np.float64))
    assert np.array_equal(_f16(z2), z.astype(np.float64))


def test_unpack_is_the_layout_definition():
    rng = np.random.default_rng(11)
    q = rng.integers(0, 16, (5, 64)).astype(np.uint8)
    assert np.array_equal(oracle.unpack_w4(_pack_words(q), 5, 64), q)
    # every level at every nibble position
    for j in range(8):
        for v in range(16):
            qq = np.zeros((1, 8), np.uint8)
            qq[0, j] = v
            word = np.array([[v << (4 * j)]], np.uint32)
            assert np.array_equal(oracle.unpack_w4(word, 1, 8), qq)


def test_w8_error_bound_and_brute_force():
    rng = np.random.default_rng(12)
    w = (rng.standard_normal((20, 300)) * 0.02).astype(np.float32)
    w[3] = 0.0
    q8, s = oracle.quantize_w8(w)
    sf = _f16(s)
    assert q8.min() >= -127 and q8.max() <= 127
    wq = q8.astype(np.float64) * sf[:, None]
    assert np.all(np.abs(w - wq) <= sf[:, None] / 2 * (1 + 1e-12))
    amax = np.abs(w.astype(np.float64)).max(1)
    assert np.all(127 * sf >= amax)
    assert sf[3] == 1.0 and np.all(q8[3] == 0)
    levels = np.arange(-127, 128)
    for n in range(0, 20, 5):
        for k in range(0, 300, 17):
            d = np.abs(w[n, k] - levels * sf[n])
            assert q8[n, k] in levels[d == d.min()]


def test_quantisers_reject_non_finite():
    w = np.zeros((2, 128), np.float32)
    w[1, 5] = np.nan
    with pytest.raises(ValueError):
        oracle.quantize_w4(w, 128)
    with pytest.raises(ValueError):
        oracle.quantize_w8(w)


@pytest.mark.parametrize("M,N,K", [(5, 40, 512), (1, 17, 256), (8, 9, 384)])
def test_w4a16_linear_matches_numpy_matmul(M, N, K):
    w = synth.weights(N, K, seed=M + N + K)
    q, s, z = oracle.quantize_w4(w, 128)
    qw = _pack_words(q)
    x = synth.activations(M, K, seed=3)
    y = oracle.w4a16_linear(x, qw, s, z, 128, N, K)
    xf = oracle.bf16_to_f64(x)
    wf = (q.astype(np.float64) - np.repeat(_f16(z), 128, 1)) * np.repeat(_f16(s), 128, 1)
    ref = xf @ wf.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_w4a16_one_hot_probes_are_exact():
    N, K = 12, 256
    w = synth.weights(N, K, seed=4)
    q, s, z = oracle.quantize_w4(w, 128)
    qw = _pack_words(q)
    wq = oracle.dequant_w4(q, s, z, 128)
    ks = [0, 1, 7, 8, 127, 128, 200, 255]
    x = np.zeros((len(ks), K), np.float32)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    y = oracle.w4a16_linear(synth.to_bf16_bits(x), qw, s, z, 128, N, K)
    for m, k in enumerate(ks):
        assert np.array_equal(y[m], wq[:, k])


def test_w8_and_bf16_linears_match_numpy():
    M, N, K = 3, 21, 160
    w = synth.weights(N, K, seed=5)
    x = synth.activations(M, K, seed=6)
    xf = oracle.bf16_to_f64(x)
    q8, s = oracle.quantize_w8(w)
    y8 = oracle.w8a16_linear(x, q8, s)
    ref8 = xf @ (q8.astype(np.float64) * _f16(s)[:, None]).T
    assert np.allclose(y8, ref8, rtol=1e-12, atol=1e-14)
    wb = synth.to_bf16_bits(w)
    yb = oracle.bf16_linear(x, wb)
    refb = xf @ oracle.bf16_to_f64(wb).T
    assert np.allclose(yb, refb, rtol=1e-12, atol=1e-14)
