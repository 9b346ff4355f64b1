"""Pins for the oracle's low-bit formats: b-bit weights (INT3 / INT2 targets,
"Speculative Decoding in Quantized Regimes" sec. 4.1-4.2) and the W4A4
draft's activations (QSPEC, reference [1] of "When Do Quantized Drafts Help
Speculative Decoding?").

What the mathematics fixes, independently of the oracle's formulas:
  * the scale is the smallest fp16 s with L s >= the group's range (L = 2^b - 1);
  * every code is a nearest level: no other level of the group lies closer;
  * so every weight is within s/2 of its dequantised value;
  * b = 4 reproduces the pinned INT4 quantiser and nibble layout exactly;
  * the packed words are the row's bit stream, rebuilt with Python integers;
  * the linears equal numpy's matmul of the dequantised operands;
  * W4A4 differs from W4A16 by at most sum_g (s_x,g / 2) sum_k |w'_k| per output.
"""
import numpy as np
import pytest

import oracle
from quantized_speculative_decoding_gb300 import synth


def _f16(bits):
    return oracle.f16_to_f64(bits)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_scale_is_the_smallest_sufficient_fp16(bits):
    L = (1 << bits) - 1
    w = synth.weights(16, 512, 40 + bits)
    q, s, z = oracle.quantize_wb(w, bits)
    sv = _f16(s)
    g = w.reshape(16, 4, 128).astype(np.float64)
    rng = np.maximum(g.max(-1), 0) - np.minimum(g.min(-1), 0)
    assert np.all(L * sv >= rng)
    prev = _f16(s.astype(np.int64) - 1)  # the fp16 just below (positive values)
    assert np.all(L * prev < rng)
    zv = _f16(z)
    assert np.all((zv == np.round(zv)) & (zv >= 0) & (zv <= L))


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codes_are_nearest_levels_and_error_is_half_a_step(bits):
    L = (1 << bits) - 1
    w = synth.weights(8, 256, 50 + bits)
    q, s, z = oracle.quantize_wb(w, bits)
    sv = np.repeat(_f16(s), 128, axis=1)
    zv = np.repeat(_f16(z), 128, axis=1)
    wd = w.astype(np.float64)
    levels = (np.arange(L + 1)[None, None, :] - zv[..., None]) * sv[..., None]
    dist = np.abs(wd[..., None] - levels)
    chosen = np.take_along_axis(dist, q[..., None].astype(np.int64), axis=-1)[..., 0]
    assert np.all(chosen <= dist.min(-1) + 1e-15)
    assert np.all(np.abs(wd - (q - zv) * sv) <= sv / 2 + 1e-15)


def test_four_bits_is_the_int4_quantiser_and_layout():
    w = synth.weights(12, 384, 7)
    q4, s4, z4 = oracle.quantize_w4(w)
    q, s, z = oracle.quantize_wb(w, 4)
    assert np.array_equal(q, q4) and np.array_equal(s, s4) and np.array_equal(z, z4)
    assert np.array_equal(oracle.unpack_w4(oracle.pack_wb(q, 4), 12, 384), q)


def test_zero_group():
    q, s, z = oracle.quantize_wb(np.zeros((2, 128), np.float32), 3)
    assert np.all(q == 0) and np.all(_f16(s) == 1.0) and np.all(_f16(z) == 0.0)


@pytest.mark.parametrize("bits,K", [(2, 16), (2, 256), (3, 32), (3, 384), (4, 8), (4, 128)])
def test_packed_words_are_the_bit_stream(bits, K):
    rng = np.random.default_rng(bits * K)
    N = 5
    q = rng.integers(0, 1 << bits, (N, K)).astype(np.uint8)
    q[0] = np.arange(K) % (1 << bits)           # every level at every position class
    q[1] = (1 << bits) - 1                      # all ones
    packed = oracle.pack_wb(q, bits)
    assert packed.shape == (N, K * bits // 32)
    for n in range(N):
        stream = sum(int(v) << (bits * k) for k, v in enumerate(q[n]))
        words = sum(int(c) << (32 * i) for i, c in enumerate(packed[n]))
        assert words == stream
    assert np.array_equal(oracle.unpack_wb(packed, N, K, bits), q)


def test_pack_rejects_a_partial_word():
    with pytest.raises(ValueError):
        oracle.pack_wb(np.zeros((1, 40), np.uint8), 3)


@pytest.mark.parametrize("bits", [2, 3])
def test_wb_linear_is_the_dequantised_matmul(bits):
    N, K, M = 24, 384, 3
    w = synth.weights(N, K, 60 + bits)
    q, s, z = oracle.quantize_wb(w, bits)
    packed = oracle.pack_wb(q, bits)
    x = synth.activations(M, K, seed=61)
    wd = (q - np.repeat(_f16(z), 128, axis=1)) * np.repeat(_f16(s), 128, axis=1)
    ref = oracle.bf16_to_f64(x) @ wd.T
    y = oracle.wb_linear(x, packed, s, z, 128, bits, N, K)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # one-hot probes return a dequantised weight exactly
    ks = [0, 127, 128, 383]
    xo = np.zeros((len(ks), K), np.float32)
    for m, k in enumerate(ks):
        xo[m, k] = 1.0
    yo = oracle.wb_linear(synth.to_bf16_bits(xo), packed, s, z, 128, bits, N, K)
    assert np.array_equal(yo, wd[:, ks].T)


def test_activation_codes():
    x = synth.activations(6, 512, seed=70)
    x[2, 128:256] = 0                                        # an all-zero group
    qx, sx = oracle.quantize_a4(x)
    xf = oracle.bf16_to_f64(x).astype(np.float32)            # exact
    amax = np.abs(xf.reshape(6, 4, 128)).max(-1)
    expect = np.where(amax > 0, amax / np.float32(7), np.float32(1))  # numpy's fp32 division
    assert np.array_equal(sx, expect)
    ratio = xf / np.repeat(sx, 128, axis=1)                  # fp32 quotients, as the codes are decided
    assert np.all(np.abs(ratio.astype(np.float64) - qx) <= 0.5)
    assert np.all((qx >= -7) & (qx <= 7))                    # |x| <= 7 s: -8 is never needed
    assert np.all(qx[2, 128:256] == 0) and sx[2, 1] == 1.0
    err = np.abs(xf.astype(np.float64) - qx * np.repeat(sx, 128, axis=1).astype(np.float64))
    assert np.all(err <= np.repeat(sx, 128, axis=1) / 2 * (1 + 2 ** -20))


def test_w4a4_linear():
    N, K, M = 20, 512, 4
    w = synth.weights(N, K, 80)
    q, s, z = oracle.quantize_w4(w)
    packed = oracle.pack_wb(q, 4)
    x = synth.activations(M, K, seed=81)
    qx, sx = oracle.quantize_a4(x)
    xd = qx * np.repeat(sx.astype(np.float64), 128, axis=1)
    wd = (q - np.repeat(_f16(z), 128, axis=1)) * np.repeat(_f16(s), 128, axis=1)
    y = oracle.w4a4_linear(x, packed, s, z, N, K)
    assert np.allclose(y, xd @ wd.T, rtol=1e-12, atol=1e-12 * np.abs(y).max())
    # against the A16 path: the activation rounding error bounds the difference
    y16 = oracle.w4a16_linear(x, packed, s, z, 128, N, K)
    bound = (np.repeat(sx.astype(np.float64) / 2, 128, axis=1) @ np.abs(wd).T) * (1 + 1e-6)
    assert np.all(np.abs(y - y16) <= bound)


# ------------------------------------------------------------ planted mistakes
def _mutant(tmp_path, pattern, repl):
    import ctypes
    import os
    import re
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    new, n = re.subn(pattern, repl, src)
    assert n >= 1, pattern
    c, so = tmp_path / "mut.c", tmp_path / "mut.so"
    c.write_text(new)
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-shared", "-fPIC", "-o", str(so), str(c), "-lm"])
    lib = ctypes.CDLL(str(so))
    good = oracle._load()
    for name in ("oracle_quantize_wb", "oracle_pack_wb", "oracle_quantize_a4"):
        getattr(lib, name).argtypes = getattr(good, name).argtypes
        getattr(lib, name).restype = getattr(good, name).restype
    return lib


@pytest.mark.parametrize("pattern,repl,what", [
    (r"const double L = \(double\)\(\(1 << bits\) - 1\);", "const double L = (double)(1 << bits);", "levels"),
    (r"long bit = \(long\)k \* bits \+ t;\n                uint32_t v", "long bit = (long)k * bits + (bits - 1 - t);\n                uint32_t v", "bit order"),
    (r"float s = amax > 0\.0f \? amax / 7\.0f : 1\.0f;", "float s = amax > 0.0f ? amax / 8.0f : 1.0f;", "act scale"),
])
def test_planted_mistakes_fail_the_pins(tmp_path, pattern, repl, what):
    lib = _mutant(tmp_path, pattern, repl)
    if what == "levels":
        bits, L = 3, 7
        w = synth.weights(4, 256, 90)
        q = np.zeros((4, 256), np.uint8)
        s = np.zeros((4, 2), np.uint16)
        z = np.zeros((4, 2), np.uint16)
        lib.oracle_quantize_wb(w, 4, 256, 128, bits, q, s, z)
        g = w.reshape(4, 2, 128).astype(np.float64)
        rng = np.maximum(g.max(-1), 0) - np.minimum(g.min(-1), 0)
        assert not (np.all(L * _f16(s) >= rng) and np.all(q <= L))
    elif what == "bit order":
        q = (np.arange(32) % 8).astype(np.uint8)[None]
        out = np.zeros((1, 3), np.uint32)
        lib.oracle_pack_wb(q, 1, 32, 3, out)
        stream = sum(int(v) << (3 * k) for k, v in enumerate(q[0]))
        assert sum(int(c) << (32 * i) for i, c in enumerate(out[0])) != stream
    else:
        x = synth.activations(1, 128, seed=91)
        qx = np.zeros((1, 128), np.int8)
        sx = np.zeros((1, 1), np.float32)
        lib.oracle_quantize_a4(x, 1, 128, qx, sx)
        xf = oracle.bf16_to_f64(x).astype(np.float32)
        assert sx[0, 0] != np.abs(xf).max() / np.float32(7)
