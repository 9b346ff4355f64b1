"""Pins for the oracle's fp16 / bf16 rounding (IEEE binary16 and bfloat16,
round to nearest even).  Checked against numpy's and torch's own conversions
and against brute-force nearest-value search over every finite code."""
import numpy as np
import pytest
import torch

import oracle


def _f16_of(x):
    return int(np.float64(x).astype(np.float16).view(np.uint16))


def test_f16_decode_all_codes_matches_numpy():
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = oracle.f16_to_f64(codes)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_bf16_decode_all_codes_matches_torch():
    codes = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_to_f64(codes)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 6, 4000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e9, 2.0 ** -24,
                  2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12), 1 / 3]),
    ])
    # exact ties between neighbouring fp16 values: (a + b) / 2
    codes = rng.integers(0, 0x7bff, 2000).astype(np.uint16)
    a = codes.view(np.float16).astype(np.float64)
    b = (codes + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    xs = np.concatenate([xs, (a + b) / 2, -(a + b) / 2])
    for x in xs:
        assert oracle.f64_to_f16_bits(x) == _f16_of(x), x


def test_bf16_rounding_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(2)
    xs = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f64_to_bf16_bits(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_is_nearest_even_by_brute_force():
    # every finite non-negative bf16 value, in increasing order
    codes = np.arange(0x7f80, dtype=np.uint16)
    vals = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    rng = np.random.default_rng(3)
    xs = np.abs(rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000))
    mid = (vals[100:3000:7] + vals[101:3001:7]) / 2  # exact ties
    for x in np.concatenate([xs, mid]):
        i = np.searchsorted(vals, x)
        cands = [c for c in (i - 1, i) if 0 <= c < len(vals)]
        d = [abs(vals[c] - x) for c in cands]
        best = [c for c, dd in zip(cands, d) if dd == min(d)]
        if len(best) > 1:
            best = [c for c in best if c % 2 == 0]
        assert oracle.f64_to_bf16_bits(x) == int(codes[best[0]]), x
        assert oracle.f64_to_bf16_bits(-x) == int(codes[best[0]]) | 0x8000


@pytest.mark.parametrize("x", [np.inf, -np.inf])
def test_infinities(x):
    assert oracle.f16_bits_to_f64(oracle.f64_to_f16_bits(x)) == x
    assert oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(x)) == x
