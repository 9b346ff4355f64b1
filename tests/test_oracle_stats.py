"""Pins for the oracle's softmax-row statistics (m, Z, argmax).

The speculative-sampling rule (references [2] Leviathan et al. and [3] Chen et
al. of "When Do Quantized Drafts Help Speculative Decoding?") needs p_v =
softmax(l / T)_v.  It is normalised by m = max l and Z = sum exp((l - m) / T),
and a consumer of chunked statistics merges slices by m = max m_i,
Z = sum Z_i exp((m_i - m) / T).  These follow from the mathematics:
  * a constant row gives m = c and Z = V exactly;
  * log Z + m / T is scipy's logsumexp of l / T (a library routine);
  * the merge law holds for any split of a row into slices;
  * the argmax takes the lowest index among equal maxima (brute force);
  * exp((l - m) / T) / Z sums to 1 and matches the closed form of two
    entries, p_0 = 1 / (1 + exp((l_1 - l_0) / T)).
Planted mistakes, each compiled from oracle.c on the CPU, must fail one pin.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest
from scipy import special

import oracle

ORACLE_C = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def test_constant_row():
    for V in (1, 7, 1024):
        m, z, a = oracle.softmax_stats(np.full(V, 2.5, np.float32), 0.7)
        assert m == 2.5 and z == float(V) and a == 0


def test_logsumexp_identity():
    rng = np.random.default_rng(3)
    for T in (0.3, 1.0, 2.5):
        for V in (2, 100, 5000):
            l = (rng.standard_normal(V) * 3).astype(np.float32)
            m, z, _ = oracle.softmax_stats(l, T)
            ref = special.logsumexp(l.astype(np.float64) / T)
            assert np.log(z) + m / T == pytest.approx(ref, rel=1e-13, abs=1e-13)


def test_two_entry_closed_form():
    for l0, l1, T in ((0.0, 1.0, 1.0), (3.0, -2.0, 0.5), (1.25, 1.25, 2.0)):
        l = np.array([l0, l1], np.float32)
        m, z, _ = oracle.softmax_stats(l, T)
        p0 = np.exp((np.float64(l0) - m) / T) / z
        assert p0 == pytest.approx(1.0 / (1.0 + np.exp((np.float64(l1) - np.float64(l0)) / T)), rel=1e-14)


@pytest.mark.parametrize("T", [0.8, 1.0])
def test_merge_of_slices(T):
    rng = np.random.default_rng(11)
    V = 3001
    l = (rng.standard_normal(V) * 3).astype(np.float32)
    m, z, a = oracle.softmax_stats(l, T)
    for cuts in ([1000, 2000], [1, 2, 3, 2999], list(range(128, V, 128))):
        edges = [0] + cuts + [V]
        parts = [oracle.softmax_stats(l[e0:e1], T) for e0, e1 in zip(edges[:-1], edges[1:])]
        mm = max(p[0] for p in parts)
        zz = sum(p[1] * np.exp((p[0] - mm) / T) for p in parts)
        assert mm == m
        assert zz == pytest.approx(z, rel=1e-13)
        # argmax: the best slice maximum, lowest global index on ties
        best = max(range(len(parts)), key=lambda i: (parts[i][0], -(edges[i] + parts[i][2])))
        assert edges[best] + parts[best][2] == a
    p = np.exp((l.astype(np.float64) - m) / T) / z
    assert p.sum() == pytest.approx(1.0, rel=1e-13)


def test_argmax_ties_take_the_lowest_index():
    rng = np.random.default_rng(5)
    for _ in range(50):
        V = int(rng.integers(1, 40))
        l = rng.integers(-3, 3, V).astype(np.float32)  # many exact ties
        _, _, a = oracle.softmax_stats(l, 0.0)
        best = max(range(V), key=lambda v: (l[v], -v))  # brute force
        assert a == best


def test_greedy_returns_no_sum():
    m, z, a = oracle.softmax_stats(np.array([1.0, 4.0, 4.0, -1.0], np.float32), 0.0)
    assert (m, z, a) == (4.0, 0.0, 1)


def test_bad_arguments():
    with pytest.raises(ValueError):
        oracle.softmax_stats(np.zeros(4, np.float32), -1.0)
    with pytest.raises(ValueError):
        oracle.softmax_stats(np.zeros(4, np.float32), float("nan"))


# ------------------------------------------------------------ planted mistakes
def _mutant_stats(tmp_path, pattern, repl):
    src = open(ORACLE_C).read()
    new, n = re.subn(pattern, repl, src)
    assert n >= 1, pattern
    c, so = tmp_path / "mut.c", tmp_path / "mut.so"
    c.write_text(new)
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-shared", "-fPIC", "-o", str(so), str(c), "-lm"])
    lib = ctypes.CDLL(str(so))
    lib.oracle_softmax_stats.argtypes = oracle._load().oracle_softmax_stats.argtypes
    lib.oracle_softmax_stats.restype = ctypes.c_int

    def stats(l, T):
        l = np.ascontiguousarray(l, np.float32)
        m, z, a = ctypes.c_double(), ctypes.c_double(), ctypes.c_int32()
        lib.oracle_softmax_stats(l, len(l), float(T), ctypes.byref(m), ctypes.byref(z), ctypes.byref(a))
        return m.value, z.value, a.value
    return stats


@pytest.mark.parametrize("pattern,repl", [
    (r"Z \+= exp\(\(\(double\)logits\[v\] - m\) / T\);", "Z += exp(((double)logits[v] - m) * T);"),  # T inverted
    (r"Z \+= exp\(\(\(double\)logits\[v\] - m\) / T\);", "Z += exp(((double)logits[v] + m) / T);"),  # sign of m
    (r"if \(row\[v\] > row\[best\]\) best = v;", "if (row[v] >= row[best]) best = v;"),            # tie to the highest
])
def test_planted_mistakes_fail_the_pins(tmp_path, pattern, repl):
    stats = _mutant_stats(tmp_path, pattern, repl)
    rng = np.random.default_rng(2)
    l = (rng.standard_normal(200) * 3).astype(np.float32)
    l[7] = l[150] = l.max() + 1.0  # a tied maximum
    T = 0.7
    m, z, a = stats(l, T)
    ok_lse = np.log(z) + m / T == pytest.approx(special.logsumexp(l.astype(np.float64) / T), rel=1e-12)
    ok_arg = a == 7
    assert not (ok_lse and ok_arg)
