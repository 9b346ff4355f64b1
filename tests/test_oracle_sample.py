"""Pins of the oracle's draft-side sampler (oracle_sample / oracle_sample_flag):
x ~ softmax(logits / T) by the exponential race on Philox stream 1.

What fixes it, independently of the oracle's own code:
- the sampled distribution is softmax(logits / T) (chi-square at V = 8, two
  temperatures), the defining property of the exponential race;
- draws for different (batch, slot) are independent streams (chi-square test
  of independence of two slots' tokens);
- T = 0 is the argmax, lowest index on ties; T -> 0+ concentrates on it;
- near-tie flags are rare at the vocabulary size of the workloads.
"""
import numpy as np
import pytest
from scipy import stats

import oracle


def _softmax(l, T):
    z = np.asarray(l, np.float64) / T
    z -= z.max()
    e = np.exp(z)
    return e / e.sum()


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_sampler_distribution_is_softmax(T):
    logits = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4, 0.9, -2.5], np.float32)
    n = 60000
    toks = np.array([oracle.sample(logits, T, seed, 0, 0) for seed in range(n)])
    counts = np.bincount(toks, minlength=8)
    expected = n * _softmax(logits, T)
    assert stats.chisquare(counts, expected).pvalue > 1e-3


def test_sampler_streams_are_independent():
    logits = np.array([0.5, 0.0, -0.5, 1.0], np.float32)
    n = 40000
    a = np.array([oracle.sample(logits, 1.0, s, 0, 0) for s in range(n)])
    b = np.array([oracle.sample(logits, 1.0, s, 0, 1) for s in range(n)])  # other slot
    c = np.array([oracle.sample(logits, 1.0, s, 1, 0) for s in range(n)])  # other batch row
    for other in (b, c):
        table = np.zeros((4, 4), np.int64)
        np.add.at(table, (a, other), 1)
        assert stats.chi2_contingency(table).pvalue > 1e-3
        assert (a != other).mean() > 0.3  # not the same stream


def test_sampler_greedy_and_low_temperature():
    logits = np.array([1.0, 3.0, 3.0, -1.0, 2.9], np.float32)
    assert oracle.sample(logits, 0.0, 0, 0, 0) == 1          # lowest index of the tie
    tok, flag = oracle.sample_flag(logits, 0.0, 5, 0, 0)
    assert tok == 1 and not flag
    sep = np.array([0.0, 1.0, 5.0, 2.0], np.float32)
    assert all(oracle.sample(sep, 1e-3, s, 0, 0) == 2 for s in range(200))


def test_sampler_flags_are_rare_at_vocab_size():
    rng = np.random.default_rng(3)
    logits = (3.0 * rng.standard_normal(152064)).astype(np.float32)
    flags = [oracle.sample_flag(logits, 1.0, s, 0, 0)[1] for s in range(60)]
    assert sum(flags) == 0


def test_sampler_matches_sample_flag():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal(1000).astype(np.float32)
    for s in range(20):
        assert oracle.sample(logits, 0.8, s, 2, 3) == oracle.sample_flag(logits, 0.8, s, 2, 3)[0]
