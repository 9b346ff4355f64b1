"""Pins for the oracle's speculative-sampling verification.

What the cited method fixes (references [2] Leviathan et al. and [3] Chen et
al. of "When Do Quantized Drafts Help Speculative Decoding?"):
  * each drafted token x_i ~ q_i is accepted with probability
    sum_v min(p_v, q_v) = 1 - TV(p, q)            (closed form)
  * positions are independent given the logits, so
    P(accept_len >= k) = prod_{i<k} alpha_i        (product law)
  * every emitted token is distributed as the target p at its position,
    the resample after a rejection as norm(max(0, p - q)), and the bonus as
    p_{gamma+1}                                    (output distribution)
  * greedy (T = 0) accepts exactly the prefix where the draft token is the
    target argmax.
"Speculative Decoding in Quantized Regimes", sec. 2.1 states alpha = 1 - KL
instead; the last test shows that formula disagrees with the sampler.

Planted mistakes: the last tests compile mutated copies of oracle.c (on the
CPU, in a temporary directory) and check that these pins catch them.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest
from scipy import special, stats

import oracle

ORACLE_C = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _probs(logits, T):
    return special.softmax(np.asarray(logits, np.float64) / T, axis=-1)


def _case(V=8, gamma=4, sigma=0.8, seed=0):
    rng = np.random.default_rng(seed)
    dl = (rng.standard_normal((gamma, V)) * 1.5).astype(np.float32)
    tl = np.concatenate([dl + rng.standard_normal((gamma, V)).astype(np.float32) * sigma,
                         (rng.standard_normal((1, V)) * 1.5).astype(np.float32)])
    return dl, tl.astype(np.float32)


def test_softmax_matches_scipy():
    rng = np.random.default_rng(1)
    for T in (0.3, 1.0, 2.5):
        lg = (rng.standard_normal(1000) * 3).astype(np.float32)
        lg[7] = -np.inf
        p = oracle.softmax(lg, T)
        ref = _probs(lg, T)
        assert np.allclose(p, ref, rtol=1e-12, atol=0)
        assert p[7] == 0.0


def test_greedy_accepts_the_argmax_prefix():
    rng = np.random.default_rng(2)
    B, gamma, V = 200, 5, 50
    tl = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    tl[:, :, 3] = tl[:, :, 9] = tl.max(-1) + 1  # ties: lowest index wins
    arg = np.argmax(tl, axis=-1)
    dt = arg[:, :gamma].copy()
    flip = rng.random((B, gamma)) < 0.3
    dt[flip] = (dt[flip] + 1) % V
    out, alen, flags = oracle.verify(np.zeros((B, gamma, V), np.float32), tl, dt, gamma, 0.0, 0)
    for b in range(B):
        j = next((i for i in range(gamma) if dt[b, i] != arg[b, i]), gamma)
        assert alen[b] == j
        assert list(out[b, :j]) == list(dt[b, :j])
        assert out[b, j] == arg[b, j]
        assert np.all(out[b, j + 1:] == -1)
    assert np.all(flags == 0)
    assert np.all(arg == 3)


def test_identical_distributions_accept_everything():
    dl, _ = _case(V=16, seed=3)
    tl = np.concatenate([dl, dl[:1]])
    B = 400
    dt = np.stack([np.array([oracle.sample(dl[i], 1.0, s, 0, i) for i in range(4)])
                   for s in range(B)])
    out, alen, _ = oracle.verify(np.broadcast_to(dl, (B, 4, 16)), np.broadcast_to(tl, (B, 5, 16)),
                                 dt, 4, 1.0, 77)
    assert np.all(alen == 4)


def test_disjoint_supports_reject_at_zero():
    V, gamma = 10, 3
    dl = np.full((gamma, V), -np.inf, np.float32)
    dl[:, :4] = np.random.default_rng(4).standard_normal((gamma, 4))
    tl = np.full((gamma + 1, V), -np.inf, np.float32)
    tl[:, 5:] = np.random.default_rng(5).standard_normal((gamma + 1, 5))
    res = oracle.verify_trials(dl, tl, gamma, 1.0, 0, 20000)
    assert res["hist_len"][0] == 20000
    # the resample is then p_0 itself (q_0 = 0 on p's support)
    p0 = _probs(tl[0], 1.0)
    cnt = res["hist_new"][0][5:]
    assert stats.chisquare(cnt, p0[5:] * cnt.sum()).pvalue > 1e-3


@pytest.fixture(scope="module")
def trials():
    dl, tl = _case(V=8, gamma=4, sigma=0.9, seed=6)
    n = 1_000_000
    return dl, tl, n, oracle.verify_trials(dl, tl, 4, 1.0, 123, n)


def test_acceptance_matches_closed_form(trials):
    dl, tl, n, res = trials
    for i in range(4):
        alpha = np.minimum(_probs(dl[i], 1.0), _probs(tl[i], 1.0)).sum()
        k, m = res["accepted"][i], res["reached"][i]
        sd = np.sqrt(alpha * (1 - alpha) / m)
        assert abs(k / m - alpha) < 4.5 * sd, (i, k / m, alpha)


def test_product_law(trials):
    dl, tl, n, res = trials
    alphas = [np.minimum(_probs(dl[i], 1.0), _probs(tl[i], 1.0)).sum() for i in range(4)]
    tail = np.cumsum(res["hist_len"][::-1])[::-1] / n  # P(len >= k)
    for k in range(1, 5):
        expect = np.prod(alphas[:k])
        sd = np.sqrt(expect * (1 - expect) / n)
        assert abs(tail[k] - expect) < 4.5 * sd
    mean_len = (np.arange(5) * res["hist_len"]).sum() / n
    assert abs(mean_len - sum(np.prod(alphas[:k]) for k in range(1, 5))) < 0.01


def test_emitted_tokens_follow_target(trials):
    dl, tl, n, res = trials
    for i in range(5):
        cnt = res["hist_tok"][i]
        p = _probs(tl[i], 1.0)
        assert stats.chisquare(cnt, p * cnt.sum()).pvalue > 0.01, i


def test_resample_follows_residual_and_bonus_follows_p(trials):
    dl, tl, n, res = trials
    for j in range(4):
        r = np.maximum(_probs(tl[j], 1.0) - _probs(dl[j], 1.0), 0)
        r /= r.sum()
        cnt = res["hist_new"][j]
        keep = r > 0
        assert cnt[~keep].sum() == 0
        assert stats.chisquare(cnt[keep], r[keep] * cnt.sum()).pvalue > 0.01, j
    cnt = res["hist_new"][4]
    assert stats.chisquare(cnt, _probs(tl[4], 1.0) * cnt.sum()).pvalue > 0.01
    assert res["nflag"] <= 1e-4 * n


def test_temperature_scales_both_distributions():
    dl, tl = _case(V=8, seed=7)
    res = oracle.verify_trials(dl, tl, 4, 0.6, 5, 200_000)
    alpha = np.minimum(_probs(dl[0], 0.6), _probs(tl[0], 0.6)).sum()
    k, m = res["accepted"][0], res["reached"][0]
    assert abs(k / m - alpha) < 4.5 * np.sqrt(alpha * (1 - alpha) / m)
    cnt = res["hist_tok"][0]
    assert stats.chisquare(cnt, _probs(tl[0], 0.6) * cnt.sum()).pvalue > 0.01


def test_rejected_kl_formula_disagrees_with_the_sampler(trials):
    # "Speculative Decoding in Quantized Regimes", sec. 2.1: alpha = 1 - KL(q||p).
    dl, tl, n, res = trials
    q, p = _probs(dl[0], 1.0), _probs(tl[0], 1.0)
    kl = np.sum(q * np.log(q / p))
    measured = res["accepted"][0] / res["reached"][0]
    tv = np.minimum(p, q).sum()
    assert abs(measured - tv) < 0.005
    assert abs(measured - (1 - kl)) > 0.02


def test_bad_arguments_rejected():
    dl, tl = _case(V=8, seed=8)
    with pytest.raises(ValueError):
        oracle.verify(dl[None], tl[None], np.array([[0, 1, 2, 9]], np.int32), 4, 1.0, 0)
    with pytest.raises(ValueError):
        oracle.verify(dl[None], tl[None], np.array([[0, 1, 2, 3]], np.int32), 4, -1.0, 0)


# ------------------------------------------------------------ planted mistakes
def _mutant(tmp_path, pattern, repl):
    src = open(ORACLE_C).read()
    new, n = re.subn(pattern, repl, src)
    assert n >= 1, pattern
    c = tmp_path / "mut.c"
    so = tmp_path / "mut.so"
    c.write_text(new)
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-shared", "-fPIC", "-o", str(so), str(c),
                           "-lm"])
    lib = ctypes.CDLL(str(so))
    lib.oracle_verify_trials.argtypes = oracle._load().oracle_verify_trials.argtypes
    lib.oracle_verify_trials.restype = ctypes.c_long
    return lib


def _run_trials(lib, dl, tl, n):
    V = tl.shape[-1]
    out = [np.zeros(5, np.int64), np.zeros((5, V), np.int64), np.zeros((5, V), np.int64),
           np.zeros(4, np.int64), np.zeros(4, np.int64)]
    lib.oracle_verify_trials(np.ascontiguousarray(dl).reshape(-1),
                             np.ascontiguousarray(tl).reshape(-1), 4, V, 1.0, 9, n, *out)
    return out


@pytest.mark.parametrize("pattern,repl", [
    (r"int accept = u \* q\[x\] < p\[x\];", "int accept = u * p[x] < q[x];"),  # inverted ratio
    (r"double d = p\[v\] - q\[v\];", "double d = q[v] - p[v];"),             # wrong residual
    (r"oracle_softmax\(tl \+ \(size_t\)gamma \* V, V, T, p\);",
     "oracle_softmax(tl + (size_t)(gamma - 1) * V, V, T, p);"),               # bonus row index
    (r"double key = r\[v\] / E;", "double key = r[v] * E;"),                  # wrong race key
])
def test_planted_mistakes_fail_the_pins(tmp_path, pattern, repl):
    dl, tl = _case(V=8, gamma=4, sigma=0.9, seed=6)
    lib = _mutant(tmp_path, pattern, repl)
    n = 200_000
    hist_len, hist_tok, hist_new, acc, reach = _run_trials(lib, dl, tl, n)
    failures = 0
    for i in range(5):
        p = _probs(tl[i], 1.0)
        if hist_tok[i].sum() and stats.chisquare(hist_tok[i], p * hist_tok[i].sum()).pvalue < 1e-6:
            failures += 1
    for i in range(4):
        alpha = np.minimum(_probs(dl[i], 1.0), _probs(tl[i], 1.0)).sum()
        if reach[i] and abs(acc[i] / reach[i] - alpha) > 6 * np.sqrt(alpha * (1 - alpha) / reach[i]):
            failures += 1
    # the emitted-token law or the closed form must catch every mutant
    assert failures > 0
