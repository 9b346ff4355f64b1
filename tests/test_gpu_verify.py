"""GPU parity of the speculative-sampling verification (sd_verify) and its
Philox generator against the CPU oracle, through the C ABI.

Bars: Philox words bit-exact; accept lengths and emitted tokens bit-exact
except batch elements whose oracle decision lies within the near-tie window
(those are counted and must stay below 1e-4 of all decisions on the large
runs); on vocab 8 with 10^6 trials the GPU's emitted tokens follow the target
distribution (chi-square p > 0.01) and its acceptance rate matches the closed
form sum_v min(p, q)."""
import numpy as np
import pytest
import torch
from scipy import special, stats

import oracle
from quantized_speculative_decoding_gb300 import synth
from tests.gpu_helpers import compare_verify, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sd():
    from quantized_speculative_decoding_gb300 import build
    build.build()
    from quantized_speculative_decoding_gb300 import binding
    return binding


def _gpu_verify(sd, dl, tl, dt, gamma, T, seed):
    B, V = dt.shape[0], tl.shape[-1]
    out = torch.full((B, gamma + 1), -7, dtype=torch.int32, device="cuda")
    alen = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    d = dev(dl) if dl is not None else None
    sd.sd_verify(d, dev(tl), dev(dt), gamma, B, V, T, seed, out, alen)
    torch.cuda.synchronize()
    return out.cpu().numpy(), alen.cpu().numpy()


def _check(sd, dl, tl, dt, gamma, T, seed):
    out_g, len_g = _gpu_verify(sd, dl, tl, dt, gamma, T, seed)
    dl_o = dl if dl is not None else np.zeros((dt.shape[0], gamma, tl.shape[-1]), np.float32)
    out_o, len_o, flags = oracle.verify(dl_o, tl, dt, gamma, T, seed)
    res = compare_verify(out_g, len_g, out_o, len_o, flags, gamma)
    assert sd.sd_device_error() == 0
    return res, len_o


def test_philox_words_bit_exact(sd):
    rng = np.random.default_rng(1)
    n = 4096
    ctr = rng.integers(0, 2 ** 32, (n, 4), dtype=np.uint64).astype(np.uint32)
    ctr[:8] = 0
    ctr[8:16] = 0xffffffff
    out = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
    for key in ([0, 0], [0x12345678, 0xdeadbeef], [0xffffffff, 1]):
        sd.sd_philox4x32(dev(ctr), key[0], key[1], n, out)
        got = out.cpu().numpy().view(np.uint32)
        ref = np.stack([oracle.philox4x32(c, key) for c in ctr[::37]])
        assert np.array_equal(got[::37], ref)


def test_verify_tiny_workload(sd):
    wl = synth.WORKLOADS["tiny"]
    dl, tl = synth.logits(1, wl["gamma"], wl["vocab"], wl["sigmas"][0], 11)
    dt = synth.draft_tokens(dl, wl["T"], 11)
    (mism, nflag, _), _ = _check(sd, dl, tl, dt, wl["gamma"], wl["T"], wl["seed"])
    assert mism <= nflag


@pytest.mark.parametrize("sigma", [0.3, 1.2])
def test_verify_many_batches(sd, sigma):
    B, gamma, V = 512, 4, 1024
    dl, tl = synth.logits(B, gamma, V, sigma, 3)
    dt = synth.draft_tokens(dl, 1.0, 3)
    (mism, nflag, dec), len_o = _check(sd, dl, tl, dt, gamma, 1.0, 12345)
    assert nflag <= max(2, 1e-4 * dec)
    assert 0 < len_o.mean() < gamma  # both accept and reject paths taken


@pytest.mark.parametrize("gamma,V", [(1, 257), (16, 131), (7, 4099), (3, 2)])
def test_verify_ragged_shapes(sd, gamma, V):
    # vocab not a multiple of 4: rows start misaligned; tiny and odd chunks
    B = 64
    dl, tl = synth.logits(B, gamma, V, 0.7, gamma * V)
    dt = synth.draft_tokens(dl, 1.0, 4)
    (_, nflag, decisions), _ = _check(sd, dl, tl, dt, gamma, 1.0, 99)
    assert nflag < 1e-4 * decisions  # near ties: the only mismatches allowed, and rare


def test_verify_temperature(sd):
    B, gamma, V = 8, 4, 32000
    dl, tl = synth.logits(B, gamma, V, 0.7, 14)
    dt = synth.draft_tokens(dl, 0.8, 14)
    _check(sd, dl, tl, dt, gamma, 0.8, 0)


@pytest.mark.parametrize("gamma", [2, 4, 6])
def test_verify_greedy(sd, gamma):
    B, V = 16, 151936
    dl, tl = synth.logits(B, gamma, V, 0.5, 15)
    dt = synth.draft_tokens(dl, 0.0, 15)
    (mism, nflag, _), len_o = _check(sd, None, tl, dt, gamma, 0.0, 0)
    assert mism == 0 and nflag == 0


def test_verify_greedy_ties_pick_lowest_index(sd):
    B, gamma, V = 4, 3, 5000
    rng = np.random.default_rng(16)
    tl = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    tl[:, :, 4321] = 10.0
    tl[:, :, 77] = 10.0
    dt = np.full((B, gamma), 77, np.int32)
    out, alen = _gpu_verify(sd, None, tl, dt, gamma, 0.0, 0)
    assert np.all(alen == gamma) and np.all(out[:, gamma] == 77)


@pytest.mark.parametrize("sigma", [0.3, 0.7, 1.2])
def test_verify_qwen7b_vocab(sd, sigma):
    wl = synth.WORKLOADS["qwen7b"]
    B = 4
    dl, tl = synth.logits(B, wl["gamma"], wl["vocab"], sigma, 12)
    dt = synth.draft_tokens(dl, 1.0, 12)
    nflag = decisions = 0
    for seed in (0, 1, 2):
        (_, f, d), _ = _check(sd, dl, tl, dt, wl["gamma"], 1.0, seed)
        nflag, decisions = nflag + f, decisions + d
    assert nflag < 1e-4 * decisions  # near ties: the only mismatches allowed, and rare


def test_verify_neg_inf_logits(sd):
    B, gamma, V = 32, 4, 600
    dl, tl = synth.logits(B, gamma, V, 0.8, 17)
    dl[:, :, 300:] = -np.inf   # the draft never proposes these
    tl[:, :, :100] = -np.inf   # the target gives these zero mass
    dt = synth.draft_tokens(dl, 1.0, 17)
    (mism, _, _), len_o = _check(sd, dl, tl, dt, gamma, 1.0, 5)
    out_g, _ = _gpu_verify(sd, dl, tl, dt, gamma, 1.0, 5)
    new = out_g[np.arange(B), len_o]
    assert np.all(new >= 100)


def test_verify_identical_logits_accept_all(sd):
    B, gamma, V = 128, 5, 3000
    dl, _ = synth.logits(B, gamma, V, 0.0, 18)
    tl = np.concatenate([dl, dl[:, :1]], axis=1)
    dt = synth.draft_tokens(dl, 1.0, 18)
    out, alen = _gpu_verify(sd, dl, tl, dt, gamma, 1.0, 3)
    assert np.all(alen == gamma)


def test_verify_bad_token_recorded_not_faulted(sd):
    B, gamma, V = 2, 4, 512
    dl, tl = synth.logits(B, gamma, V, 0.3, 19)
    dt = synth.draft_tokens(dl, 1.0, 19)
    dt[1, 2] = V + 5
    out, alen = _gpu_verify(sd, dl, tl, dt, gamma, 1.0, 0)
    assert sd.sd_device_error() == sd.SD_ERR_INVALID_ARG
    assert alen[1] <= 2
    assert sd.sd_device_error() == 0  # cleared


def test_verify_statistics_vocab8(sd):
    """10^6 independent trials (batch index = trial) on one set of logits."""
    gamma, V, n = 4, 8, 1_000_000
    rng = np.random.default_rng(20)
    dl1 = (rng.standard_normal((gamma, V)) * 1.5).astype(np.float32)
    tl1 = np.concatenate([dl1 + rng.standard_normal((gamma, V)).astype(np.float32) * 0.9,
                          (rng.standard_normal((1, V)) * 1.5).astype(np.float32)])
    dl = np.broadcast_to(dl1, (n, gamma, V)).copy()
    tl = np.broadcast_to(tl1, (n, gamma + 1, V)).copy()
    dt = synth.draft_tokens(dl, 1.0, 20)
    out, alen = _gpu_verify(sd, dl, tl, dt, gamma, 1.0, 2024)
    p = special.softmax(tl1.astype(np.float64), axis=-1)
    q = special.softmax(dl1.astype(np.float64), axis=-1)
    # first emitted token ~ p_0; emitted token at position i ~ p_i
    for i in range(gamma + 1):
        reached = alen >= i
        cnt = np.bincount(out[reached, i], minlength=V)
        assert stats.chisquare(cnt, p[i] * cnt.sum()).pvalue > 0.01, i
    # per-position acceptance = sum min(p, q)
    for i in range(gamma):
        reached = alen >= i
        acc = (alen[reached] > i).mean()
        a = np.minimum(p[i], q[i]).sum()
        assert abs(acc - a) < 4.5 * np.sqrt(a * (1 - a) / reached.sum()), i
    # bit-exact against the oracle on a slice of the trials
    sl = slice(0, 4000)
    out_o, len_o, flags = oracle.verify(dl[sl], tl[sl], dt[sl], gamma, 1.0, 2024)
    compare_verify(out[sl], alen[sl], out_o, len_o, flags, gamma)
