"""sd_verify_noalloc: the verification for callers that cannot allocate device
memory (engines that own every device byte, loops that must not block on the
allocator, memory-capped sandboxes).

Through the C ABI, two calls in a row on different inputs must give exactly
the tokens and accept lengths of sd_verify on the same inputs (bit-exact, the
bar of the other verify tests), and the oracle's, except near ties the oracle
flags: the second call also shows that the shared scratch left by the first
call does not leak into the next.  A draft token outside the vocabulary is
reported through sd_device_error, as for sd_verify.  This file sorts last so
that a run stopping at its first failure has already run every other test; it
passes alone in a fresh process as well."""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_gb300 import synth
from tests.gpu_helpers import compare_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sd():
    from quantized_speculative_decoding_gb300 import build
    build.build()
    from quantized_speculative_decoding_gb300 import binding
    return binding


def _host_inputs(B, gamma, V, sigma, T, seed):
    dl, tl = synth.logits(B, gamma, V, sigma, seed)
    return dl, tl, synth.draft_tokens(dl, T, seed)


def _inputs(B, gamma, V, sigma, T, seed):
    return tuple(torch.from_numpy(a).cuda() for a in _host_inputs(B, gamma, V, sigma, T, seed))


def _run(fn, d, B, gamma, V, T, seed):
    dl, tl, dt = d
    out = torch.full((B, gamma + 1), -7, dtype=torch.int32, device="cuda")
    alen = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    fn(dl, tl, dt, gamma, B, V, T, seed, out, alen)
    torch.cuda.synchronize()
    return out.cpu().numpy(), alen.cpu().numpy()


@pytest.mark.parametrize("B,gamma,V,T", [(1, 4, 152064, 1.0), (64, 4, 32000, 0.8),
                                         (16, 6, 151936, 0.0)])
def test_noalloc_matches_sd_verify_on_two_calls(sd, B, gamma, V, T):
    first = _inputs(B, gamma, V, 0.7, T, 31)
    second = _inputs(B, gamma, V, 1.2, T, 32)
    got1 = _run(sd.sd_verify_noalloc, first, B, gamma, V, T, 5)
    got2 = _run(sd.sd_verify_noalloc, second, B, gamma, V, T, 6)
    ref1 = _run(sd.sd_verify, first, B, gamma, V, T, 5)
    ref2 = _run(sd.sd_verify, second, B, gamma, V, T, 6)
    for got, ref in ((got1, ref1), (got2, ref2)):
        assert np.array_equal(got[0], ref[0])
        assert np.array_equal(got[1], ref[1])
    assert sd.sd_device_error() == 0
    # and the oracle's result on the same inputs (near ties excepted)
    for got, (sigma, dseed, pseed) in ((got1, (0.7, 31, 5)), (got2, (1.2, 32, 6))):
        dl, tl, dt = _host_inputs(B, gamma, V, sigma, T, dseed)
        out_o, len_o, flags = oracle.verify(dl, tl, dt, gamma, T, pseed)
        _, nflag, decisions = compare_verify(got[0], got[1], out_o, len_o, flags, gamma)
        assert nflag < 1e-4 * decisions or nflag == 0


def test_noalloc_reports_a_bad_draft_token(sd):
    B, gamma, V = 2, 4, 512
    dl, tl, dt = _host_inputs(B, gamma, V, 0.3, 1.0, 19)
    dt[1, 2] = V + 5
    d = tuple(torch.from_numpy(a).cuda() for a in (dl, tl, dt))
    _, alen = _run(sd.sd_verify_noalloc, d, B, gamma, V, 1.0, 0)
    assert sd.sd_device_error() == sd.SD_ERR_INVALID_ARG
    assert alen[1] <= 2
    assert sd.sd_device_error() == 0  # read and cleared


def test_noalloc_rejects_problems_beyond_its_scratch(sd):
    # 1 MiB of scratch: about 320 bytes per batch element at gamma 16
    B, gamma, V = 8192, 16, 64
    rc = sd.lib.sd_verify_noalloc(1 << 20, 1 << 20, 1 << 20, gamma, B, V, 1.0, 0, 1 << 20,
                                  1 << 20, None)
    assert rc == sd.SD_ERR_INVALID_ARG
