"""GPU checks of the draft-then-verify step graph (spec_step.SpecStep): every
draft token is the oracle sampler's draw for its slot (bit-exact unless the
oracle flags a near tie), the verification of those tokens matches the oracle
(same rule), the graph replays deterministically and agrees with the eager
launch sequence, and every linear's output is finite."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_helpers import compare_verify

pytestmark = pytest.mark.gpu

SMALL_LAYER = [("q", 512, 512), ("k", 512, 128), ("v", 512, 128), ("o", 512, 512),
               ("gate", 512, 1024), ("up", 512, 1024), ("down", 1024, 512)]


@pytest.fixture(scope="module")
def spec():
    from quantized_speculative_decoding_gb300 import build
    build.build()
    from quantized_speculative_decoding_gb300 import spec_step
    return spec_step


def _check_step(step, seed):
    g = step.gamma
    dl = step.draft_logits.cpu().numpy()
    tl = step.target_logits.cpu().numpy()
    dt = step.draft_tokens.cpu().numpy()
    for i in range(g):
        tok, flag = oracle.sample_flag(dl[0, i], step.T, seed, 0, i)
        assert flag or dt[0, i] == tok, (i, dt[0, i], tok)
    out_o, len_o, flags = oracle.verify(dl if step.T > 0 else np.zeros_like(dl), tl, dt, g, step.T, seed)
    compare_verify(step.out_tokens.cpu().numpy(), step.accept_len.cpu().numpy(), out_o, len_o, flags, g)
    for y in list(step.draft_y.values()) + list(step.target_y.values()):
        assert torch.isfinite(y.float()).all()


@pytest.mark.parametrize("fmt", ["int4-tiled", "int8", "bf16"])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_step_graph_matches_oracle(spec, fmt, T):
    from quantized_speculative_decoding_gb300 import binding as sd
    step = spec.SpecStep(draft_layer=SMALL_LAYER, draft_layers=2, draft_fmt=fmt, target_layer=SMALL_LAYER,
                         target_layers=2, gamma=4, vocab=1024, temperature=T, sigma=0.7, seed=21)
    st = torch.cuda.Stream()
    for seed in (0, 7):
        g = step.capture("step", seed, st)
        step.draft_tokens.fill_(-1)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            g.replay()
        st.synchronize()
        _check_step(step, seed)
        first = (step.draft_tokens.clone(), step.out_tokens.clone(), step.accept_len.clone())
        with torch.cuda.stream(st):
            g.replay()
        st.synchronize()
        assert torch.equal(first[0], step.draft_tokens) and torch.equal(first[1], step.out_tokens)
        # the eager launch sequence gives the same result
        step.draft_tokens.fill_(-1)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            step.step(seed, st)
        st.synchronize()
        assert torch.equal(first[0], step.draft_tokens) and torch.equal(first[2], step.accept_len)
    assert sd.sd_device_error() == 0


@pytest.mark.parametrize("gamma", [1, 3, 6])
def test_step_gamma_and_large_vocab(spec, gamma):
    step = spec.SpecStep(draft_layer=SMALL_LAYER, draft_layers=1, draft_fmt="int4-tiled",
                         target_layer=SMALL_LAYER, target_layers=1, gamma=gamma, vocab=152064,
                         temperature=1.0, sigma=0.5, seed=22 + gamma)
    st = torch.cuda.Stream()
    g = step.capture("step", 3, st)
    step.draft_tokens.fill_(-1)
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        g.replay()
    st.synchronize()
    _check_step(step, 3)


def test_step_rejects_bad_arguments(spec):
    with pytest.raises(ValueError):
        spec.SpecStep(draft_layer=SMALL_LAYER, draft_layers=1, draft_fmt="fp8", target_layer=SMALL_LAYER,
                      target_layers=1, gamma=4, vocab=1024, temperature=1.0, sigma=0.5, seed=0)
    with pytest.raises(ValueError):
        spec.SpecStep(draft_layer=SMALL_LAYER, draft_layers=1, draft_fmt="int8", target_layer=SMALL_LAYER,
                      target_layers=1, gamma=8, vocab=1024, temperature=1.0, sigma=0.5, seed=0)
