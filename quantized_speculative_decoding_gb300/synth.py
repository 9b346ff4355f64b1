"""Seeded synthetic inputs shared by the tests, the bench and the oracle legs.

This module holds input RECIPES only: random weights, activations, logits and
draft tokens with the shapes and distributions of the workloads below.  It
contains none of the method's arithmetic (no quantisation, softmax, acceptance
rule or sampling of the verifier) so that the CUDA path and the CPU oracle
stay independent of each other.

Workloads (shapes are in x out, i.e. K x N, of a y = x W^T linear):
  tiny      K=512, N=1024 linear at M=5; verify vocab 1024, gamma 4, batch 1,
            T=1, draft ~ N(0, 3^2), target = draft + N(0, 0.5^2), seed 0.
  qwen7b    28 decoder layers, hidden 3584: q/o 3584x3584, k/v 3584x512,
            gate/up 3584x18944, down 18944x3584, INT4 g128, M=5 (batch 1,
            gamma 4); verify vocab 152064, sigma in {0.3, 0.7, 1.2}.
            (Qwen2.5-7B-shaped, the target of "When Do Quantized Drafts Help
            Speculative Decoding?", pilot setup.)
  qwen1p5b  28 layers, hidden 1536: q/o 1536^2, k/v 1536x256, gate/up
            1536x8960, down 8960x1536, M=1 decode, bf16 / INT8 / INT4.
            (the pilot's Qwen2.5-1.5B draft)
  llama7b   hidden 4096: q/k/v/o 4096^2, gate/up 4096x11008, down 11008x4096,
            batch 8/16/32 x (gamma+1 = 5) -> M = 40/80/160; verify vocab
            32000, sigma 0.7, T 0.8.  (the batched regime the pilot cites.)
  qwen4b    hidden 2560: q 2560x4096, k/v 2560x1024, o 4096x2560, gate/up
            2560x9728, down 9728x2560, batch 1, gamma 2..6 (M = gamma+1);
            verify vocab 151936, sigma 0.5, T in {0, 1}.
Weights ~ N(0, 0.02^2) fp32; activations ~ N(0, 1) rounded to bf16.
Seeds: weights 1000 + 100*config + 10*layer + shape index; x 7; logits
11 + config.  No dataset, prompt or trained weight stands behind any of it:
the synthetic logits stand in for model outputs and the shapes for the
models.
"""
from __future__ import annotations

import numpy as np

# (name, K, N) per linear of one decoder layer
QWEN7B_LAYER = [("q", 3584, 3584), ("k", 3584, 512), ("v", 3584, 512), ("o", 3584, 3584),
                ("gate", 3584, 18944), ("up", 3584, 18944), ("down", 18944, 3584)]
QWEN1P5B_LAYER = [("q", 1536, 1536), ("k", 1536, 256), ("v", 1536, 256), ("o", 1536, 1536),
                  ("gate", 1536, 8960), ("up", 1536, 8960), ("down", 8960, 1536)]
LLAMA7B_LAYER = [("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
                 ("gate", 4096, 11008), ("up", 4096, 11008), ("down", 11008, 4096)]
QWEN4B_LAYER = [("q", 2560, 4096), ("k", 2560, 1024), ("v", 2560, 1024), ("o", 4096, 2560),
                ("gate", 2560, 9728), ("up", 2560, 9728), ("down", 9728, 2560)]

# Linears of a layer that read the same input, packed as one weight matrix
# (rows concatenated in this order): the q/k/v and gate/up projections.
FUSED = (("qkv", ("q", "k", "v")), ("gate_up", ("gate", "up")))


def fused_layer(layer):
    """(name, K, N, member indices) per launch of a layer whose same-input
    linears are concatenated along N (rows); other linears stay alone."""
    names = [n for n, _, _ in layer]
    out, used = [], set()
    for i, (name, K, N) in enumerate(layer):
        if i in used:
            continue
        fused = next(((fname, members) for fname, members in FUSED if members[0] == name), None)
        if fused and all(m in names for m in fused[1]):
            idx = [names.index(m) for m in fused[1]]
            assert len({layer[j][1] for j in idx}) == 1
            out.append((fused[0], K, sum(layer[j][2] for j in idx), tuple(idx)))
            used.update(idx)
        else:
            out.append((name, K, N, (i,)))
            used.add(i)
    return out


WORKLOADS = {
    "tiny": dict(config=0, layers=1, layer=[("tiny", 512, 1024)], M=5, vocab=1024, gamma=4,
                 batch=1, T=1.0, sigmas=(0.5,), seed=0),
    "qwen7b": dict(config=1, layers=28, layer=QWEN7B_LAYER, M=5, vocab=152064, gamma=4,
                   batch=1, T=1.0, sigmas=(0.3, 0.7, 1.2), seed=0),
    "qwen1p5b": dict(config=2, layers=28, layer=QWEN1P5B_LAYER, M=1),
    "llama7b": dict(config=3, layers=32, layer=LLAMA7B_LAYER, batches=(8, 16, 32), gamma=4,
                    vocab=32000, T=0.8, sigmas=(0.7,), seed=0),
    "qwen4b": dict(config=4, layers=1, layer=QWEN4B_LAYER, gammas=(2, 3, 4, 5, 6), batch=1,
                   vocab=151936, temps=(0.0, 1.0), sigmas=(0.5,), seed=0),
}

DRAFT_LOGIT_STD = 3.0
WEIGHT_STD = 0.02


def weight_seed(config: int, layer: int, shape_index: int) -> int:
    return 1000 + 100 * config + 10 * layer + shape_index


def weights(N: int, K: int, seed: int) -> np.ndarray:
    """fp32 [N][K] ~ N(0, 0.02^2)."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((N, K), dtype=np.float32) * np.float32(WEIGHT_STD))


def packed_w4(N: int, K: int, seed: int):
    """A random INT4 g128 weight already in the packed layout, for shapes too
    large to draw in fp32 (the lm_head): qweight uint32 [N][K/8] uniform bits
    (every nibble uniform in 0..15), scales fp16 bits [N][K/128] uniform in
    [2^-8, 2^-7) (the range of 0.02-std weights over 15 levels), zeros fp16
    bits [N][K/128] of integers uniform in 0..15."""
    rng = np.random.default_rng(seed)
    qweight = rng.integers(0, 1 << 32, (N, K // 8), dtype=np.uint64).astype(np.uint32)
    scales = (0x1C00 + rng.integers(0, 1 << 10, (N, K // 128))).astype(np.uint16)
    zeros = rng.integers(0, 16, (N, K // 128)).astype(np.float16).view(np.uint16)
    return qweight, scales, zeros


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16) with torch's round-to-nearest-even."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def activations(M: int, K: int, seed: int = 7) -> np.ndarray:
    """bf16 bits [M][K], x ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    return to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))


def logits(batch: int, gamma: int, vocab: int, sigma: float, seed: int):
    """(draft [B][gamma][V], target [B][gamma+1][V]) fp32.

    draft ~ N(0, 3^2); target row i < gamma = draft row i + N(0, sigma^2);
    the target's bonus row gamma is a fresh N(0, 3^2) row."""
    rng = np.random.default_rng(seed)
    draft = (rng.standard_normal((batch, gamma, vocab), dtype=np.float32)
             * np.float32(DRAFT_LOGIT_STD))
    target = np.empty((batch, gamma + 1, vocab), np.float32)
    target[:, :gamma] = draft + rng.standard_normal((batch, gamma, vocab),
                                                    dtype=np.float32) * np.float32(sigma)
    target[:, gamma] = rng.standard_normal((batch, vocab), dtype=np.float32) * np.float32(
        DRAFT_LOGIT_STD)
    return draft, target


def draft_tokens(draft: np.ndarray, T: float, seed: int) -> np.ndarray:
    """The draft model's proposals, int32 [B][gamma]: a Gumbel-max draw from
    softmax(draft / T) with numpy's own generator (T > 0), or argmax (T == 0).
    These are inputs of the verifier, drawn independently of its Philox."""
    if T == 0.0:
        return np.argmax(draft, axis=-1).astype(np.int32)
    rng = np.random.default_rng(seed + 1_000_003)
    g = rng.gumbel(size=draft.shape)
    return np.argmax(draft.astype(np.float64) / T + g, axis=-1).astype(np.int32)
