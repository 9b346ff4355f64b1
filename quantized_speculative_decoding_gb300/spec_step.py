"""One speculative-decoding step, draft gamma tokens then verify, as one CUDA graph.

"When Do Quantized Drafts Help Speculative Decoding?" (pilot setup): a small
draft model proposes gamma tokens one at a time, x_i ~ q_i, and the target
model scores all gamma + 1 positions in one forward pass at batch 1, after
which speculative sampling accepts a prefix and emits one more token.  The
pages time the draft's share of that step against the draft's precision.

This module strings the library's calls together on one stream, in that
order, and captures them in a CUDA graph:

    for i in 0 .. gamma - 1:
        the draft's linears at M = 1 (every layer, its precision: INT4 tiled,
        INT8 per channel or bf16)
        sd_sample(draft logits of position i, slot i) -> draft token i
    the target's W4A16 linears at M = gamma + 1 (every layer, tiled layout)
    sd_verify(draft logits, target logits, draft tokens) -> tokens, accept length

Only the linears' weight streams and the sampling / verification are on the
path: attention, normalisation, embeddings and the lm_head are not, so the
logits are synthetic resident buffers (the stand-ins for model outputs) and
every linear reads a fixed resident activation.  The draft tokens are real
data flow: sd_sample writes token i into column i of the buffer sd_verify
reads.  Batch 1, as in the pilot setup.

The module does host-side orchestration only: every step runs in the
library's kernels, through the C ABI.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as sd
from . import synth


def _dev16(a: np.ndarray, dev) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    view = {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16}.get(a.dtype)
    return torch.from_numpy(a.view(view) if view is not None else a).to(dev)


def weight_bytes(fmt: str, N: int, K: int) -> int:
    """Bytes of one linear's weights in a format (the stream each call reads)."""
    if fmt == "bf16":
        return 2 * N * K
    if fmt == "int8":
        return N * K + 2 * N
    return N * K // 2 + 4 * N * (K // 128)


def _layer_weights(layer, config: int, fmt: str, dev):
    """(shapes, weights) of one layer in a format, same-input linears packed as
    one matrix (q|k|v, gate|up): shapes (name, K, N) and one tuple of device
    tensors per packed matrix, in the argument order of its linear call."""
    shapes, out = [], []
    for name, K, N, idx in synth.fused_layer(layer):
        w = np.concatenate([synth.weights(layer[j][2], K, synth.weight_seed(config, 0, j)) for j in idx])
        if fmt == "bf16":
            out.append((_dev16(synth.to_bf16_bits(w), dev),))
        elif fmt == "int8":
            q = np.zeros((N, K), np.int8)
            s = np.zeros((N,), np.uint16)
            sd.sd_w8_pack(w, N, K, q, s)
            out.append((torch.from_numpy(q).to(dev), _dev16(s, dev)))
        else:
            qw = np.zeros((N, K // 8), np.uint32)
            s = np.zeros((N, K // 128), np.uint16)
            z = np.zeros((N, K // 128), np.uint16)
            sd.sd_w4_pack(w, N, K, 128, qw, s, z)
            t = tuple(_dev16(a, dev) for a in (qw, s, z))
            qb, sb = sd.sd_w4_tiled_bytes(N, K, 128)
            tt = (torch.empty(qb, dtype=torch.uint8, device=dev),
                  torch.empty(sb // 2, dtype=torch.int16, device=dev))
            sd.sd_w4_tile(*t, 128, N, K, *tt)
            torch.cuda.synchronize(dev)
            out.append(tt)
        shapes.append((name, K, N))
    return shapes, out


def build_weights(layer, layers: int, config: int, fmt: str, dev):
    """(shapes, weights[layer][matrix]) of a model's linears: layer 0 built
    on the host and copied to every layer, so each layer reads its own buffers."""
    shapes, base = _layer_weights(layer, config, fmt, dev)
    return shapes, [[tuple(t.clone() for t in b) for b in base] for _ in range(layers)]


class SpecStep:
    """Device buffers and the launch sequence of one draft-then-verify step.

    draft_layer / target_layer: (name, K, N) per linear of one layer; in both
    models the same-input linears are packed as one matrix (q|k|v, gate|up).
    draft_weights / target_weights: prebuilt build_weights() results, else
    built here."""

    def __init__(self, *, draft_layer, draft_layers: int, draft_fmt: str, target_layer,
                 target_layers: int, gamma: int, vocab: int, temperature: float, sigma: float,
                 seed: int, device=None, draft_config: int = 2, target_config: int = 1,
                 draft_weights=None, target_weights=None):
        if draft_fmt not in ("int4-tiled", "int8", "bf16"):
            raise ValueError(f"draft format {draft_fmt}")
        if not 1 <= gamma <= 7:
            raise ValueError("gamma must be 1..7 (target M = gamma + 1 <= 8)")
        self.dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.gamma, self.vocab, self.T = gamma, vocab, float(temperature)
        self.draft_fmt = draft_fmt
        dev = self.dev
        # draft (M = 1) and target (M = gamma + 1): one launch per packed matrix;
        # (shapes, per-layer weights) from build_weights() may be shared by steps
        self.draft_shapes, self.draft_w = draft_weights or build_weights(
            draft_layer, draft_layers, draft_config, draft_fmt, dev)
        self.draft_x = {K: _dev16(synth.activations(1, K), dev) for _, K, _ in self.draft_shapes}
        self.draft_y = {N: torch.empty((1, N), dtype=torch.bfloat16, device=dev) for _, _, N in self.draft_shapes}
        self.target_shapes, self.target_w = target_weights or build_weights(
            target_layer, target_layers, target_config, "int4-tiled", dev)
        M = gamma + 1
        self.target_x = {K: _dev16(synth.activations(M, K), dev) for _, K, _ in self.target_shapes}
        self.target_y = {N: torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _, _, N in self.target_shapes}
        # logits (synthetic stand-ins for the two models' outputs), tokens, results
        dl, tl = synth.logits(1, gamma, vocab, sigma, seed)
        self.draft_logits = torch.from_numpy(dl).to(dev)
        self.target_logits = torch.from_numpy(tl).to(dev)
        self.draft_tokens = torch.full((1, gamma), -1, dtype=torch.int32, device=dev)
        self.out_tokens = torch.full((1, gamma + 1), -1, dtype=torch.int32, device=dev)
        self.accept_len = torch.full((1,), -1, dtype=torch.int32, device=dev)

    # -- the launch sequence ------------------------------------------------
    def draft(self, seed: int, stream) -> int:
        """gamma x (draft linears + sd_sample); returns the launches issued."""
        n = 0
        for i in range(self.gamma):
            for layer in self.draft_w:
                for (_, K, N), b in zip(self.draft_shapes, layer):
                    x, y = self.draft_x[K], self.draft_y[N]
                    if self.draft_fmt == "int4-tiled":
                        sd.sd_w4a16_linear_tiled(x, *b, 128, 1, N, K, y, stream)
                    elif self.draft_fmt == "int8":
                        sd.sd_w8a16_linear(x, *b, 1, N, K, y, stream)
                    else:
                        sd.sd_bf16_linear(x, b[0], 1, N, K, y, stream)
                    n += 1
            sd.sd_sample(self.draft_logits[0, i], 1, self.vocab, self.T, seed, i,
                         self.draft_tokens[0, i:i + 1], stream)
            n += 1
        return n

    def target(self, seed: int, stream) -> int:
        """Target linears at M = gamma + 1, then sd_verify; returns launches."""
        M, n = self.gamma + 1, 0
        for layer in self.target_w:
            for (_, K, N), b in zip(self.target_shapes, layer):
                sd.sd_w4a16_linear_tiled(self.target_x[K], *b, 128, M, N, K, self.target_y[N], stream)
                n += 1
        sd.sd_verify(self.draft_logits, self.target_logits, self.draft_tokens, self.gamma, 1, self.vocab,
                     self.T, seed, self.out_tokens, self.accept_len, stream)
        return n + (2 if self.T > 0 else 1)

    def step(self, seed: int, stream) -> int:
        return self.draft(seed, stream) + self.target(seed, stream)

    def capture(self, part: str, seed: int, stream) -> torch.cuda.CUDAGraph:
        """A CUDA graph of the step ("step"), or of its draft or target part.

        The Philox seed is a kernel argument and is recorded in the graph:
        every replay draws the same uniforms for sd_sample and sd_verify, so
        replays repeat one step (what timing needs) rather than advance a
        decode.  A decode loop captures one graph per seed, or calls step()
        with a new seed each time."""
        body = {"step": self.step, "draft": self.draft, "target": self.target}[part]
        with torch.cuda.stream(stream):
            body(seed, stream)  # first call outside capture: library workspaces
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body(seed, stream)
        return g

    # -- byte counts ---------------------------------------------------------
    def draft_weight_bytes(self) -> int:
        return len(self.draft_w) * sum(weight_bytes(self.draft_fmt, N, K) for _, K, N in self.draft_shapes)

    def target_weight_bytes(self) -> int:
        return len(self.target_w) * sum(weight_bytes("int4", N, K) for _, K, N in self.target_shapes)
