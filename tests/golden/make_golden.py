"""Writes tests/golden/oracle_tiny.json from the CPU oracle alone.

The fixture is the tiny workload (one K=512, N=1024 W4A16 linear at M=5; a
verify on vocab 1024, gamma 4, batch 1, T 1, draft ~ N(0, 3^2), target = draft
+ N(0, 0.5^2), Philox seed 0; the target rows' softmax statistics; the same
linear with INT3 / INT2 weights and with W4A4 activations) evaluated by the
oracle: a regression record
that later changes to the oracle's arithmetic must either reproduce or
justify.  The pages print no worked example of this arithmetic, so every
stored value here comes from the oracle and none from the CUDA path.

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from quantized_speculative_decoding_gb300 import synth  # noqa: E402


def _pack(q):
    N, K = q.shape
    q = q.astype(np.uint32).reshape(N, K // 8, 8)
    return np.bitwise_or.reduce(q << (4 * np.arange(8, dtype=np.uint32)), axis=2).astype(np.uint32)


def make():
    wl = synth.WORKLOADS["tiny"]
    _, K, N = wl["layer"][0]
    w = synth.weights(N, K, synth.weight_seed(0, 0, 0))
    q, s, z = oracle.quantize_w4(w, 128)
    x = synth.activations(wl["M"], K)
    y = oracle.w4a16_linear(x, _pack(q), s, z, 128, N, K)
    dl, tl = synth.logits(wl["batch"], wl["gamma"], wl["vocab"], wl["sigmas"][0], 11)
    dt = synth.draft_tokens(dl, wl["T"], 11)
    out, alen, flags = oracle.verify(dl, tl, dt, wl["gamma"], wl["T"], wl["seed"])
    cols = [0, 1, 511, 512, 1023]
    # the softmax row statistics of the tiny target rows, and the low-bit
    # formats on the tiny linear: INT3 / INT2 weights, W4A4 activations
    stats = [list(oracle.softmax_stats(tl[0, i], wl["T"])) for i in range(wl["gamma"] + 1)]
    lowbit = {}
    for bits in (3, 2):
        qb, sb, zb = oracle.quantize_wb(w, bits)
        pb = oracle.pack_wb(qb, bits)
        yb = oracle.wb_linear(x, pb, sb, zb, 128, bits, N, K)
        lowbit[f"int{bits}"] = {"packed_first": [int(v) for v in pb[0, :4]], "q_sum": int(qb.astype(np.int64).sum()),
                                "y": [[float(yb[m, c]) for c in cols] for m in range(wl["M"])]}
    qx, sx = oracle.quantize_a4(x)
    y44 = oracle.w4a4_linear(x, _pack(q), s, z, N, K)
    lowbit["w4a4"] = {"qx_first": [int(v) for v in qx[0, :16]], "sx": [float(v) for v in sx.reshape(-1)],
                      "y": [[float(y44[m, c]) for c in cols] for m in range(wl["M"])]}
    return {
        "source": "oracle only (tests/golden/make_golden.py); workload 'tiny' of synth.py",
        "w4a16": {"q_sum": int(q.astype(np.int64).sum()),
                  "scales_first": [int(v) for v in s[0]], "zeros_first": [int(v) for v in z[0]],
                  "y_cols": cols, "y": [[float(y[m, c]) for c in cols] for m in range(wl["M"])]},
        "verify": {"draft_tokens": dt.tolist(), "out_tokens": out.tolist(),
                   "accept_len": alen.tolist(), "flags": flags.tolist()},
        "softmax_stats": [[float(a), float(b), int(c)] for a, b, c in stats],
        "lowbit": lowbit,
    }


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json")
    with open(path, "w") as f:
        json.dump(make(), f, indent=1)
    print("wrote", path)
