"""GPU parity of the lm_head fused with the verification statistics
(sd_lm_head_parts, sd_w4a16_lm_head, sd_verify_parts), through the C ABI.

The lm_head's logits are the INT4 GEMM of the target's last layer; the
speculative-sampling rule (references [2], [3] of "When Do Quantized Drafts
Help Speculative Decoding?") normalises each of its rows by the softmax
statistics m = max l, Z = sum exp((l - m) / T), which the lm_head also
emits as one partial per CTA.

Bars:
  * logits: max-abs error <= 2e-4 * max|ref| against the oracle's fp64 GEMM.
    Derivation: the kernel dequantises exactly and accumulates in fp32; per
    128-input group its raw sums reach about 143 * sum|x| (levels 128 + q),
    so an fp32 rounding of them is about 2^-24 * 143 * 128 * 0.8 * s ~ 1e-5 s
    per group; over K / 128 <= 148 groups that stays below 1e-4 of a logit
    of typical size.  The bar doubles that.
  * partials, property at any size: over the logits the call wrote, the
    merged partials give m bit-exactly (the same fp32 values), log Z within
    1e-5 of scipy's logsumexp, and the argmax index exactly (lowest index on
    ties); every partial of rows < M is written and nothing past it.
  * partials against the oracle: m within the logit bar, log Z within
    2 * bar / T + 1e-5, the argmax equal unless the oracle's top two logits
    are within twice the bar.
  * sd_verify_parts against the oracle's verification on the same logits,
    with partials the oracle computes over ragged slices: tokens and accept
    lengths bit-exact except near ties the oracle flags.
  * lm_head then sd_verify_parts against sd_verify on the same logits: equal.
"""
import numpy as np
import pytest
import torch
from scipy import special

import oracle
from quantized_speculative_decoding_gb300 import synth
from tests.gpu_helpers import compare_verify, dev

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-4


@pytest.fixture(scope="module")
def sd():
    from quantized_speculative_decoding_gb300 import build
    build.build()
    from quantized_speculative_decoding_gb300 import binding
    return binding


def _tile(sd, qw, s, z, N, K):
    qb, sb = sd.sd_w4_tiled_bytes(N, K, 128)
    tq = torch.zeros(qb, dtype=torch.uint8, device="cuda")
    tsz = torch.zeros(sb // 2, dtype=torch.int16, device="cuda")
    sd.sd_w4_tile(dev(qw), dev(s), dev(z), 128, N, K, tq, tsz)
    torch.cuda.synchronize()
    return tq, tsz


def _lm_head(sd, x, tq, tsz, M, V, K, T, ld_logits=None, ld_stats=None):
    parts = sd.sd_lm_head_parts(M, V, K)
    ldl = V if ld_logits is None else ld_logits
    lds = parts if ld_stats is None else ld_stats
    logits = torch.full((M, ldl), float("nan"), dtype=torch.float32, device="cuda")
    stats = torch.full((M, lds, 2), float("nan"), dtype=torch.float32, device="cuda")
    sd.sd_w4a16_lm_head(dev(x), tq, tsz, 128, M, V, K, T, logits, ldl, stats, lds)
    torch.cuda.synchronize()
    return logits.cpu().numpy(), stats.cpu().numpy(), parts


def _merge(st, T):
    """Row statistics from one row's partials [parts][2]: (m, Z) or (m, argmax)."""
    a = st[:, 0].astype(np.float64)
    if T > 0:
        m = a.max()
        ok = a != -np.inf
        return m, float(np.sum(st[ok, 1].astype(np.float64) * np.exp((a[ok] - m) / T)))
    idx = st[:, 1].copy().view(np.int32)
    best = max(range(len(a)), key=lambda i: (a[i], -int(idx[i])))
    return a[best], int(idx[best])


def _check_partials(logits, stats, parts, M, V, T):
    """The property bars: partials describe the logits the call wrote."""
    # a written partial's max is finite or -inf (never NaN); at T = 0 its
    # index is a vocabulary index, or INT32_MAX (a NaN pattern) when empty
    assert not np.isnan(stats[:M, :parts, 0]).any(), "a partial was not written"
    if T > 0:
        assert not np.isnan(stats[:M, :parts, 1]).any()
    else:
        idx = stats[:M, :parts, 1].copy().view(np.int32)
        empty = stats[:M, :parts, 0] == -np.inf
        assert np.all(np.where(empty, idx == np.iinfo(np.int32).max, (idx >= 0) & (idx < V)))
    assert np.isnan(stats[:, parts:]).all(), "a partial past the count was written"
    for m in range(M):
        row = logits[m, :V].astype(np.float64)
        mm, zz = _merge(stats[m, :parts], T)
        assert mm == row.max()
        if T > 0:
            assert np.log(zz) + mm / T == pytest.approx(special.logsumexp(row / T), abs=1e-5)
        else:
            assert zz == int(np.argmax(logits[m, :V]))


def _against_oracle(logits, stats, parts, y_ref, rows, T):
    """Logits of the sampled vocabulary rows against the oracle's fp64 GEMM;
    with every row sampled, the merged partials against the oracle's stats."""
    M = y_ref.shape[0]
    scale = np.abs(y_ref).max()
    err = np.abs(logits[:M][:, rows].astype(np.float64) - y_ref).max()
    assert err <= LOGIT_TOL * scale, f"logits: max-abs err {err:.3e} > {LOGIT_TOL * scale:.3e}"
    if len(rows) != logits.shape[1] or not np.array_equal(rows, np.arange(len(rows))):
        return
    bar = LOGIT_TOL * scale
    for m in range(M):
        ref32 = y_ref[m].astype(np.float32)
        om, oz, oa = oracle.softmax_stats(ref32, T)
        gm, gz = _merge(stats[m, :parts], T)
        assert abs(gm - om) <= bar
        if T > 0:
            assert abs(np.log(gz) - np.log(oz)) <= 2 * bar / T + 1e-5
        else:
            top2 = np.sort(y_ref[m])[-2:]
            if top2[1] - top2[0] > 2 * bar:
                assert gz == oa


@pytest.mark.parametrize("M,V,K", [(5, 1024, 512), (1, 1000, 1536), (8, 4099, 3584), (13, 777, 1024),
                                   (32, 300, 256), (3, 16, 128)])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_lm_head_parity(sd, M, V, K, T):
    seed = 7 * M + V + K
    w = synth.weights(V, K, seed)
    qw = np.zeros((V, K // 8), np.uint32)
    s = np.zeros((V, K // 128), np.uint16)
    z = np.zeros((V, K // 128), np.uint16)
    sd.sd_w4_pack(w, V, K, 128, qw, s, z)
    tq, tsz = _tile(sd, qw, s, z, V, K)
    x = synth.activations(M, K, seed=seed + 1)
    logits, stats, parts = _lm_head(sd, x, tq, tsz, M, V, K, T)
    assert parts >= 1
    _check_partials(logits, stats, parts, M, V, T)
    _against_oracle(logits, stats, parts, oracle.w4a16_linear(x, qw, s, z, 128, V, K), np.arange(V), T)
    assert sd.sd_device_error() == 0


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_lm_head_qwen7b_vocab(sd, T):
    """The 7B target's lm_head at verify M = 5: V = 152064, K = 3584 (random
    packed INT4 weights); sampled vocabulary rows against the oracle, the
    partials' properties over every row."""
    M, V, K = 5, 152064, 3584
    qw, s, z = synth.packed_w4(V, K, 4242)
    tq, tsz = _tile(sd, qw, s, z, V, K)
    x = synth.activations(M, K, seed=4243)
    logits, stats, parts = _lm_head(sd, x, tq, tsz, M, V, K, T)
    _check_partials(logits, stats, parts, M, V, T)
    rows = np.unique(np.concatenate([np.arange(0, V, 997), [V - 17, V - 1]]))
    _against_oracle(logits, stats, parts, oracle.w4a16_linear(x, qw[rows], s[rows], z[rows], 128, len(rows), K),
                    rows, T)
    assert sd.sd_device_error() == 0


def test_lm_head_strided_rows(sd):
    """The draft-step layout: row strides past the vocabulary and the parts."""
    M, V, K, T = 3, 1000, 512, 0.8
    w = synth.weights(V, K, 90)
    qw = np.zeros((V, K // 8), np.uint32)
    s = np.zeros((V, K // 128), np.uint16)
    z = np.zeros((V, K // 128), np.uint16)
    sd.sd_w4_pack(w, V, K, 128, qw, s, z)
    tq, tsz = _tile(sd, qw, s, z, V, K)
    x = synth.activations(M, K, seed=91)
    parts = sd.sd_lm_head_parts(M, V, K)
    logits, stats, _ = _lm_head(sd, x, tq, tsz, M, V, K, T, ld_logits=4 * V, ld_stats=4 * parts)
    assert np.isnan(logits[:, V:]).all()
    _check_partials(logits, stats, parts, M, V, T)
    _against_oracle(logits[:, :V], stats, parts, oracle.w4a16_linear(x, qw, s, z, 128, V, K), np.arange(V), T)


# ------------------------------------------------------------- verify_parts
def _oracle_partials(rows, T, edges):
    """Partials the oracle computes over the slices [edges[i], edges[i+1])."""
    R = rows.shape[0]
    out = np.empty((R, len(edges) - 1, 2), np.float32)
    for r in range(R):
        for i, (e0, e1) in enumerate(zip(edges[:-1], edges[1:])):
            m, zz, a = oracle.softmax_stats(rows[r, e0:e1], T)
            out[r, i, 0] = m
            out[r, i, 1] = zz if T > 0 else np.array([e0 + a], np.int32).view(np.float32)[0]
    return out


def _ragged_edges(V, n, seed):
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, V), size=min(n - 1, V - 1), replace=False))
    return [0] + [int(c) for c in cuts] + [V]


def _pad_empty(parts, npad, T, seed):
    """Insert npad empty partials ((-inf, 0), or (-inf, INT32_MAX) at T = 0),
    as CTAs that stored no logit of a row write them, at random positions."""
    if npad == 0:
        return parts
    R, n, _ = parts.shape
    empty = np.array([-np.inf, 0.0 if T > 0 else np.array([2 ** 31 - 1], np.int32).view(np.float32)[0]],
                     np.float32)
    pos = np.sort(np.random.default_rng(seed).integers(0, n + 1, npad))
    return np.ascontiguousarray(np.insert(parts, pos, empty, axis=1))


@pytest.mark.parametrize("B,gamma,V,sigma,T,nparts,npad", [
    (64, 4, 1000, 0.7, 1.0, 7, 0), (16, 7, 4099, 0.3, 0.8, 1, 0), (32, 4, 1000, 1.2, 1.0, 300, 0),
    (48, 4, 1000, 0.5, 0.0, 9, 0), (8, 16, 257, 0.7, 1.0, 2, 1500), (2, 4, 152064, 0.7, 1.0, 300, 0),
    (16, 4, 8, 0.7, 1.0, 3, 40), (16, 4, 8, 0.7, 0.0, 3, 40), (4, 4, 1000, 0.7, 0.0, 5, 2000)])
def test_verify_parts_parity(sd, B, gamma, V, sigma, T, nparts, npad):
    """Oracle partials over ragged slices, with empty partials mixed in (more
    partials than vocabulary entries, several chunks of partials per row)."""
    dl, tl = synth.logits(B, gamma, V, sigma, 100 + B)
    dt = synth.draft_tokens(dl, T, 100 + B)
    edges = _ragged_edges(V, nparts, B + gamma)
    tstats = _pad_empty(_oracle_partials(tl.reshape(-1, V), T, edges), npad, T, 1)
    dstats = _pad_empty(_oracle_partials(dl.reshape(-1, V), T, edges), npad, T, 2) if T > 0 else None
    tp = tstats.shape[1]
    out = torch.full((B, gamma + 1), -7, dtype=torch.int32, device="cuda")
    alen = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    seed = 31 + B
    sd.sd_verify_parts(dev(dl) if T > 0 else None, dev(tl), dev(dstats) if T > 0 else None, tp if T > 0 else 0,
                       dev(tstats), tp, dev(dt), gamma, B, V, T, seed, out, alen)
    torch.cuda.synchronize()
    out_o, len_o, flags = oracle.verify(dl, tl, dt, gamma, T, seed)
    compare_verify(out.cpu().numpy(), alen.cpu().numpy(), out_o, len_o, flags, gamma)
    assert sd.sd_device_error() == 0


# ------------------------------------------------------------- composition
@pytest.mark.parametrize("B,T,V,K", [(1, 1.0, 4099, 512), (3, 1.0, 4099, 512), (2, 0.0, 4099, 512),
                                     (1, 1.0, 16, 3584), (2, 0.0, 16, 3584)])
def test_lm_head_then_verify_parts_matches_verify(sd, B, T, V, K):
    gamma = 4
    qw, s, z = synth.packed_w4(V, K, 77)
    tq, tsz = _tile(sd, qw, s, z, V, K)
    # the target's rows b (gamma + 1) + i in one call
    Mt = B * (gamma + 1)
    pt = sd.sd_lm_head_parts(Mt, V, K)
    xt = synth.activations(Mt, K, seed=78)
    tl = torch.empty((B, gamma + 1, V), dtype=torch.float32, device="cuda")
    ts = torch.full((B, gamma + 1, pt, 2), float("nan"), dtype=torch.float32, device="cuda")
    sd.sd_w4a16_lm_head(dev(xt), tq, tsz, 128, Mt, V, K, T, tl, V, ts, pt)
    # the draft's step i writes row (b, i) of [B][gamma][...] through the strides
    pd = sd.sd_lm_head_parts(B, V, K)
    dl = torch.empty((B, gamma, V), dtype=torch.float32, device="cuda")
    ds = torch.full((B, gamma, pd, 2), float("nan"), dtype=torch.float32, device="cuda")
    for i in range(gamma):
        xd = dev(synth.activations(B, K, seed=80 + i))
        sd.sd_w4a16_lm_head(xd, tq, tsz, 128, B, V, K, T, dl[:, i].data_ptr(), gamma * V,
                            ds[:, i].data_ptr(), gamma * pd)
    torch.cuda.synchronize()
    assert not torch.isnan(ts[..., 0]).any() and not torch.isnan(ds[..., 0]).any()  # every partial written
    dt = dev(synth.draft_tokens(dl.cpu().numpy(), T, 79))
    outs = []
    for parts_path in (True, False):
        out = torch.full((B, gamma + 1), -7, dtype=torch.int32, device="cuda")
        alen = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        if parts_path:
            sd.sd_verify_parts(dl, tl, ds, pd, ts, pt, dt, gamma, B, V, T, 5, out, alen)
        else:
            sd.sd_verify(dl, tl, dt, gamma, B, V, T, 5, out, alen)
        torch.cuda.synchronize()
        outs.append((out.cpu().numpy(), alen.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    assert sd.sd_device_error() == 0
