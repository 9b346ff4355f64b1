"""GPU parity of the quantisation variants against the fp64 CPU oracle, through
the C ABI: the INT3 / INT2 group-128 linear on the b-bit tiled layout
(sd_wb_tile + sd_wb_linear_tiled, the INT3 / INT2 targets of "Speculative
Decoding in Quantized Regimes", sec. 4.1-4.2) and the W4A4 draft linear
(sd_a4_quantize + sd_w4a4_linear_tiled, QSPEC as cited by "When Do Quantized
Drafts Help Speculative Decoding?").

Inputs are packed by the oracle's own quantisers.  Bars: activation codes and
scales bit-exact; one-hot probes bit-exact where the arithmetic is exact;
everything else max-abs error <= 1e-2 * max|ref|.  The 7B shapes are checked
on sampled output rows the oracle computes one by one."""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_gb300 import synth
from tests.gpu_helpers import assert_close, bf16_bits, bf16_out, bf16_to_np64, dev

pytestmark = pytest.mark.gpu

SAMPLE = np.array([0, 1, 15, 16, 17, 255, 256, 511, 1000, 2047, 3583, 4095, 9000, 18943, 37887])


@pytest.fixture(scope="module")
def sd():
    from quantized_speculative_decoding_gb300 import build
    build.build()
    from quantized_speculative_decoding_gb300 import binding
    return binding


def _tiled_wb(sd, w, bits):
    """Oracle-quantised b-bit weights, their R11 stream and the device tiled copy."""
    N, K = w.shape
    q, s, z = oracle.quantize_wb(w, bits)
    packed = oracle.pack_wb(q, bits)
    qb, sb = sd.sd_wb_tiled_bytes(N, K, bits)
    tq = torch.full((qb,), 0x5A, dtype=torch.uint8, device="cuda")
    tsz = torch.full((sb // 4,), -1, dtype=torch.int32, device="cuda")
    sd.sd_wb_tile(dev(packed), dev(s), dev(z), 128, bits, N, K, tq, tsz)
    torch.cuda.synchronize()
    assert sd.sd_device_error() == 0
    return packed, s, z, tq, tsz


def _wb_run(sd, xb, tq, tsz, bits, M, N, K):
    out = bf16_out(M, N)
    sd.sd_wb_linear_tiled(dev(xb), tq, tsz, 128, bits, M, N, K, out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("M,N,K", [(5, 1024, 512), (1, 1000, 384), (8, 77, 1024), (3, 4096, 256),
                                   (13, 520, 1024)])
def test_wb_linear_matches_oracle(sd, bits, M, N, K):
    w = synth.weights(N, K, 40 + bits + N)
    packed, s, z, tq, tsz = _tiled_wb(sd, w, bits)
    xb = synth.activations(M, K, seed=M + K)
    out = _wb_run(sd, xb, tq, tsz, bits, M, N, K)
    ref = oracle.wb_linear(xb, packed, s, z, 128, bits, N, K)
    assert_close(bf16_to_np64(out), ref, f"int{bits} M={M} N={N} K={K}")


@pytest.mark.parametrize("bits", [2, 3])
def test_wb_one_hot_probes_bit_exact(sd, bits):
    # x = e_k: output column n is bf16(w'[n][k]) exactly (s (128 + q) and
    # s (128 + z) are exact in fp32, so is their difference)
    N, K = 200, 1024
    w = synth.weights(N, K, 50 + bits)
    packed, s, z, tq, tsz = _tiled_wb(sd, w, bits)
    ks = [0, 1, 2, 3, 16, 63, 64, 127, 128, 129, 513, 1016, 1023]
    x = np.zeros((len(ks), K), np.float32)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    xb = synth.to_bf16_bits(x)
    outs = []
    for m0 in range(0, len(ks), 8):  # the kernel takes rows of x in blocks of 8
        outs.append(bf16_bits(_wb_run(sd, xb[m0:m0 + 8], tq, tsz, bits, min(8, len(ks) - m0), N, K)))
    q = oracle.unpack_wb(packed, N, K, bits)
    wq = (q.astype(np.float64) - np.repeat(oracle.f16_to_f64(z), 128, axis=1)) * np.repeat(
        oracle.f16_to_f64(s), 128, axis=1)
    assert np.array_equal(np.concatenate(outs), oracle.round_bf16(wq[:, ks].T.copy()))


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("name,K,N", synth.QWEN7B_LAYER)
def test_wb_qwen7b_shapes_sampled_rows(sd, bits, name, K, N):
    # full-size shapes at M = 5: every output against the oracle on sampled rows
    w = synth.weights(N, K, synth.weight_seed(1, 0, 0))
    packed, s, z, tq, tsz = _tiled_wb(sd, w, bits)
    xb = synth.activations(5, K, seed=3)
    out = bf16_to_np64(_wb_run(sd, xb, tq, tsz, bits, 5, N, K))
    rows = np.unique(np.concatenate([SAMPLE[SAMPLE < N], [N - 1]]))
    ref = oracle.wb_linear(xb, packed[rows], s[rows], z[rows], 128, bits, len(rows), K)
    assert_close(out[:, rows], ref, f"int{bits} {name}")


def test_wb_tile_reports_a_bad_zero_point(sd):
    N, K, bits = 32, 256, 2
    w = synth.weights(N, K, 61)
    q, s, z = oracle.quantize_wb(w, bits)
    z = z.copy()
    z[3, 1] = oracle.f64_to_f16_bits(5.0)  # outside [0, 3]
    packed = oracle.pack_wb(q, bits)
    qb, sb = sd.sd_wb_tiled_bytes(N, K, bits)
    tq = torch.empty((qb,), dtype=torch.uint8, device="cuda")
    tsz = torch.empty((sb // 4,), dtype=torch.int32, device="cuda")
    sd.sd_wb_tile(dev(packed), dev(s), dev(z), 128, bits, N, K, tq, tsz)
    torch.cuda.synchronize()
    assert sd.sd_device_error() == sd.SD_ERR_INVALID_ARG
    assert sd.sd_device_error() == 0


def test_wb_bits4_is_the_int4_path(sd):
    N, K, M = 300, 512, 5
    w = synth.weights(N, K, 62)
    packed, s, z, tq, tsz = _tiled_wb(sd, w, 4)
    xb = synth.activations(M, K, seed=4)
    out = _wb_run(sd, xb, tq, tsz, 4, M, N, K)
    ref = oracle.wb_linear(xb, packed, s, z, 128, 4, N, K)
    assert_close(bf16_to_np64(out), ref, "int4 through sd_wb_linear_tiled")


# ------------------------------------------------------------------ W4A4
def _a4(sd, xb):
    M, K = xb.shape
    qx = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    sx = torch.full((M, K // 128), float("nan"), dtype=torch.float32, device="cuda")
    sd.sd_a4_quantize(dev(xb), M, K, qx, sx)
    torch.cuda.synchronize()
    return qx, sx


def _tiled_w4(sd, w):
    N, K = w.shape
    q, s, z = oracle.quantize_w4(w)
    qw = oracle.pack_wb(q, 4)
    qb, sb = sd.sd_w4_tiled_bytes(N, K)
    tq = torch.empty((qb,), dtype=torch.uint8, device="cuda")
    tsz = torch.empty((sb // 4,), dtype=torch.int32, device="cuda")
    sd.sd_w4_tile(dev(qw), dev(s), dev(z), 128, N, K, tq, tsz)
    torch.cuda.synchronize()
    return qw, s, z, tq, tsz


@pytest.mark.parametrize("M,K,scale", [(1, 1536, 1.0), (5, 3584, 1.0), (8, 8960, 30.0), (3, 256, 1e-30),
                                       (2, 128, 1e3)])
def test_a4_codes_and_scales_bit_exact(sd, M, K, scale):
    x = synth.activations(M, K, seed=K + M)
    xb = synth.to_bf16_bits(oracle.bf16_to_f64(x).astype(np.float32) * np.float32(scale))
    xb[0, :128] = 0  # an all-zero group: s = 1, codes 0
    qx, sx = _a4(sd, xb)
    assert sd.sd_device_error() == 0
    q_ref, s_ref = oracle.quantize_a4(xb)
    assert np.array_equal(qx.float().cpu().numpy().astype(np.int8), q_ref)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


def test_a4_quantize_reports_non_finite_input(sd):
    xb = synth.activations(2, 256, seed=5)
    xb[1, 130] = 0x7F80  # +inf
    _a4(sd, xb)
    assert sd.sd_device_error() == sd.SD_ERR_INVALID_ARG
    assert sd.sd_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(1, 2048, 1536), (5, 1024, 512), (8, 77, 1024), (13, 300, 384)])
def test_w4a4_linear_matches_oracle(sd, M, N, K):
    w = synth.weights(N, K, 70 + M)
    qw, s, z, tq, tsz = _tiled_w4(sd, w)
    xb = synth.activations(M, K, seed=71 + M)
    qx, sx = _a4(sd, xb)
    out = bf16_out(M, N)
    sd.sd_w4a4_linear_tiled(qx, sx, tq, tsz, 128, M, N, K, out)
    torch.cuda.synchronize()
    ref = oracle.w4a4_linear(xb, qw, s, z, N, K)
    assert_close(bf16_to_np64(out), ref, f"w4a4 M={M} N={N} K={K}")


def test_w4a4_one_hot_probes_bit_exact(sd):
    # x = 7 * 2^e * e_k: s_x = 2^e exactly, code 7, every other group all zero;
    # the output is 2^e * s * 7 (q - z), exact in fp32, then rounded to bf16
    N, K = 136, 1024
    w = synth.weights(N, K, 72)
    qw, s, z, tq, tsz = _tiled_w4(sd, w)
    ks = [0, 5, 127, 128, 300, 777, 1023]
    x = np.zeros((len(ks), K), np.float32)
    for m, k in enumerate(ks):
        x[m, k] = 7.0 * 2.0 ** (m - 3)
    xb = synth.to_bf16_bits(x)
    qx, sx = _a4(sd, xb)
    out = bf16_out(len(ks), N)
    sd.sd_w4a4_linear_tiled(qx, sx, tq, tsz, 128, len(ks), N, K, out)
    torch.cuda.synchronize()
    ref = oracle.w4a4_linear(xb, qw, s, z, N, K)
    assert np.array_equal(bf16_bits(out), oracle.round_bf16(ref))


@pytest.mark.parametrize("name,K,N", synth.QWEN1P5B_LAYER)
def test_w4a4_qwen1p5b_draft_shapes(sd, name, K, N):
    # the 1.5B draft's shapes at M = 1, sampled rows
    w = synth.weights(N, K, synth.weight_seed(2, 0, 0))
    qw, s, z, tq, tsz = _tiled_w4(sd, w)
    xb = synth.activations(1, K, seed=9)
    qx, sx = _a4(sd, xb)
    out = bf16_out(1, N)
    sd.sd_w4a4_linear_tiled(qx, sx, tq, tsz, 128, 1, N, K, out)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([SAMPLE[SAMPLE < N], [N - 1]]))
    ref = oracle.w4a4_linear(xb, qw[rows], s[rows], z[rows], len(rows), K)
    assert_close(bf16_to_np64(out)[:, rows], ref, f"w4a4 {name}")


def test_lowbit_repeated_launches_bit_identical(sd):
    N, K, M = 3584, 3584, 5
    w = synth.weights(N, K, 80)
    _, _, _, tq3, tsz3 = _tiled_wb(sd, w, 3)
    _, _, _, tq4, tsz4 = _tiled_w4(sd, w)
    xb = synth.activations(M, K, seed=81)
    qx, sx = _a4(sd, xb)
    first3 = first4 = None
    for _ in range(4):
        o3 = bf16_bits(_wb_run(sd, xb, tq3, tsz3, 3, M, N, K))
        o4 = bf16_out(M, N)
        sd.sd_w4a4_linear_tiled(qx, sx, tq4, tsz4, 128, M, N, K, o4)
        torch.cuda.synchronize()
        o4 = bf16_bits(o4)
        if first3 is None:
            first3, first4 = o3, o4
        assert np.array_equal(o3, first3) and np.array_equal(o4, first4)
