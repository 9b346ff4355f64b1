"""GPU parity of the linear layers (sd_w4a16_linear, sd_w8a16_linear,
sd_bf16_linear, sd_w4_unpack) against the fp64 CPU oracle, through the C ABI.

Bars: unpack and one-hot probes bit-exact; everything else max-abs error
<= 1e-2 * max|ref|.  Full-size workload shapes are checked on sampled output
rows the oracle computes one by one."""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_gb300 import synth
from tests.gpu_helpers import (assert_close, bf16_bits, bf16_out, bf16_to_np64, dev, pack_w4)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sd():
    from quantized_speculative_decoding_gb300 import build
    build.build()
    from quantized_speculative_decoding_gb300 import binding
    return binding


def _linear(sd, path, *args):
    """sd_w4a16_linear, or its test hook with the kernel family forced."""
    if path is None:
        sd.sd_w4a16_linear(*args)
    else:
        sd.sd_test_w4a16_linear_path(*args, path)


def _w4_case(sd, M, N, K, seed, rows=None, path=None):
    w = synth.weights(N, K, seed)
    qw, s, z = pack_w4(sd, w)
    x = synth.activations(M, K, seed=seed + 1)
    out = bf16_out(M, N)
    _linear(sd, path, dev(x), dev(qw), dev(s), dev(z), 128, M, N, K, out)
    torch.cuda.synchronize()
    y = bf16_to_np64(out)
    if rows is None:
        ref = oracle.w4a16_linear(x, qw, s, z, 128, N, K)
        return assert_close(y, ref, f"W4 M={M} N={N} K={K}")
    ref = oracle.w4a16_linear(x, qw[rows], s[rows], z[rows], 128, len(rows), K)
    return assert_close(y[:, rows], ref, f"W4 M={M} N={N} K={K} sampled")


def test_w4_unpack_bit_exact(sd):
    rng = np.random.default_rng(0)
    N, K = 37, 1024
    qw = rng.integers(0, 2 ** 32, (N, K // 8), dtype=np.uint64).astype(np.uint32)
    q = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    sd.sd_w4_unpack(dev(qw), N, K, q)
    assert np.array_equal(q.cpu().numpy(), oracle.unpack_w4(qw, N, K))


def test_w4a16_tiny_workload(sd):
    wl = synth.WORKLOADS["tiny"]
    _, K, N = wl["layer"][0]
    _w4_case(sd, wl["M"], N, K, synth.weight_seed(0, 0, 0))


CUDA_CORE, TENSOR_CORE, MMA = 1, 2, 3  # kernel families of sd_test_w4a16_linear_path


@pytest.fixture(params=[CUDA_CORE, TENSOR_CORE], ids=["cuda_core", "tensor_core"])
def w4_path(request):
    """Run a test through the CUDA-core GEMV and through the tcgen05 kernels."""
    return request.param


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("N,K", [(300, 1024), (129, 128), (64, 3584)])
def test_w4a16_small_m(sd, w4_path, M, N, K):
    _w4_case(sd, M, N, K, seed=100 * M + N, path=w4_path)


@pytest.mark.parametrize("M", [1, 5, 8])
def test_w4a16_small_m_one_hot(sd, w4_path, M):
    N, K = 136, 512
    w = synth.weights(N, K, 23 + M)
    qw, s, z = pack_w4(sd, w)
    ks = [0, 5, 127, 128, 300, 511, 64, 77][:M]
    x = np.zeros((M, K), np.float32)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    out = bf16_out(M, N)
    _linear(sd, w4_path, dev(synth.to_bf16_bits(x)), dev(qw), dev(s), dev(z), 128, M, N, K, out)
    torch.cuda.synchronize()
    wq = oracle.dequant_w4(oracle.unpack_w4(qw, N, K), s, z, 128)
    assert np.array_equal(bf16_bits(out), oracle.round_bf16(wq[:, ks].T.copy()))


@pytest.mark.parametrize("M", [9, 16, 40, 80, 160, 256, 300])
def test_w4a16_batched_m(sd, M):
    _w4_case(sd, M, 520, 1024, seed=M)


@pytest.mark.parametrize("M", [1, 3, 5, 8, 16, 17, 31, 32, 33])
@pytest.mark.parametrize("N,K", [(300, 1024), (128, 128), (1000, 3584), (77, 18944)])
def test_w4a16_tc_path_all_m(sd, M, N, K):
    _w4_case(sd, M, N, K, seed=7 * M + N, path=TENSOR_CORE)


def test_w4a16_tc_one_hot_probes_bit_exact(sd):
    test_w4a16_one_hot_probes_bit_exact(sd, path=TENSOR_CORE)


@pytest.mark.parametrize("name,K,N", synth.QWEN7B_LAYER)
def test_w4a16_tc_qwen7b_shapes_m5(sd, name, K, N):
    rows = np.unique(np.concatenate([SAMPLE[SAMPLE < N], [N - 2, N - 1]]))
    _w4_case(sd, 5, N, K, synth.weight_seed(1, 0, 0), rows=rows, path=TENSOR_CORE)


def test_w4a16_one_hot_probes_bit_exact(sd, path=None):
    N, K = 200, 1024
    w = synth.weights(N, K, 21)
    qw, s, z = pack_w4(sd, w)
    ks = [0, 1, 127, 128, 129, 513, 1016, 1023]
    x = np.zeros((len(ks), K), np.float32)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    xb = synth.to_bf16_bits(x)
    out = bf16_out(len(ks), N)
    _linear(sd, path, dev(xb), dev(qw), dev(s), dev(z), 128, len(ks), N, K, out)
    torch.cuda.synchronize()
    q = oracle.unpack_w4(qw, N, K)
    wq = oracle.dequant_w4(q, s, z, 128)
    expect = oracle.round_bf16(wq[:, ks].T.copy())
    assert np.array_equal(bf16_bits(out), expect)


def test_w4a16_constant_probe(sd):
    # x = 1: the outputs are the row sums of W'
    N, K = 96, 2048
    w = synth.weights(N, K, 22)
    qw, s, z = pack_w4(sd, w)
    xb = synth.to_bf16_bits(np.ones((1, K), np.float32))
    out = bf16_out(1, N)
    sd.sd_w4a16_linear(dev(xb), dev(qw), dev(s), dev(z), 128, 1, N, K, out)
    torch.cuda.synchronize()
    wq = oracle.dequant_w4(oracle.unpack_w4(qw, N, K), s, z, 128)
    assert_close(bf16_to_np64(out)[0], wq.sum(1), "row sums")


SAMPLE = np.array([0, 1, 2, 63, 64, 127, 255, 256, 511, 1000, 1023])


@pytest.mark.parametrize("name,K,N", synth.QWEN7B_LAYER)
def test_w4a16_qwen7b_shapes_m5(sd, name, K, N):
    rows = np.unique(np.concatenate([SAMPLE[SAMPLE < N], [N - 2, N - 1]]))
    _w4_case(sd, 5, N, K, synth.weight_seed(1, 0, 0), rows=rows)


# ---- the register-operand mma.sync kernel reading the row-major layout
@pytest.mark.parametrize("M", [1, 2, 5, 8, 9, 16, 17, 24, 25, 32])
@pytest.mark.parametrize("N,K", [(300, 1024), (129, 256), (64, 3584), (1000, 18944)])
def test_w4a16_rowmajor_mma(sd, M, N, K):
    rows = None if N * K <= 300 * 3584 else np.unique(np.concatenate([SAMPLE, [N - 1]]))
    _w4_case(sd, M, N, K, seed=31 * M + N, rows=rows, path=MMA)


def test_w4a16_rowmajor_mma_one_hot_probes_bit_exact(sd):
    test_w4a16_one_hot_probes_bit_exact(sd, path=MMA)


@pytest.mark.parametrize("name,K,N", synth.QWEN7B_LAYER)
def test_w4a16_rowmajor_mma_qwen7b_m5(sd, name, K, N):
    rows = np.unique(np.concatenate([SAMPLE[SAMPLE < N], [N - 2, N - 1]]))
    _w4_case(sd, 5, N, K, synth.weight_seed(1, 0, 1), rows=rows, path=MMA)


@pytest.mark.parametrize("name,K,N", synth.QWEN1P5B_LAYER)
def test_w4a16_rowmajor_mma_qwen1p5b_m1(sd, name, K, N):
    rows = np.unique(np.concatenate([SAMPLE[SAMPLE < N], [N - 1]]))
    _w4_case(sd, 1, N, K, synth.weight_seed(2, 0, 1), rows=rows, path=MMA)


def test_w4a16_auto_path_takes_the_rowmajor_mma_kernel(sd):
    # sd_w4a16_linear at M <= 32 with K % 256 == 0 is the mma kernel, bit for bit
    M, N, K = 5, 700, 3584
    w = synth.weights(N, K, 91)
    qw, s, z = pack_w4(sd, w)
    x = dev(synth.activations(M, K, seed=92))
    outs = []
    for path in (None, MMA):
        out = bf16_out(M, N)
        _linear(sd, path, x, dev(qw), dev(s), dev(z), 128, M, N, K, out)
        torch.cuda.synchronize()
        outs.append(bf16_bits(out))
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("M,K", [(1, 384), (5, 640), (5, 128)])
def test_w4a16_auto_path_with_an_odd_group_count(sd, M, K):
    # K / 128 odd: the mma kernel's scale pairs do not apply; the other kernels serve
    _w4_case(sd, M, 260, K, seed=93 + K)


def test_w4a16_rowmajor_mma_repeated_launches_bit_identical(sd):
    M, N, K = 5, 3584, 18944
    w = synth.weights(N, K, 94)
    qw, s, z = pack_w4(sd, w)
    args = (dev(synth.activations(M, K, seed=95)), dev(qw), dev(s), dev(z), 128, M, N, K)
    first = None
    for _ in range(5):
        out = bf16_out(M, N)
        _linear(sd, MMA, *args, out)
        torch.cuda.synchronize()
        if first is None:
            first = bf16_bits(out)
        assert np.array_equal(bf16_bits(out), first)


@pytest.mark.parametrize("name,K,N,M", [("gate", 4096, 11008, 40), ("gate", 4096, 11008, 80),
                                         ("o", 4096, 4096, 40), ("o", 4096, 4096, 160)])
def test_w4a16_llama7b_batched_split_counts(sd, name, K, N, M):
    # the K-split (cluster) counts the batched kernel picks for these shapes:
    # gate at M = 40 splits K in 3, o in 4, gate at M = 80 not at all
    rows = np.unique(np.concatenate([SAMPLE, [N - 1]]))
    _w4_case(sd, M, N, K, synth.weight_seed(3, 0, 4 if name == "gate" else 3), rows=rows)


@pytest.mark.parametrize("M", [40, 160])
def test_w4a16_llama7b_down_batched(sd, M):
    K, N = 11008, 4096
    rows = np.unique(np.concatenate([SAMPLE, [N - 1]]))
    _w4_case(sd, M, N, K, synth.weight_seed(3, 0, 6), rows=rows)


@pytest.mark.parametrize("M,N,K", [(1, 300, 1024), (5, 257, 512), (8, 64, 4096)])
def test_w8a16_parity(sd, M, N, K):
    w = synth.weights(N, K, 31 + M)
    q8 = np.zeros((N, K), np.int8)
    s = np.zeros((N,), np.uint16)
    sd.sd_w8_pack(w, N, K, q8, s)
    x = synth.activations(M, K, 5)
    out = bf16_out(M, N)
    sd.sd_w8a16_linear(dev(x), dev(q8), dev(s), M, N, K, out)
    torch.cuda.synchronize()
    assert_close(bf16_to_np64(out), oracle.w8a16_linear(x, q8, s), "W8")


@pytest.mark.parametrize("M,N,K", [(1, 300, 1024), (5, 257, 520), (8, 64, 4096)])
def test_bf16_parity(sd, M, N, K):
    w = synth.to_bf16_bits(synth.weights(N, K, 41 + M))
    x = synth.activations(M, K, 6)
    out = bf16_out(M, N)
    sd.sd_bf16_linear(dev(x), dev(w), M, N, K, out)
    torch.cuda.synchronize()
    assert_close(bf16_to_np64(out), oracle.bf16_linear(x, w), "bf16")


@pytest.mark.parametrize("name,K,N", synth.QWEN1P5B_LAYER[4:])
def test_draft_precisions_qwen1p5b_m1(sd, name, K, N):
    w = synth.weights(N, K, synth.weight_seed(2, 0, 4))
    x = synth.activations(1, K)
    rows = np.unique(np.concatenate([SAMPLE[SAMPLE < N], [N - 1]]))
    # INT4
    qw, s, z = pack_w4(sd, w)
    out = bf16_out(1, N)
    sd.sd_w4a16_linear(dev(x), dev(qw), dev(s), dev(z), 128, 1, N, K, out)
    # INT8
    q8 = np.zeros((N, K), np.int8)
    s8 = np.zeros((N,), np.uint16)
    sd.sd_w8_pack(w, N, K, q8, s8)
    out8 = bf16_out(1, N)
    sd.sd_w8a16_linear(dev(x), dev(q8), dev(s8), 1, N, K, out8)
    # bf16
    wb = synth.to_bf16_bits(w)
    outb = bf16_out(1, N)
    sd.sd_bf16_linear(dev(x), dev(wb), 1, N, K, outb)
    torch.cuda.synchronize()
    assert_close(bf16_to_np64(out)[:, rows],
                 oracle.w4a16_linear(x, qw[rows], s[rows], z[rows], 128, len(rows), K), "W4")
    assert_close(bf16_to_np64(out8)[:, rows], oracle.w8a16_linear(x, q8[rows], s8[rows]), "W8")
    assert_close(bf16_to_np64(outb)[:, rows], oracle.bf16_linear(x, wb[rows]), "bf16")


def test_linear_is_deterministic(sd):
    N, K, M = 4096, 3584, 5
    w = synth.weights(N, K, 51)
    qw, s, z = (dev(a) for a in pack_w4(sd, w))
    x = dev(synth.activations(M, K))
    outs = []
    for _ in range(3):
        out = bf16_out(M, N)
        sd.sd_w4a16_linear(x, qw, s, z, 128, M, N, K, out)
        outs.append(bf16_bits(out))
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


@pytest.mark.parametrize("layout,M,N,K", [
    ("rowmajor", 160, 4096, 11008),   # batched tcgen05, K split in clusters
    ("rowmajor", 40, 4096, 11008),
    ("rowmajor", 160, 11008, 4096),
    ("tiled", 5, 3584, 18944),        # mma.sync, clusters of 12
    ("tiled", 5, 37888, 3584),        # mma.sync, clusters of 3, a near-full wave
])
def test_repeated_launches_are_bit_identical(sd, layout, M, N, K):
    """Several launches of one configuration give the same bits (the K-split
    reductions add in a fixed order) and the oracle's values: a race between
    a kernel's pipeline stages shows up here as launch-to-launch differences."""
    w = synth.weights(N, K, 71 + M)
    qw, s, z = pack_w4(sd, w)
    x = synth.activations(M, K, seed=72)
    dx = dev(x)
    if layout == "tiled":
        tq, tsz = _tile_on_gpu(sd, qw, s, z, N, K)
        call = lambda out: sd.sd_w4a16_linear_tiled(dx, tq, tsz, 128, M, N, K, out)
    else:
        dq, ds, dz = dev(qw), dev(s), dev(z)
        torch.cuda.synchronize()
        call = lambda out: sd.sd_w4a16_linear(dx, dq, ds, dz, 128, M, N, K, out)
    outs = []
    for _ in range(6):
        out = bf16_out(M, N)
        call(out)
        torch.cuda.synchronize()
        outs.append(bf16_bits(out))
    assert sd.sd_device_error() == 0
    for i, o in enumerate(outs[1:], 1):
        bad = np.argwhere(o != outs[0])
        assert bad.size == 0, f"launch {i} differs from launch 0 at {len(bad)} outputs, first {bad[0]}"
    rows = np.unique(np.concatenate([SAMPLE[SAMPLE < N], [N - 1]]))
    y = outs[0].view(np.uint16).astype(np.uint32) << 16
    y = y.view(np.float32).astype(np.float64)
    assert_close(y[:, rows], oracle.w4a16_linear(x, qw[rows], s[rows], z[rows], 128, len(rows), K), "repeat")


# ------------------------------------------------------------ tiled layout
def _tiled_reference(qw, s, z, N, K):
    """The fragment-ordered tiled layout from its definition in sd.h (numpy)."""
    T, G, KC = (N + 15) // 16, K // 128, K // 64
    q = np.zeros((T * 16, K), np.uint32)
    q[:N] = oracle.unpack_w4(qw, N, K)
    # k = 64 j + 16 c + 4 s + e
    Q = q.reshape(T, 16, KC, 4, 4, 4)
    Qg, Qh = Q[:, :8], Q[:, 8:]
    word = (Qg[..., 0] | Qh[..., 0] << 4 | Qg[..., 2] << 8 | Qh[..., 2] << 12 |
            Qg[..., 1] << 16 | Qh[..., 1] << 20 | Qg[..., 3] << 24 | Qh[..., 3] << 28)
    # (T, g, j, c, s) -> units [T][j][l = 4 g + c][s]
    tq = np.ascontiguousarray(word.transpose(0, 2, 1, 3, 4)).astype(np.uint32).view(np.uint8)
    sp = np.zeros((T * 16, G), np.uint16)
    zp = np.full((T * 16, G), 0x4300, np.uint16)
    sp[:N] = s
    zp[:N] = 0x4300 + z.view(np.float16).astype(np.float64).astype(np.uint16)  # bf16 128 + z
    sp, zp = sp.reshape(T, 16, G), zp.reshape(T, 16, G)
    ent = np.stack([sp[:, :8], zp[:, :8], sp[:, 8:], zp[:, 8:]], axis=-1)  # (T, g, G, 4)
    tsz = np.ascontiguousarray(ent.transpose(0, 2, 1, 3))               # [T][G][8][4]
    return tq.reshape(-1), tsz.reshape(-1)


def _tile_on_gpu(sd, qw, s, z, N, K):
    qb, sb = sd.sd_w4_tiled_bytes(N, K, 128)
    tq = torch.zeros(qb, dtype=torch.uint8, device="cuda")
    tsz = torch.zeros(sb // 2, dtype=torch.int16, device="cuda")
    sd.sd_w4_tile(dev(qw), dev(s), dev(z), 128, N, K, tq, tsz)
    torch.cuda.synchronize()  # the tiled copy is read before the next kernel's dependency wait
    return tq, tsz


@pytest.mark.parametrize("N,K", [(128, 128), (300, 1024), (77, 3584), (16, 256)])
def test_w4_tile_layout_bit_exact(sd, N, K):
    w = synth.weights(N, K, 61)
    qw, s, z = pack_w4(sd, w)
    tq, tsz = _tile_on_gpu(sd, qw, s, z, N, K)
    rq, rsz = _tiled_reference(qw, s, z, N, K)
    assert sd.sd_w4_tiled_bytes(N, K, 128) == (rq.size, rsz.size * 2)
    assert np.array_equal(tq.cpu().numpy(), rq)
    assert np.array_equal(tsz.cpu().numpy().view(np.uint16), rsz)
    assert sd.sd_device_error() == 0


def test_w4_tile_rejects_fractional_zero(sd):
    N, K = 32, 256
    qw, s, z = pack_w4(sd, synth.weights(N, K, 62))
    z = z.copy()
    z[5, 1] = 0x3C00 + 0x200  # fp16 1.5
    _tile_on_gpu(sd, qw, s, z, N, K)
    assert sd.sd_device_error() == sd.SD_ERR_INVALID_ARG  # then cleared
    assert sd.sd_device_error() == 0


def _tiled_case(sd, M, N, K, seed, rows=None):
    w = synth.weights(N, K, seed)
    qw, s, z = pack_w4(sd, w)
    tq, tsz = _tile_on_gpu(sd, qw, s, z, N, K)
    x = synth.activations(M, K, seed=seed + 1)
    out = bf16_out(M, N)
    sd.sd_w4a16_linear_tiled(dev(x), tq, tsz, 128, M, N, K, out)
    torch.cuda.synchronize()
    y = bf16_to_np64(out)
    if rows is None:
        return assert_close(y, oracle.w4a16_linear(x, qw, s, z, 128, N, K), f"tiled M={M}")
    ref = oracle.w4a16_linear(x, qw[rows], s[rows], z[rows], 128, len(rows), K)
    return assert_close(y[:, rows], ref, f"tiled M={M} sampled")


@pytest.mark.parametrize("M", [1, 2, 5, 8, 16, 17, 32, 33, 40])
@pytest.mark.parametrize("N,K", [(300, 1024), (128, 128), (1000, 3584), (77, 18944)])
def test_w4a16_tiled_parity(sd, M, N, K):
    _tiled_case(sd, M, N, K, seed=11 * M + N)


@pytest.mark.parametrize("name,K,N", synth.QWEN7B_LAYER)
def test_w4a16_tiled_qwen7b_shapes_m5(sd, name, K, N):
    rows = np.unique(np.concatenate([SAMPLE[SAMPLE < N], [N - 2, N - 1]]))
    _tiled_case(sd, 5, N, K, synth.weight_seed(1, 0, 0), rows=rows)


def test_w4a16_tiled_one_hot_bit_exact(sd):
    N, K = 200, 1024
    w = synth.weights(N, K, 21)
    qw, s, z = pack_w4(sd, w)
    tq, tsz = _tile_on_gpu(sd, qw, s, z, N, K)
    ks = [0, 1, 127, 128, 129, 513, 1016, 1023]
    x = np.zeros((len(ks), K), np.float32)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    out = bf16_out(len(ks), N)
    sd.sd_w4a16_linear_tiled(dev(synth.to_bf16_bits(x)), tq, tsz, 128, len(ks), N, K, out)
    torch.cuda.synchronize()
    wq = oracle.dequant_w4(oracle.unpack_w4(qw, N, K), s, z, 128)
    assert np.array_equal(bf16_bits(out), oracle.round_bf16(wq[:, ks].T.copy()))

