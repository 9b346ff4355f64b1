"""GPU tests of two properties every kernel of libsd.so relies on.

1. Bounded device waits: a wait on an mbarrier that nothing arrives on, run
   with the bounded wait routine of the tensor-core W4A16 pipelines and a short
   limit, gives up, records SD_ERR_TIMEOUT (read by sd_device_error) and
   returns; the context stays usable for the next call.
2. Programmatic dependent launch: linears launched back to back on one stream,
   each reading the previous one's output with no host synchronisation in
   between, read x only after the previous kernel has finished (layer i's
   output is the oracle's linear of what layer i - 1 actually wrote; the
   buffers start as NaN)."""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_gb300 import synth
from tests.gpu_helpers import assert_close, bf16_bits, bf16_out, bf16_to_np64, dev, pack_w4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sd():
    from quantized_speculative_decoding_gb300 import build
    build.build()
    from quantized_speculative_decoding_gb300 import binding
    return binding


def test_bounded_wait_runs_out(sd):
    assert sd.sd_device_error() == 0
    sd.sd_test_wait_expiry(2_000_000)  # about 1 ms at the SM clock
    assert sd.sd_device_error() == sd.SD_ERR_TIMEOUT
    assert sd.sd_device_error() == 0  # read and cleared
    # the next calls run normally
    N, K, M = 300, 1024, 5
    qw, s, z = pack_w4(sd, synth.weights(N, K, 77))
    x = synth.activations(M, K, seed=78)
    out = bf16_out(M, N)
    sd.sd_w4a16_linear(dev(x), dev(qw), dev(s), dev(z), 128, M, N, K, out)
    torch.cuda.synchronize()
    assert_close(bf16_to_np64(out), oracle.w4a16_linear(x, qw, s, z, 128, N, K), "after expiry")
    assert sd.sd_device_error() == 0


def _tile(sd, qw, s, z, N, K):
    qb, sb = sd.sd_w4_tiled_bytes(N, K, 128)
    tq = torch.zeros(qb, dtype=torch.uint8, device="cuda")
    tsz = torch.zeros(sb // 2, dtype=torch.int16, device="cuda")
    sd.sd_w4_tile(dev(qw), dev(s), dev(z), 128, N, K, tq, tsz)
    torch.cuda.synchronize()  # weights are read before the kernels' dependency wait
    return tq, tsz


@pytest.mark.parametrize("layout", ["tiled", "rowmajor"])
@pytest.mark.parametrize("M", [1, 5, 40])
def test_chain_reads_previous_output(sd, layout, M):
    dims = [1024, 2048, 512, 3584, 1536, 1024]  # K of layer i = N of layer i - 1
    layers = []
    for i in range(len(dims) - 1):
        K, N = dims[i], dims[i + 1]
        w = synth.weights(N, K, 500 + i) * np.float32(1.0 / np.sqrt(K * 0.02 ** 2))  # keeps |x| near 1
        qw, s, z = pack_w4(sd, w.astype(np.float32))
        dq = _tile(sd, qw, s, z, N, K) if layout == "tiled" else (dev(qw), dev(s), dev(z))
        layers.append((K, N, qw, s, z, dq))
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    for rep in range(3):
        x0 = synth.activations(M, dims[0], seed=600 + rep)
        bufs = [dev(x0)] + [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
                            for (_, N, *_r) in layers]
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for i, (K, N, qw, s, z, dq) in enumerate(layers):
                if layout == "tiled":
                    sd.sd_w4a16_linear_tiled(bufs[i], dq[0], dq[1], 128, M, N, K, bufs[i + 1], stream)
                else:
                    sd.sd_w4a16_linear(bufs[i], dq[0], dq[1], dq[2], 128, M, N, K, bufs[i + 1], stream)
        stream.synchronize()
        assert sd.sd_device_error(stream) == 0
        xin = x0
        for i, (K, N, qw, s, z, dq) in enumerate(layers):
            y = bf16_to_np64(bufs[i + 1])
            assert_close(y, oracle.w4a16_linear(xin, qw, s, z, 128, N, K), f"{layout} chain layer {i} rep {rep}")
            xin = bf16_bits(bufs[i + 1])
