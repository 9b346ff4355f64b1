"""Host-side tests of libsd.so: the library loads and exports every function
include/sd.h declares; the CPU packers match the oracle's quantisers bit for
bit; argument checks and injected faults return their status codes without
launching anything (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_decoding_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sd():
    from quantized_speculative_decoding_gb300 import build
    build.build()
    from quantized_speculative_decoding_gb300 import binding
    return binding


def _declared():
    src = open(os.path.join(ROOT, "include", "sd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sd_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(sd):
    names = _declared()
    assert len(names) >= 11
    assert set(names) == set(sd.EXPORTS)
    lib = ctypes.CDLL(sd.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(sd):
    assert sd.status_string(0) == "SD_OK"
    assert sd.status_string(1) == "SD_ERR_INVALID_ARG"
    assert sd.status_string(99) == "SD_ERR_UNKNOWN"
    assert sd.sd_version() >> 16 == 1


def _pack_words(q):
    N, K = q.shape
    q = q.astype(np.uint32).reshape(N, K // 8, 8)
    return np.bitwise_or.reduce(q << (4 * np.arange(8, dtype=np.uint32)), axis=2).astype(np.uint32)


@pytest.mark.parametrize("N,K,scale", [(64, 512, 0.02), (3, 1024, 1.0), (17, 128, 1e-4),
                                       (5, 384, 300.0)])
def test_w4_pack_matches_oracle(sd, N, K, scale):
    rng = np.random.default_rng(N + K)
    w = (rng.standard_normal((N, K)) * scale).astype(np.float32)
    w[0, :128] = 0.0
    w[-1, -128:] = np.abs(w[-1, -128:])
    w[1 % N, 5] = 0.0
    qw = np.zeros((N, K // 8), np.uint32)
    s = np.zeros((N, K // 128), np.uint16)
    z = np.zeros((N, K // 128), np.uint16)
    sd.sd_w4_pack(w, N, K, 128, qw, s, z)
    q, s_ref, z_ref = oracle.quantize_w4(w, 128)
    assert np.array_equal(qw, _pack_words(q))
    assert np.array_equal(s, s_ref)
    assert np.array_equal(z, z_ref)


def test_w4_pack_on_workload_weights(sd):
    w = synth.weights(256, 3584, synth.weight_seed(1, 0, 0))
    qw = np.zeros((256, 448), np.uint32)
    s = np.zeros((256, 28), np.uint16)
    z = np.zeros((256, 28), np.uint16)
    sd.sd_w4_pack(w, 256, 3584, 128, qw, s, z)
    q, s_ref, z_ref = oracle.quantize_w4(w, 128)
    assert np.array_equal(qw, _pack_words(q))
    assert np.array_equal(s, s_ref) and np.array_equal(z, z_ref)


@pytest.mark.parametrize("N,K,scale", [(40, 160, 0.02), (2, 16, 5e3), (9, 4096, 1e-3)])
def test_w8_pack_matches_oracle(sd, N, K, scale):
    rng = np.random.default_rng(N * K)
    w = (rng.standard_normal((N, K)) * scale).astype(np.float32)
    w[0] = 0.0
    q8 = np.zeros((N, K), np.int8)
    s = np.zeros((N,), np.uint16)
    sd.sd_w8_pack(w, N, K, q8, s)
    q_ref, s_ref = oracle.quantize_w8(w)
    assert np.array_equal(q8, q_ref)
    assert np.array_equal(s, s_ref)


@pytest.mark.parametrize("bits,N,K", [(2, 7, 128), (3, 5, 384), (3, 64, 3584), (4, 9, 256), (2, 33, 1536)])
def test_wb_pack_matches_oracle(sd, bits, N, K):
    w = synth.weights(N, K, 7 * bits + N)
    w[0, :128] = 0.0          # an all-zero group
    w[1, 5] = 0.3             # an outlier group
    packed = np.zeros((N, K * bits // 32), np.uint32)
    s = np.zeros((N, K // 128), np.uint16)
    z = np.zeros((N, K // 128), np.uint16)
    sd.sd_wb_pack(w, N, K, 128, bits, packed, s, z)
    q_o, s_o, z_o = oracle.quantize_wb(w, bits)
    assert np.array_equal(packed, oracle.pack_wb(q_o, bits))
    assert np.array_equal(s, s_o) and np.array_equal(z, z_o)
    if bits == 4:  # the INT4 packer's layout
        qw = np.zeros((N, K // 8), np.uint32)
        sd.sd_w4_pack(w, N, K, 128, qw, s, z)
        assert np.array_equal(packed, qw)


def test_wb_pack_rejects_bad_input(sd):
    w = np.zeros((2, 128), np.float32)
    buf = np.zeros(64, np.uint32)
    s = np.zeros(8, np.uint16)
    L = sd.lib

    def call(w=w.ctypes.data, N=2, K=128, group=128, bits=3, packed=buf.ctypes.data):
        return L.sd_wb_pack(w, N, K, group, bits, packed, s.ctypes.data, s.ctypes.data)

    assert call(w=None) == sd.SD_ERR_INVALID_ARG
    assert call(packed=None) == sd.SD_ERR_INVALID_ARG
    assert call(N=0) == sd.SD_ERR_INVALID_ARG
    assert call(group=96) == sd.SD_ERR_INVALID_ARG     # K % group != 0
    assert call(bits=1) == sd.SD_ERR_UNSUPPORTED
    assert call(bits=5) == sd.SD_ERR_UNSUPPORTED
    w40 = np.zeros((1, 40), np.float32)
    assert call(w=w40.ctypes.data, N=1, K=40, group=40) == sd.SD_ERR_INVALID_ARG  # 120 bits: no whole word
    bad = w.copy()
    bad[1, 3] = np.inf
    assert call(w=bad.ctypes.data) == sd.SD_ERR_INVALID_ARG
    assert call() == sd.SD_OK


def test_packers_reject_bad_input(sd):
    w = np.zeros((4, 256), np.float32)
    qw = np.zeros((4, 32), np.uint32)
    s = np.zeros((4, 2), np.uint16)
    z = np.zeros((4, 2), np.uint16)
    st = sd.lib.sd_w4_pack
    assert st(None, 4, 256, 128, qw.ctypes.data, s.ctypes.data, z.ctypes.data) == sd.SD_ERR_INVALID_ARG
    assert st(w.ctypes.data, 4, 260, 128, qw.ctypes.data, s.ctypes.data, z.ctypes.data) == sd.SD_ERR_INVALID_ARG
    assert st(w.ctypes.data, 0, 256, 128, qw.ctypes.data, s.ctypes.data, z.ctypes.data) == sd.SD_ERR_INVALID_ARG
    w[2, 3] = np.inf
    assert st(w.ctypes.data, 4, 256, 128, qw.ctypes.data, s.ctypes.data, z.ctypes.data) == sd.SD_ERR_INVALID_ARG
    big = np.full((1, 128), 1e9, np.float32)  # scale 1e9/15 overflows fp16
    assert st(big.ctypes.data, 1, 128, 128, qw.ctypes.data, s.ctypes.data, z.ctypes.data) == sd.SD_ERR_INVALID_ARG
    q8 = np.zeros((1, 128), np.int8)
    s8 = np.zeros(1, np.uint16)
    assert sd.lib.sd_w8_pack(big.ctypes.data, 1, 128, q8.ctypes.data, s8.ctypes.data) == sd.SD_ERR_INVALID_ARG


# Fake device addresses: argument checks run before anything touches them.
A = 1 << 20


def test_linear_argument_checks(sd):
    L = sd.lib
    E = sd.SD_ERR_INVALID_ARG
    assert L.sd_w4a16_linear(None, A, A, A, 128, 5, 64, 512, A, None) == E
    assert L.sd_w4a16_linear(A, A, A, A, 128, 0, 64, 512, A, None) == E
    assert L.sd_w4a16_linear(A, A, A, A, 128, 5, 64, 500, A, None) == E      # K % 8
    assert L.sd_w4a16_linear(A, A, A, A, 128, 5, 64, 520, A, None) == E      # K % group
    assert L.sd_w4a16_linear(A + 8, A, A, A, 128, 5, 64, 512, A, None) == E  # x alignment
    assert L.sd_w4a16_linear(A, A + 4, A, A, 128, 5, 64, 512, A, None) == E  # qweight alignment
    assert L.sd_w4a16_linear(A, A, A, A, 64, 5, 64, 512, A, None) == sd.SD_ERR_UNSUPPORTED
    assert L.sd_w8a16_linear(A, A, A, 1, 64, 24, A, None) == E               # K % 16
    assert L.sd_bf16_linear(A, A, 1, 64, 12, A, None) == E                   # K % 8
    assert L.sd_bf16_linear(A, A, 1, -1, 16, A, None) == E
    assert L.sd_w4_unpack(A, 4, 12, A, None) == E


def test_tiled_layout_sizes_and_checks(sd):
    # sizes from the layout's definition: 16-byte units [ceil(N/16)][K/64][32],
    # 8-byte scale/zero entries [ceil(N/16)][K/128][8]
    for N, K in [(16, 128), (17, 128), (18944, 3584), (3584, 18944), (1, 256)]:
        T = (N + 15) // 16
        assert sd.sd_w4_tiled_bytes(N, K, 128) == (T * (K // 64) * 32 * 16, T * (K // 128) * 8 * 8)
    L = sd.lib
    E = sd.SD_ERR_INVALID_ARG
    q, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert L.sd_w4_tiled_bytes(0, 128, 128, ctypes.byref(q), ctypes.byref(b)) == E
    assert L.sd_w4_tiled_bytes(16, 200, 128, ctypes.byref(q), ctypes.byref(b)) == E
    assert L.sd_w4_tiled_bytes(16, 128, 128, None, ctypes.byref(b)) == E
    assert L.sd_w4_tiled_bytes(16, 256, 64, ctypes.byref(q), ctypes.byref(b)) == sd.SD_ERR_UNSUPPORTED
    assert L.sd_w4_tile(None, A, A, 128, 16, 128, A, A, None) == E
    assert L.sd_w4_tile(A, A, A, 128, 16, 128, A + 8, A, None) == E          # tiled_qweight alignment
    assert L.sd_w4_tile(A, A, A, 128, 16, 128, A, A + 4, None) == E          # tiled_sz alignment
    assert L.sd_w4_tile(A, A, A, 128, 16, 128, A, A + 8, None) == E          # tiled_sz alignment (16)
    assert L.sd_w4_tile(A, A, A, 64, 16, 128, A, A, None) == sd.SD_ERR_UNSUPPORTED
    assert L.sd_w4a16_linear_tiled(A, A, A, 128, 0, 16, 128, A, None) == E
    assert L.sd_w4a16_linear_tiled(A + 4, A, A, 128, 5, 16, 128, A, None) == E  # x alignment
    assert L.sd_w4a16_linear_tiled(A, A, A + 4, 128, 5, 16, 128, A, None) == E  # tiled_sz alignment
    assert L.sd_w4a16_linear_tiled(A, A, A + 8, 128, 5, 16, 128, A, None) == E  # tiled_sz alignment (16)
    assert L.sd_w4a16_linear_tiled(A, A, A, 128, 5, 16, 200, A, None) == E
    assert L.sd_w4a16_linear_tiled(A, A, A, 64, 5, 16, 256, A, None) == sd.SD_ERR_UNSUPPORTED


def test_lowbit_layout_sizes_and_checks(sd):
    # b-bit tiled sizes from the layout's definition: b x 256 bytes per
    # (16-row tile, 128-input group); the scale/zero entries as for INT4
    for N, K in [(16, 128), (17, 256), (18944, 3584), (1, 384)]:
        T = (N + 15) // 16
        for bits in (2, 3):
            assert sd.sd_wb_tiled_bytes(N, K, bits) == (T * (K // 128) * bits * 256, T * (K // 128) * 64)
        assert sd.sd_wb_tiled_bytes(N, K, 4) == sd.sd_w4_tiled_bytes(N, K)
    L = sd.lib
    E = sd.SD_ERR_INVALID_ARG
    q, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert L.sd_wb_tiled_bytes(16, 128, 128, 1, ctypes.byref(q), ctypes.byref(b)) == E
    assert L.sd_wb_tiled_bytes(16, 128, 128, 5, ctypes.byref(q), ctypes.byref(b)) == E
    assert L.sd_wb_tiled_bytes(16, 256, 64, 2, ctypes.byref(q), ctypes.byref(b)) == sd.SD_ERR_UNSUPPORTED
    assert L.sd_wb_tile(None, A, A, 128, 2, 16, 128, A, A, None) == E
    assert L.sd_wb_tile(A, A, A, 128, 5, 16, 128, A, A, None) == E
    assert L.sd_wb_tile(A + 2, A, A, 128, 3, 16, 128, A, A, None) == E       # packed alignment
    assert L.sd_wb_tile(A, A, A, 128, 3, 16, 128, A + 8, A, None) == E       # tiled_qweight alignment
    assert L.sd_wb_linear_tiled(A, A, A, 128, 2, 0, 16, 128, A, None) == E
    assert L.sd_wb_linear_tiled(A, A, A, 128, 1, 5, 16, 128, A, None) == E
    assert L.sd_wb_linear_tiled(A + 4, A, A, 128, 3, 5, 16, 128, A, None) == E  # x alignment
    assert L.sd_wb_linear_tiled(A, A, A, 64, 2, 5, 16, 256, A, None) == sd.SD_ERR_UNSUPPORTED
    assert L.sd_a4_quantize(None, 1, 128, A, A, None) == E
    assert L.sd_a4_quantize(A, 1, 200, A, A, None) == E                       # K % 128
    assert L.sd_a4_quantize(A, 0, 128, A, A, None) == E
    assert L.sd_a4_quantize(A, 1, 128, A + 8, A, None) == E                   # qx alignment
    assert L.sd_w4a4_linear_tiled(A, A, A, A, 128, 0, 16, 128, A, None) == E
    assert L.sd_w4a4_linear_tiled(A, A + 2, A, A, 128, 1, 16, 128, A, None) == E  # sx alignment
    assert L.sd_w4a4_linear_tiled(A, A, A, A, 64, 1, 16, 256, A, None) == sd.SD_ERR_UNSUPPORTED


def test_verify_argument_checks(sd):
    L = sd.lib
    E = sd.SD_ERR_INVALID_ARG
    ok = dict(gamma=4, batch=1, vocab=1024, T=1.0)

    def call(draft=A, target=A, tokens=A, gamma=4, batch=1, vocab=1024, T=1.0, out=A, alen=A):
        return L.sd_verify(draft, target, tokens, gamma, batch, vocab, T, 0, out, alen, None)

    assert ok
    assert call(gamma=0) == E
    assert call(gamma=17) == E
    assert call(batch=-1) == E
    assert call(vocab=0) == E
    assert call(T=-0.5) == E
    assert call(T=float("nan")) == E
    assert call(T=1e-9) == E
    assert call(T=2e6) == E
    assert call(target=None) == E
    assert call(draft=None) == E          # T > 0 needs draft logits
    assert call(tokens=A + 2) == E        # alignment
    assert call(batch=0) == sd.SD_OK      # no-op, nothing launched


def test_sample_argument_checks(sd):
    L = sd.lib
    E = sd.SD_ERR_INVALID_ARG

    def call(logits=A, batch=1, vocab=1024, T=1.0, slot=0, out=A):
        return L.sd_sample(logits, batch, vocab, T, 0, slot, out, None)

    assert call(logits=None) == E
    assert call(out=None) == E
    assert call(batch=-1) == E
    assert call(vocab=0) == E
    assert call(slot=-1) == E
    assert call(slot=(1 << 30) + 1) == E
    assert call(T=-1.0) == E
    assert call(T=float("nan")) == E
    assert call(T=1e-8) == E
    assert call(T=2e6) == E
    assert call(logits=A + 2) == E        # alignment
    assert call(out=A + 1) == E
    assert call(batch=0) == sd.SD_OK      # no-op, nothing launched


def test_lm_head_argument_checks(sd):
    L = sd.lib
    E, U = sd.SD_ERR_INVALID_ARG, sd.SD_ERR_UNSUPPORTED
    n = ctypes.c_int(0)
    assert L.sd_lm_head_parts(5, 1024, 512, None) == E
    for M, V, K in ((0, 1024, 512), (33, 1024, 512), (5, 0, 512), (5, 1024, 64), (5, 1024, 200)):
        assert L.sd_lm_head_parts(M, V, K, ctypes.byref(n)) == E

    def call(x=A, wq=A, wsz=A, group=128, M=5, V=1024, K=512, T=1.0, logits=A, ldl=1024, stats=A, lds=4096):
        return L.sd_w4a16_lm_head(x, wq, wsz, group, M, V, K, T, logits, ldl, stats, lds, None)

    assert call(x=None) == E
    assert call(logits=None) == E
    assert call(stats=None) == E
    assert call(M=0) == E
    assert call(K=500) == E
    assert call(ldl=1023) == E            # rows would overlap
    assert call(T=-1.0) == E
    assert call(T=float("nan")) == E
    assert call(T=1e-8) == E
    assert call(x=A + 8) == E             # alignment
    assert call(logits=A + 2) == E
    assert call(stats=A + 4) == E
    assert call(group=64) == U
    assert call(M=40) == U                # rows of x in one call: at most 32

    def vcall(dl=A, tl=A, ds=A, dp=10, ts=A, tp=10, tok=A, gamma=4, batch=1, V=1024, T=1.0, out=A, ln=A):
        return L.sd_verify_parts(dl, tl, ds, dp, ts, tp, tok, gamma, batch, V, T, 0, out, ln, None)

    assert vcall(ts=None) == E
    assert vcall(tp=0) == E
    assert vcall(ds=None) == E            # read at T > 0
    assert vcall(dp=0) == E
    assert vcall(dl=None) == E
    assert vcall(gamma=0) == E
    assert vcall(gamma=17) == E
    assert vcall(T=-0.5) == E
    assert vcall(ts=A + 4) == E           # pairs are 8-byte aligned
    assert vcall(ds=A + 4) == E
    assert vcall(batch=0) == sd.SD_OK     # no-op
    assert vcall(ds=None, dp=0, dl=None, T=0.0, batch=0) == sd.SD_OK  # greedy reads no draft rows


def test_linear_path_hook_argument_checks(sd):
    x = np.zeros((1, 512), np.uint16)
    E = sd.SD_ERR_INVALID_ARG
    call = lambda path, M=1: sd.lib.sd_test_w4a16_linear_path(x.ctypes.data, A, A, A, 128, M, 64, 512, A,
                                                               path, None)
    assert call(0) == E and call(4) == E and call(-1) == E
    assert call(1, M=9) == sd.SD_ERR_UNSUPPORTED  # the GEMV serves M <= 8
    assert call(3, M=33) == sd.SD_ERR_UNSUPPORTED  # the row-major mma kernel serves M <= 32
    # ... with K % 256 == 0 and 4-byte aligned scales and zero points
    k384 = lambda s_ptr: sd.lib.sd_test_w4a16_linear_path(x.ctypes.data, A, s_ptr, A, 128, 1, 64, 384, A, 3, None)
    assert k384(A) == sd.SD_ERR_UNSUPPORTED
    assert sd.lib.sd_test_w4a16_linear_path(x.ctypes.data, A, A + 2, A, 128, 1, 64, 512, A, 3,
                                            None) == sd.SD_ERR_UNSUPPORTED


def test_wait_expiry_argument_checks(sd):
    assert sd.lib.sd_test_wait_expiry(0, None) == sd.SD_ERR_INVALID_ARG
    assert sd.lib.sd_test_wait_expiry(-5, None) == sd.SD_ERR_INVALID_ARG
    assert sd.lib.sd_test_wait_expiry((1 << 40) + 1, None) == sd.SD_ERR_INVALID_ARG


def test_fault_injection(sd, monkeypatch):
    w = np.zeros((2, 128), np.float32)
    qw = np.zeros((2, 16), np.uint32)
    s = np.zeros((2, 1), np.uint16)
    z = np.zeros((2, 1), np.uint16)
    monkeypatch.setenv("SD_FAULT_INJECT", "sd_verify:3,sd_w4_pack:5")
    assert sd.lib.sd_verify(A, A, A, 4, 1, 8, 1.0, 0, A, A, None) == sd.SD_ERR_CUDA
    assert sd.lib.sd_w4_pack(w.ctypes.data, 2, 128, 128, qw.ctypes.data, s.ctypes.data,
                             z.ctypes.data) == sd.SD_ERR_INTERNAL
    with pytest.raises(sd.SdError) as ei:
        sd.sd_w4_pack(w, 2, 128, 128, qw, s, z)
    assert ei.value.status == sd.SD_ERR_INTERNAL
    monkeypatch.setenv("SD_FAULT_INJECT", "sd_w4a16_linear:4")
    assert sd.lib.sd_w4a16_linear(A, A, A, A, 128, 5, 64, 512, A, None) == sd.SD_ERR_TIMEOUT
    # other functions unaffected
    assert sd.lib.sd_w4_pack(w.ctypes.data, 2, 128, 128, qw.ctypes.data, s.ctypes.data,
                             z.ctypes.data) == sd.SD_OK
    # the lm_head pair, its parts query and the b-bit packer take injected faults too
    monkeypatch.setenv("SD_FAULT_INJECT", "sd_lm_head_parts:3,sd_w4a16_lm_head:4,sd_verify_parts:5,sd_wb_pack:2")
    n = ctypes.c_int(0)
    assert sd.lib.sd_lm_head_parts(5, 1024, 512, ctypes.byref(n)) == sd.SD_ERR_CUDA
    assert sd.lib.sd_w4a16_lm_head(A, A, A, 128, 5, 1024, 512, 1.0, A, 1024, A, 4096, None) == sd.SD_ERR_TIMEOUT
    assert sd.lib.sd_verify_parts(A, A, A, 8, A, 8, A, 4, 1, 1024, 1.0, 0, A, A, None) == sd.SD_ERR_INTERNAL
    assert sd.lib.sd_wb_pack(w.ctypes.data, 2, 128, 128, 3, qw.ctypes.data, s.ctypes.data,
                             z.ctypes.data) == sd.SD_ERR_UNSUPPORTED
    monkeypatch.setenv("SD_FAULT_INJECT", "sd_test_wait_expiry:4")
    assert sd.lib.sd_test_wait_expiry(1000, None) == sd.SD_ERR_TIMEOUT
    monkeypatch.setenv("SD_FAULT_INJECT", "sd_wb_tile:3,sd_wb_linear_tiled:4,sd_a4_quantize:5,sd_w4a4_linear_tiled:3")
    assert sd.lib.sd_wb_tile(A, A, A, 128, 2, 16, 128, A, A, None) == sd.SD_ERR_CUDA
    assert sd.lib.sd_wb_linear_tiled(A, A, A, 128, 2, 5, 16, 128, A, None) == sd.SD_ERR_TIMEOUT
    assert sd.lib.sd_a4_quantize(A, 1, 128, A, A, None) == sd.SD_ERR_INTERNAL
    assert sd.lib.sd_w4a4_linear_tiled(A, A, A, A, 128, 1, 16, 128, A, None) == sd.SD_ERR_CUDA
    monkeypatch.delenv("SD_FAULT_INJECT")


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_device_call_without_gpu_reports_cuda_error(sd):
    x = np.zeros((1, 512), np.uint16)
    st = sd.lib.sd_w4a16_linear(x.ctypes.data, A, A, A, 128, 1, 64, 512, A, None)
    assert st == sd.SD_ERR_CUDA
