"""CPU oracle for the quantized speculative-decoding hot path (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference legs of ``bench.py`` may import this package.
The GPU library never does.  ``oracle.c`` holds the arithmetic (fp64,
sequential); this file only marshals numpy arrays and builds the shared
object with the host C compiler on first use.

Each function's source passage is cited in ``oracle.c``.  Parity is pinned by
the ``-m "not gpu"`` tests in tests/test_oracle_*.py, against closed forms,
library routines and brute force.  One function is unpinned: the exact fp64
GEMM rounding below the 1e-2 bound is not pinned by anything but itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_c_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_c_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_c_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_c_i8p = np.ctypeslib.ndpointer(dtype=np.int8, flags="C_CONTIGUOUS")
_c_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_c_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_c_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_c_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_ci, _cu32, _cu64, _cd = ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with the host C compiler."""
    with _lock:
        fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
        if force or not fresh:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cc = os.environ.get("CC", "gcc")
            subprocess.check_call([cc, "-std=c11", "-O2", "-Wall", "-shared", "-fPIC",
                                   "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    lib.oracle_philox4x32.argtypes = [_c_u32p, _c_u32p, _ci, _c_u32p]
    lib.oracle_accept_uniform.argtypes = [_cu64, _cu32, _cu32]
    lib.oracle_accept_uniform.restype = _cd
    lib.oracle_race_exponential.argtypes = [_cu64, _cu32, _cu32, _cu32, _cu32]
    lib.oracle_race_exponential.restype = _cd
    lib.oracle_f64_to_f16.argtypes = [_cd]
    lib.oracle_f64_to_f16.restype = ctypes.c_uint16
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = _cd
    lib.oracle_f64_to_bf16.argtypes = [_cd]
    lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = _cd
    lib.oracle_quantize_w4.argtypes = [_c_f32p, _ci, _ci, _ci, _c_u8p, _c_u16p, _c_u16p]
    lib.oracle_quantize_w4.restype = _ci
    lib.oracle_unpack_w4.argtypes = [_c_u32p, _ci, _ci, _c_u8p]
    lib.oracle_dequant_w4.argtypes = [_c_u8p, _c_u16p, _c_u16p, _ci, _ci, _ci, _c_f64p]
    lib.oracle_w4a16_linear.argtypes = [_c_u16p, _c_u32p, _c_u16p, _c_u16p, _ci, _ci, _ci, _ci,
                                        _c_f64p]
    lib.oracle_quantize_w8.argtypes = [_c_f32p, _ci, _ci, _c_i8p, _c_u16p]
    lib.oracle_quantize_w8.restype = _ci
    lib.oracle_w8a16_linear.argtypes = [_c_u16p, _c_i8p, _c_u16p, _ci, _ci, _ci, _c_f64p]
    lib.oracle_bf16_linear.argtypes = [_c_u16p, _c_u16p, _ci, _ci, _ci, _c_f64p]
    lib.oracle_round_bf16.argtypes = [_c_f64p, ctypes.c_size_t, _c_u16p]
    lib.oracle_softmax.argtypes = [_c_f32p, _ci, _cd, _c_f64p]
    lib.oracle_quantize_wb.argtypes = [_c_f32p, _ci, _ci, _ci, _ci, _c_u8p, _c_u16p, _c_u16p]
    lib.oracle_quantize_wb.restype = _ci
    lib.oracle_pack_wb.argtypes = [_c_u8p, _ci, _ci, _ci, _c_u32p]
    lib.oracle_pack_wb.restype = _ci
    lib.oracle_unpack_wb.argtypes = [_c_u32p, _ci, _ci, _ci, _c_u8p]
    lib.oracle_wb_linear.argtypes = [_c_u16p, _c_u32p, _c_u16p, _c_u16p, _ci, _ci, _ci, _ci, _ci, _c_f64p]
    lib.oracle_quantize_a4.argtypes = [_c_u16p, _ci, _ci, _c_i8p, _c_f32p]
    lib.oracle_quantize_a4.restype = _ci
    lib.oracle_w4a4_linear.argtypes = [_c_u16p, _c_u32p, _c_u16p, _c_u16p, _ci, _ci, _ci, _c_f64p]
    lib.oracle_w4a4_linear.restype = _ci
    lib.oracle_softmax_stats.argtypes = [_c_f32p, _ci, _cd, ctypes.POINTER(_cd), ctypes.POINTER(_cd),
                                         ctypes.POINTER(ctypes.c_int32)]
    lib.oracle_softmax_stats.restype = _ci
    lib.oracle_verify.argtypes = [_c_f32p, _c_f32p, _c_i32p, _ci, _ci, _ci, _cd, _cu64,
                                  _c_i32p, _c_i32p, _c_i32p]
    lib.oracle_verify.restype = _ci
    lib.oracle_sample.argtypes = [_c_f32p, _ci, _cd, _cu64, _cu32, _cu32]
    lib.oracle_sample.restype = _ci
    lib.oracle_sample_flag.argtypes = [_c_f32p, _ci, _cd, _cu64, _cu32, _cu32, ctypes.POINTER(ctypes.c_int32)]
    lib.oracle_sample_flag.restype = _ci
    lib.oracle_verify_trials.argtypes = [_c_f32p, _c_f32p, _ci, _ci, _cd, _cu64, ctypes.c_long,
                                         _c_i64p, _c_i64p, _c_i64p, _c_i64p, _c_i64p]
    lib.oracle_verify_trials.restype = ctypes.c_long
    _lib = lib
    return lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- Philox
def philox4x32(ctr, key, rounds: int = 10) -> np.ndarray:
    out = np.zeros(4, np.uint32)
    _load().oracle_philox4x32(_c(ctr, np.uint32), _c(key, np.uint32), int(rounds), out)
    return out


def accept_uniform(seed: int, b: int, i: int) -> float:
    return _load().oracle_accept_uniform(seed, b, i)


def race_exponential(seed: int, b: int, slot: int, v: int, stream: int = 0) -> float:
    return _load().oracle_race_exponential(seed, b, slot, v, stream)


# ----------------------------------------------------------- float formats
def f64_to_f16_bits(x: float) -> int:
    return int(_load().oracle_f64_to_f16(float(x)))


def f16_bits_to_f64(h: int) -> float:
    return _load().oracle_f16_to_f64(int(h))


def f64_to_bf16_bits(x: float) -> int:
    return int(_load().oracle_f64_to_bf16(float(x)))


def bf16_bits_to_f64(h: int) -> float:
    return _load().oracle_bf16_to_f64(int(h))


def round_bf16(y) -> np.ndarray:
    """fp64 array -> bf16 bit patterns (uint16), round to nearest even."""
    y = _c(y, np.float64)
    out = np.zeros(y.shape, np.uint16)
    _load().oracle_round_bf16(y.reshape(-1), y.size, out.reshape(-1))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    f = _load().oracle_bf16_to_f64
    return np.array([f(int(h)) for h in bits.reshape(-1)], np.float64).reshape(bits.shape)


def f16_to_f64(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    f = _load().oracle_f16_to_f64
    return np.array([f(int(h)) for h in bits.reshape(-1)], np.float64).reshape(bits.shape)


# ------------------------------------------------------------- weights
def quantize_w4(w, group: int = 128):
    """fp32 w [N][K] -> (q uint8 [N][K], scales fp16 bits, zeros fp16 bits)."""
    w = _c(w, np.float32)
    N, K = w.shape
    q = np.zeros((N, K), np.uint8)
    s = np.zeros((N, K // group), np.uint16)
    z = np.zeros((N, K // group), np.uint16)
    if _load().oracle_quantize_w4(w, N, K, group, q, s, z) != 0:
        raise ValueError("oracle_quantize_w4 rejected the input")
    return q, s, z


def unpack_w4(qweight, N: int, K: int) -> np.ndarray:
    q = np.zeros((N, K), np.uint8)
    _load().oracle_unpack_w4(_c(qweight, np.uint32), N, K, q)
    return q


def dequant_w4(q, scales, zeros, group: int = 128) -> np.ndarray:
    q = _c(q, np.uint8)
    N, K = q.shape
    out = np.zeros((N, K), np.float64)
    _load().oracle_dequant_w4(q, _c(scales, np.uint16), _c(zeros, np.uint16), N, K, group, out)
    return out


def w4a16_linear(x_bf16_bits, qweight, scales, zeros, group: int, N: int, K: int) -> np.ndarray:
    x = _c(x_bf16_bits, np.uint16)
    M = x.shape[0]
    y = np.zeros((M, N), np.float64)
    _load().oracle_w4a16_linear(x, _c(qweight, np.uint32), _c(scales, np.uint16),
                                _c(zeros, np.uint16), group, M, N, K, y)
    return y


def quantize_wb(w, bits: int, group: int = 128):
    """R11: fp32 w [N][K] -> (q uint8 [N][K] in 0..2^bits-1, scales, zeros fp16 bits)."""
    w = _c(w, np.float32)
    N, K = w.shape
    q = np.zeros((N, K), np.uint8)
    s = np.zeros((N, K // group), np.uint16)
    z = np.zeros((N, K // group), np.uint16)
    if _load().oracle_quantize_wb(w, N, K, group, bits, q, s, z) != 0:
        raise ValueError("oracle_quantize_wb rejected the input")
    return q, s, z


def pack_wb(q, bits: int) -> np.ndarray:
    """R11 layout: uint32 [N][K*bits/32], each row one little-endian bit stream."""
    q = _c(q, np.uint8)
    N, K = q.shape
    if (K * bits) % 32:
        raise ValueError("K * bits must be a multiple of 32")
    out = np.zeros((N, K * bits // 32), np.uint32)
    if _load().oracle_pack_wb(q, N, K, bits, out) != 0:
        raise ValueError("oracle_pack_wb rejected the input")
    return out


def unpack_wb(packed, N: int, K: int, bits: int) -> np.ndarray:
    q = np.zeros((N, K), np.uint8)
    _load().oracle_unpack_wb(_c(packed, np.uint32), N, K, bits, q)
    return q


def wb_linear(x_bf16_bits, packed, scales, zeros, group: int, bits: int, N: int, K: int) -> np.ndarray:
    x = _c(x_bf16_bits, np.uint16)
    M = x.shape[0]
    y = np.zeros((M, N), np.float64)
    _load().oracle_wb_linear(x, _c(packed, np.uint32), _c(scales, np.uint16), _c(zeros, np.uint16),
                             group, bits, M, N, K, y)
    return y


def quantize_a4(x_bf16_bits):
    """R12: bf16 bits [M][K] -> (codes int8 [M][K] in -8..7, fp32 scales [M][K/128])."""
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    qx = np.zeros((M, K), np.int8)
    sx = np.zeros((M, K // 128), np.float32)
    if _load().oracle_quantize_a4(x, M, K, qx, sx) != 0:
        raise ValueError("oracle_quantize_a4 rejected the input")
    return qx, sx


def w4a4_linear(x_bf16_bits, qweight, scales, zeros, N: int, K: int) -> np.ndarray:
    x = _c(x_bf16_bits, np.uint16)
    M = x.shape[0]
    y = np.zeros((M, N), np.float64)
    if _load().oracle_w4a4_linear(x, _c(qweight, np.uint32), _c(scales, np.uint16), _c(zeros, np.uint16),
                                  M, N, K, y) != 0:
        raise ValueError("oracle_w4a4_linear rejected the input")
    return y


def quantize_w8(w):
    w = _c(w, np.float32)
    N, K = w.shape
    q = np.zeros((N, K), np.int8)
    s = np.zeros((N,), np.uint16)
    if _load().oracle_quantize_w8(w, N, K, q, s) != 0:
        raise ValueError("oracle_quantize_w8 rejected the input")
    return q, s


def w8a16_linear(x_bf16_bits, q8, scales) -> np.ndarray:
    x = _c(x_bf16_bits, np.uint16)
    q8 = _c(q8, np.int8)
    M, K = x.shape
    N = q8.shape[0]
    y = np.zeros((M, N), np.float64)
    _load().oracle_w8a16_linear(x, q8, _c(scales, np.uint16), M, N, K, y)
    return y


def bf16_linear(x_bf16_bits, w_bf16_bits) -> np.ndarray:
    x = _c(x_bf16_bits, np.uint16)
    w = _c(w_bf16_bits, np.uint16)
    M, K = x.shape
    N = w.shape[0]
    y = np.zeros((M, N), np.float64)
    _load().oracle_bf16_linear(x, w, M, N, K, y)
    return y


# -------------------------------------------------------------- verify
def softmax(logits, T: float) -> np.ndarray:
    lg = _c(logits, np.float32)
    p = np.zeros(lg.shape[-1], np.float64)
    _load().oracle_softmax(lg, lg.shape[-1], float(T), p)
    return p


def softmax_stats(logits, T: float):
    """(m, Z, argmax) of one row or slice: m = max logit, Z = sum exp((l - m)/T)
    (0.0 at T = 0), argmax with the lowest index on ties."""
    lg = _c(logits, np.float32)
    m, z, a = ctypes.c_double(0.0), ctypes.c_double(0.0), ctypes.c_int32(0)
    rc = _load().oracle_softmax_stats(lg, lg.shape[-1], float(T), ctypes.byref(m), ctypes.byref(z),
                                      ctypes.byref(a))
    if rc != 0:
        raise ValueError("oracle_softmax_stats rejected the input")
    return m.value, z.value, int(a.value)


def verify(draft_logits, target_logits, draft_tokens, gamma: int, T: float, seed: int):
    """Returns (out_tokens [B][gamma+1], accept_len [B], flags [B])."""
    dl = _c(draft_logits, np.float32)
    tl = _c(target_logits, np.float32)
    dt = _c(draft_tokens, np.int32)
    B = dt.shape[0]
    V = tl.shape[-1]
    out = np.zeros((B, gamma + 1), np.int32)
    alen = np.zeros((B,), np.int32)
    flags = np.zeros((B,), np.int32)
    rc = _load().oracle_verify(dl.reshape(-1) if B else np.zeros(1, np.float32),
                               tl.reshape(-1) if B else np.zeros(1, np.float32),
                               dt.reshape(-1) if B else np.zeros(1, np.int32),
                               gamma, B, V, float(T), int(seed),
                               out.reshape(-1) if B else np.zeros(1, np.int32),
                               alen if B else np.zeros(1, np.int32),
                               flags if B else np.zeros(1, np.int32))
    if rc != 0:
        raise ValueError("oracle_verify rejected the input")
    return out, alen, flags


FLAG_RACE = 1 << 30


def sample(logits, T: float, seed: int, b: int, slot: int) -> int:
    return int(_load().oracle_sample(_c(logits, np.float32), len(logits), float(T), seed, b, slot))


def sample_flag(logits, T: float, seed: int, b: int, slot: int):
    """(token, near-tie flag) of the draft-side sampler for one row."""
    f = ctypes.c_int32(0)
    tok = int(_load().oracle_sample_flag(_c(logits, np.float32), len(logits), float(T), seed, b, slot,
                                         ctypes.byref(f)))
    return tok, bool(f.value)


def verify_trials(draft_logits, target_logits, gamma: int, T: float, seed0: int, ntrials: int):
    dl = _c(draft_logits, np.float32)
    tl = _c(target_logits, np.float32)
    V = tl.shape[-1]
    hist_len = np.zeros(gamma + 1, np.int64)
    hist_tok = np.zeros((gamma + 1, V), np.int64)
    hist_new = np.zeros((gamma + 1, V), np.int64)
    accepted = np.zeros(gamma, np.int64)
    reached = np.zeros(gamma, np.int64)
    nflag = _load().oracle_verify_trials(dl.reshape(-1), tl.reshape(-1), gamma, V, float(T),
                                         int(seed0), int(ntrials), hist_len, hist_tok, hist_new,
                                         accepted, reached)
    if nflag < 0:
        raise ValueError("oracle_verify_trials failed")
    return dict(hist_len=hist_len, hist_tok=hist_tok, hist_new=hist_new, accepted=accepted,
                reached=reached, nflag=nflag)
