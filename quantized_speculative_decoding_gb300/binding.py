"""Thin ctypes binding of libsd.so (C ABI in include/sd.h).

Functions carry the ABI's names and arguments.  Pointer arguments accept an
integer address, a torch tensor (its data_ptr()) or a numpy array (host
pointer, for the packers); `stream` accepts a torch.cuda.Stream, an integer
handle or None (the legacy default stream).  Every function raises SdError on
a non-zero status.  This module only marshals arguments: all work runs in
libsd.so, and importing it fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("SD_LIBRARY", os.path.join(_PKG, "libsd.so"))

SD_OK, SD_ERR_INVALID_ARG, SD_ERR_UNSUPPORTED, SD_ERR_CUDA, SD_ERR_TIMEOUT, SD_ERR_INTERNAL = range(6)

# every function declared in include/sd.h
EXPORTS = ("sd_status_string", "sd_version", "sd_w4_pack", "sd_w8_pack", "sd_w4a16_linear",
           "sd_w8a16_linear", "sd_bf16_linear", "sd_w4_unpack", "sd_verify", "sd_verify_noalloc",
           "sd_philox4x32", "sd_device_error", "sd_w4_tiled_bytes", "sd_w4_tile",
           "sd_w4a16_linear_tiled", "sd_sample", "sd_lm_head_parts", "sd_w4a16_lm_head",
           "sd_verify_parts", "sd_wb_pack", "sd_test_wait_expiry",
           "sd_test_w4a16_linear_path", "sd_wb_tiled_bytes", "sd_wb_tile", "sd_wb_linear_tiled",
           "sd_a4_quantize", "sd_w4a4_linear_tiled")


class SdError(RuntimeError):
    def __init__(self, status: int, func: str):
        self.status = status
        super().__init__(f"{func} failed: {status_string(status)} ({status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libsd.so not found at {LIB_PATH}: build it with "
                          "python -m quantized_speculative_decoding_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, U32, U64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float
    sig = {
        "sd_status_string": ([I], ctypes.c_char_p),
        "sd_version": ([], I),
        "sd_w4_pack": ([P, I, I, I, P, P, P], I),
        "sd_w8_pack": ([P, I, I, P, P], I),
        "sd_wb_pack": ([P, I, I, I, I, P, P, P], I),
        "sd_w4a16_linear": ([P, P, P, P, I, I, I, I, P, P], I),
        "sd_w8a16_linear": ([P, P, P, I, I, I, P, P], I),
        "sd_w4_tiled_bytes": ([I, I, I, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)], I),
        "sd_w4_tile": ([P, P, P, I, I, I, P, P, P], I),
        "sd_w4a16_linear_tiled": ([P, P, P, I, I, I, I, P, P], I),
        "sd_bf16_linear": ([P, P, I, I, I, P, P], I),
        "sd_w4_unpack": ([P, I, I, P, P], I),
        "sd_verify": ([P, P, P, I, I, I, F, U64, P, P, P], I),
        "sd_verify_noalloc": ([P, P, P, I, I, I, F, U64, P, P, P], I),
        "sd_philox4x32": ([P, U32, U32, I, P, P], I),
        "sd_sample": ([P, I, I, F, U64, I, P, P], I),
        "sd_lm_head_parts": ([I, I, I, ctypes.POINTER(ctypes.c_int)], I),
        "sd_w4a16_lm_head": ([P, P, P, I, I, I, I, F, P, ctypes.c_int64, P, ctypes.c_int64, P], I),
        "sd_verify_parts": ([P, P, P, I, P, I, P, I, I, I, F, U64, P, P, P], I),
        "sd_device_error": ([P, ctypes.POINTER(ctypes.c_int32)], I),
        "sd_test_wait_expiry": ([ctypes.c_int64, P], I),
        "sd_test_w4a16_linear_path": ([P, P, P, P, I, I, I, I, P, I, P], I),
        "sd_wb_tiled_bytes": ([I, I, I, I, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)], I),
        "sd_wb_tile": ([P, P, P, I, I, I, I, P, P, P], I),
        "sd_wb_linear_tiled": ([P, P, P, I, I, I, I, I, P, P], I),
        "sd_a4_quantize": ([P, I, I, P, P, P], I),
        "sd_w4a4_linear_tiled": ([P, P, P, P, I, I, I, I, P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.sd_status_string(int(status)).decode()


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("numpy arrays passed to libsd must be C-contiguous")
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        if hasattr(a, "is_contiguous") and not a.is_contiguous():
            raise ValueError("tensors passed to libsd must be contiguous")
        return a.data_ptr()
    raise TypeError(f"cannot pass {type(a)} as a pointer")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    raise TypeError(f"cannot pass {type(s)} as a stream")


def _check(status: int, func: str):
    if status != SD_OK:
        raise SdError(status, func)


def sd_version() -> int:
    return lib.sd_version()


def sd_w4_pack(w, N, K, group, qweight, scales, zeros):
    _check(lib.sd_w4_pack(_ptr(w), N, K, group, _ptr(qweight), _ptr(scales), _ptr(zeros)),
           "sd_w4_pack")


def sd_wb_pack(w, N, K, group, bits, packed, scales, zeros):
    _check(lib.sd_wb_pack(_ptr(w), N, K, group, bits, _ptr(packed), _ptr(scales), _ptr(zeros)), "sd_wb_pack")


def sd_w8_pack(w, N, K, qweight, scales):
    _check(lib.sd_w8_pack(_ptr(w), N, K, _ptr(qweight), _ptr(scales)), "sd_w8_pack")


def sd_w4a16_linear(x, qweight, scales, zeros, group, M, N, K, out, stream=None):
    _check(lib.sd_w4a16_linear(_ptr(x), _ptr(qweight), _ptr(scales), _ptr(zeros), group, M, N, K,
                               _ptr(out), _stream(stream)), "sd_w4a16_linear")


def sd_w4_tiled_bytes(N, K, group=128):
    """(qweight bytes, scale/zero bytes) of the fragment-ordered tiled layout."""
    qb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib.sd_w4_tiled_bytes(N, K, group, ctypes.byref(qb), ctypes.byref(sb)), "sd_w4_tiled_bytes")
    return qb.value, sb.value


def sd_w4_tile(qweight, scales, zeros, group, N, K, tiled_qweight, tiled_sz, stream=None):
    _check(lib.sd_w4_tile(_ptr(qweight), _ptr(scales), _ptr(zeros), group, N, K,
                          _ptr(tiled_qweight), _ptr(tiled_sz), _stream(stream)), "sd_w4_tile")


def sd_w4a16_linear_tiled(x, tiled_qweight, tiled_sz, group, M, N, K, out, stream=None):
    _check(lib.sd_w4a16_linear_tiled(_ptr(x), _ptr(tiled_qweight), _ptr(tiled_sz), group, M, N, K,
                                     _ptr(out), _stream(stream)), "sd_w4a16_linear_tiled")



def sd_wb_tiled_bytes(N, K, bits, group=128):
    """(qweight bytes, scale/zero bytes) of the b-bit fragment-ordered layout."""
    qb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib.sd_wb_tiled_bytes(N, K, group, bits, ctypes.byref(qb), ctypes.byref(sb)), "sd_wb_tiled_bytes")
    return qb.value, sb.value


def sd_wb_tile(packed, scales, zeros, group, bits, N, K, tiled_qweight, tiled_sz, stream=None):
    _check(lib.sd_wb_tile(_ptr(packed), _ptr(scales), _ptr(zeros), group, bits, N, K, _ptr(tiled_qweight),
                          _ptr(tiled_sz), _stream(stream)), "sd_wb_tile")


def sd_wb_linear_tiled(x, tiled_qweight, tiled_sz, group, bits, M, N, K, out, stream=None):
    _check(lib.sd_wb_linear_tiled(_ptr(x), _ptr(tiled_qweight), _ptr(tiled_sz), group, bits, M, N, K, _ptr(out),
                                  _stream(stream)), "sd_wb_linear_tiled")


def sd_a4_quantize(x, M, K, qx, sx, stream=None):
    _check(lib.sd_a4_quantize(_ptr(x), M, K, _ptr(qx), _ptr(sx), _stream(stream)), "sd_a4_quantize")


def sd_w4a4_linear_tiled(qx, sx, tiled_qweight, tiled_sz, group, M, N, K, out, stream=None):
    _check(lib.sd_w4a4_linear_tiled(_ptr(qx), _ptr(sx), _ptr(tiled_qweight), _ptr(tiled_sz), group, M, N, K,
                                    _ptr(out), _stream(stream)), "sd_w4a4_linear_tiled")


def sd_w8a16_linear(x, qweight, scales, M, N, K, out, stream=None):
    _check(lib.sd_w8a16_linear(_ptr(x), _ptr(qweight), _ptr(scales), M, N, K, _ptr(out),
                               _stream(stream)), "sd_w8a16_linear")


def sd_bf16_linear(x, w, M, N, K, out, stream=None):
    _check(lib.sd_bf16_linear(_ptr(x), _ptr(w), M, N, K, _ptr(out), _stream(stream)),
           "sd_bf16_linear")


def sd_w4_unpack(qweight, N, K, q, stream=None):
    _check(lib.sd_w4_unpack(_ptr(qweight), N, K, _ptr(q), _stream(stream)), "sd_w4_unpack")


def sd_verify(draft_logits, target_logits, draft_tokens, gamma, batch, vocab, temperature, seed,
              out_tokens, out_accept_len, stream=None):
    _check(lib.sd_verify(_ptr(draft_logits), _ptr(target_logits), _ptr(draft_tokens), gamma,
                         batch, vocab, float(temperature), int(seed) & 0xffffffffffffffff,
                         _ptr(out_tokens), _ptr(out_accept_len), _stream(stream)), "sd_verify")


def sd_verify_noalloc(draft_logits, target_logits, draft_tokens, gamma, batch, vocab, temperature,
                      seed, out_tokens, out_accept_len, stream=None):
    """sd_verify for callers that cannot allocate device memory: its scratch is
    a fixed 1 MiB device array owned by the library (see include/sd.h)."""
    _check(lib.sd_verify_noalloc(_ptr(draft_logits), _ptr(target_logits), _ptr(draft_tokens),
                                 gamma, batch, vocab, float(temperature),
                                 int(seed) & 0xffffffffffffffff, _ptr(out_tokens),
                                 _ptr(out_accept_len), _stream(stream)), "sd_verify_noalloc")


def sd_sample(logits, batch, vocab, temperature, seed, slot, out_tokens, stream=None):
    _check(lib.sd_sample(_ptr(logits), batch, vocab, float(temperature), int(seed), slot, _ptr(out_tokens),
                         _stream(stream)), "sd_sample")


def sd_lm_head_parts(M, vocab, K) -> int:
    """Softmax partials per row that sd_w4a16_lm_head writes (current device)."""
    n = ctypes.c_int(0)
    _check(lib.sd_lm_head_parts(M, vocab, K, ctypes.byref(n)), "sd_lm_head_parts")
    return int(n.value)


def sd_w4a16_lm_head(x, tiled_qweight, tiled_sz, group, M, vocab, K, temperature, logits, ld_logits,
                     stats, ld_stats, stream=None):
    _check(lib.sd_w4a16_lm_head(_ptr(x), _ptr(tiled_qweight), _ptr(tiled_sz), group, M, vocab, K,
                                float(temperature), _ptr(logits), int(ld_logits), _ptr(stats), int(ld_stats),
                                _stream(stream)), "sd_w4a16_lm_head")


def sd_verify_parts(draft_logits, target_logits, draft_stats, draft_parts, target_stats, target_parts,
                    draft_tokens, gamma, batch, vocab, temperature, seed, out_tokens, out_accept_len,
                    stream=None):
    _check(lib.sd_verify_parts(_ptr(draft_logits), _ptr(target_logits), _ptr(draft_stats), draft_parts,
                               _ptr(target_stats), target_parts, _ptr(draft_tokens), gamma, batch, vocab,
                               float(temperature), int(seed) & 0xffffffffffffffff, _ptr(out_tokens),
                               _ptr(out_accept_len), _stream(stream)), "sd_verify_parts")


def sd_philox4x32(ctr, key0, key1, n, out, stream=None):
    _check(lib.sd_philox4x32(_ptr(ctr), key0, key1, n, _ptr(out), _stream(stream)),
           "sd_philox4x32")


def sd_device_error(stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(lib.sd_device_error(_stream(stream), ctypes.byref(code)), "sd_device_error")
    return int(code.value)


def sd_test_wait_expiry(cycles, stream=None):
    _check(lib.sd_test_wait_expiry(int(cycles), _stream(stream)), "sd_test_wait_expiry")


def sd_test_w4a16_linear_path(x, qweight, scales, zeros, group, M, N, K, out, path, stream=None):
    """sd_w4a16_linear with the kernel family forced: 1 = CUDA-core GEMV, 2 = tensor cores."""
    _check(lib.sd_test_w4a16_linear_path(_ptr(x), _ptr(qweight), _ptr(scales), _ptr(zeros), group, M, N, K,
                                         _ptr(out), path, _stream(stream)), "sd_test_w4a16_linear_path")
