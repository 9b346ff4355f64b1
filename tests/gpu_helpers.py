"""Helpers shared by the -m gpu tests: device upload/download and the
GPU-vs-oracle comparison rules."""
import numpy as np
import torch

import oracle

TOL = 1e-2  # GEMM: max-abs error <= 1e-2 * max|ref| (bf16 out, fp32 accumulate)


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).cuda()
    return torch.from_numpy(a).cuda()


def bf16_out(M: int, N: int) -> torch.Tensor:
    return torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")


def bf16_to_np64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def pack_w4(sd, w: np.ndarray):
    N, K = w.shape
    qw = np.zeros((N, K // 8), np.uint32)
    s = np.zeros((N, K // 128), np.uint16)
    z = np.zeros((N, K // 128), np.uint16)
    sd.sd_w4_pack(w, N, K, 128, qw, s, z)
    return qw, s, z


def assert_close(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = ""):
    assert np.all(np.isfinite(y_gpu)), what
    err = np.abs(y_gpu - y_ref).max()
    bound = TOL * np.abs(y_ref).max()
    assert err <= bound, f"{what}: max-abs err {err:.3e} > {bound:.3e}"
    return err / np.abs(y_ref).max()


def compare_verify(out_g, len_g, out_o, len_o, flags, gamma):
    """Bit-exact tokens and accept lengths, except batch elements whose
    oracle decisions were flagged as near ties.  Returns (#mismatch, #flagged,
    #decisions)."""
    out_g = np.asarray(out_g)
    len_g = np.asarray(len_g)
    mism = np.flatnonzero((len_g != len_o) | np.any(out_g != out_o, axis=1))
    flagged = flags != 0
    bad = [b for b in mism if not flagged[b]]
    assert not bad, (f"{len(bad)} unflagged mismatches, e.g. b={bad[0]}: gpu {out_g[bad[0]]} "
                     f"len {len_g[bad[0]]} vs oracle {out_o[bad[0]]} len {len_o[bad[0]]}")
    decisions = int(np.sum(np.minimum(len_o + 1, gamma)) + len(len_o))
    nflag = int(sum(bin(int(f) & 0xffff).count("1") + (1 if f & oracle.FLAG_RACE else 0)
                    for f in flags))
    return len(mism), nflag, decisions
