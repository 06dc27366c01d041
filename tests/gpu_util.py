"""Helpers shared by the GPU parity tests: upload synthetic inputs, call the
library through its C ABI binding, and compare with the oracle."""
import numpy as np
import torch

import oracle
import speculative_decode_verification_w4_gb300 as vw4

FMT = {"nvfp4": vw4.FMT_NVFP4, "q4_0": vw4.FMT_Q4_0}
ORACLE_FMT = {"nvfp4": oracle.FMT_NVFP4, "q4_0": oracle.FMT_Q4_0}

# Pass rule of the verify GEMM: |gpu - oracle| <= 1e-3 * sum_k |a_k * w_k|.
GEMM_REL = 1e-3


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def upload_weight(q, s, fmt):
    qd = dev(q)
    sd = dev(s) if fmt == "nvfp4" else dev(s.view(np.uint16)).view(torch.float16)
    return qd, sd


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def gemm_gpu(fmt, q, s, ts, A_bits, out=None, row_argmax=None, lda_pad=0, ldo_pad=0):
    qd, sd = upload_weight(q, s, fmt)
    M, K = A_bits.shape
    if lda_pad:
        big = np.zeros((M, K + lda_pad), np.uint16)
        big[:, :K] = A_bits
        Ad = bf16_dev(big)[:, :K]
    else:
        Ad = bf16_dev(A_bits)
    N = q.shape[0]
    if ldo_pad and out is None:
        out = torch.full((M, N + ldo_pad), float("nan"), dtype=torch.float32, device="cuda")[:, :N]
    o = vw4.verify_gemm_w4(FMT[fmt], qd, sd, ts, Ad, out=out, row_argmax=row_argmax)
    torch.cuda.synchronize()
    st = vw4.vw4_get_device_status()
    assert st == 0, f"device status {st:#x} after verify_gemm_w4"
    return o


def assert_gemm_close(gpu, ref, bound, what=""):
    gpu = np.asarray(gpu, np.float64)
    err = np.abs(gpu - ref)
    lim = GEMM_REL * bound
    bad = ~(err <= lim)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside 1e-3*sum|a*w|; first at "
                             f"{tuple(i)} gpu={gpu[tuple(i)]} ref={ref[tuple(i)]} "
                             f"bound={bound[tuple(i)]}")
    return float(np.max(err / np.maximum(bound, 1e-300)))
