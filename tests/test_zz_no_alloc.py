"""The allocation-free verify GEMM entry point, for callers that cannot
allocate device memory (a plugin handed only its tensors, code inside another
framework's memory pool, a path where cudaMalloc would synchronize).

It must give the same results as verify_gemm_w4 with a caller workspace,
within the GEMM pass rule, on consecutive calls that reuse the library's one
fixed scratch array.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decode_verification_w4_gb300 as vw4
from gpu_util import assert_gemm_close, bf16_dev

pytestmark = pytest.mark.gpu


def _call_noalloc(W, A, out, row_argmax=None):
    lib = vw4.load_library()
    code = lib.verify_gemm_w4_noalloc(ctypes.byref(W), ctypes.c_void_p(A.data_ptr()), A.shape[0],
                                      A.stride(0), ctypes.c_void_p(out.data_ptr()), out.stride(0),
                                      None if row_argmax is None else
                                      ctypes.c_void_p(row_argmax.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, lib.vw4_last_error_string()


@pytest.mark.parametrize("fmt,N,K,M", [("nvfp4", 1000, 2304, 8), ("q4_0", 2049, 512, 3),
                                       ("nvfp4", 17408, 5120, 8), ("nvfp4", 40000, 512, 16),
                                       ("q4_0", 1000, 2304, 12)])
def test_noalloc_matches_workspace_entry_point_twice(fmt, N, K, M):
    q, s, ts = synth.linear(300 + N, N, K, fmt)
    qd = torch.from_numpy(q).cuda()
    sd = torch.from_numpy(s).cuda() if fmt == "nvfp4" else \
        torch.from_numpy(s.view(np.uint16)).cuda().view(torch.float16)
    f = vw4.FMT_NVFP4 if fmt == "nvfp4" else vw4.FMT_Q4_0
    cols = np.unique(np.concatenate([[0, N - 1], synth.rng(5).integers(0, N, 64)])).astype(np.int32)
    for call in range(2):  # two calls in a row share the scratch array
        A = synth.activations(synth.rng(40 + call), M, K)
        Ad = bf16_dev(A)
        ref_out = vw4.verify_gemm_w4(f, qd, sd, ts, Ad)
        W = vw4.make_weight(f, qd, sd, ts, N, K)
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        _call_noalloc(W, Ad, out)
        torch.cuda.synchronize()
        got, want = out.cpu().numpy(), ref_out.cpu().numpy()
        _, bnd = oracle.gemm_w4(oracle.FMT_NVFP4 if fmt == "nvfp4" else oracle.FMT_Q4_0, N, K, q, s,
                                ts, A, cols=cols)
        assert_gemm_close(got[:, cols], want[:, cols].astype(np.float64), bnd, "noalloc vs workspace")
        assert not np.isnan(got).any()


def test_noalloc_fused_argmax_twice():
    """The fused row argmax through the fixed scratch array (its per-row keys
    and ticket live there): two calls in a row, M = 16 and N = 40000, each
    argmax bit-exact against the argmax of the workspace entry point's own
    output (ties to the lowest index)."""
    N, K, M = 40000, 512, 16
    q, s, ts = synth.linear(77, N, K, "nvfp4")
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    W = vw4.make_weight(vw4.FMT_NVFP4, qd, sd, ts, N, K)
    for call in range(2):
        Ad = bf16_dev(synth.activations(synth.rng(60 + call), M, K))
        ref_am = torch.full((M,), -1, dtype=torch.int32, device="cuda")
        ref_out = vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, row_argmax=ref_am)
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        am = torch.full((M,), -1, dtype=torch.int32, device="cuda")
        _call_noalloc(W, Ad, out, row_argmax=am)
        torch.cuda.synchronize()
        assert vw4.vw4_get_device_status() == 0
        want = np.argmax(ref_out.cpu().numpy(), axis=1)
        assert np.array_equal(am.cpu().numpy(), want), (call, am.cpu().numpy(), want)
        assert torch.equal(am, ref_am)
        assert torch.equal(out, ref_out)   # same kernel, same split: the same sums


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = vw4.load_library()
    W = vw4.Weight(vw4.FMT_NVFP4, 2048, 1 << 20, 0, 0x1000, 0x2000, 1.0, 0.0)  # K = 1M: too big
    code = lib.verify_gemm_w4_noalloc(ctypes.byref(W), 0x3000, 8, 1 << 20, 0x4000, 2048, None, None)
    assert code == 6
    assert b"above the fixed" in lib.vw4_last_error_string()
