"""The bounded waits of the verify GEMM, driven to run out without a fault.

A device-side failure must surface as a status, never as a hang or a
half-committed run (Ollama's mtp.go commit log: the run is recorded before it
is streamed, so a cancelled stream leaves no partial state).  The test hook
vw4_test_inject_stall makes a launch's consumer warps wait on a barrier that
nothing completes; with a short wait limit the launch must set
VW4_DEV_WAIT_TIMEOUT, drain its copies and return, and the next call must be
correct again.  Each tile-finish mode is covered: stream-K with L2 tickets,
tile-aligned split-K combined in a thread-block cluster, and the fused argmax
with the greedy accept in the same launch (whose tokens are then not written).
The rejection accept has no waits to bound."""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decode_verification_w4_gb300 as vw4
from gpu_util import assert_gemm_close, bf16_dev, upload_weight

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,M,mode", [(40000, 512, 8, "stream-K"),
                                        (1024, 5120, 8, "cluster split-K"),
                                        (20000, 1024, 8, "fused argmax + greedy"),
                                        (1000, 2304, 12, "16-row cluster split-K")])
def test_wait_limit_runs_out_then_recovers(N, K, M, mode):
    q, s, ts = synth.linear(50 + M, N, K, "nvfp4")
    A = synth.activations(synth.rng(51), M, K)
    qd, sd = upload_weight(q, s, "nvfp4")
    Ad = bf16_dev(A)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    drafts = torch.zeros((1, M - 1), dtype=torch.int32, device="cuda")
    tokens = torch.full((1, M), -7, dtype=torch.int32, device="cuda")
    length = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    vw4.vw4_get_device_status()
    vw4.vw4_set_wait_limit_ns(2_000_000)        # 2 ms
    vw4.vw4_test_inject_stall(1)
    try:
        if mode.startswith("fused"):
            vw4.verify_greedy_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, drafts, out=out, tokens=tokens,
                                 length=length)
        else:
            vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, out=out)
        torch.cuda.synchronize()
        st = vw4.vw4_get_device_status()
    finally:
        vw4.vw4_test_inject_stall(0)
        vw4.vw4_set_wait_limit_ns(0)
    assert st & vw4.DEV_WAIT_TIMEOUT, (mode, st)
    if mode.startswith("fused"):    # no partial run was committed
        assert torch.all(tokens == -7) and int(length[0]) == -7
    # the next call, with the default limit, is complete and correct
    gpu = vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad).cpu().numpy()
    assert vw4.vw4_get_device_status() == 0
    cols = np.unique(np.concatenate([[0, N - 1], synth.rng(52).integers(0, N, 200)])).astype(
        np.int32)
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A, cols=cols)
    assert_gemm_close(gpu[:, cols], ref, bnd, f"after the timeout ({mode})")
