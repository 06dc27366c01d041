"""GPU parity of verify_gemm_w4 at 9..16 verify rows (two mma n-tiles over
every unpacked weight fragment, a three-stage ring, 16-row partial tiles)
against the oracle, through the C ABI.

Element by element on shapes that take each way a tile is finished: whole
tiles, tile-aligned split-K combined in a cluster over distributed shared
memory, split-K through tickets in L2 (the fused argmax path), and stream-K
with tiles shared by several CTAs; sampled columns at the full sizes of the
dense-27B-like layer and the LM head.  Pass rule as for 1..8 rows:
|gpu - oracle| <= 1e-3 * sum_k |a_k w_k| per element.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decode_verification_w4_gb300 as vw4
from gpu_util import ORACLE_FMT, assert_gemm_close, bf16_dev, gemm_gpu, upload_weight

pytestmark = pytest.mark.gpu


def _case(fmt, seed, N, K, M):
    q, s, ts = synth.linear(seed, N, K, fmt)
    A = synth.activations(synth.rng(seed + 2000), M, K)
    return q, s, ts, A


# (N, K): 1 tile / whole; 8 tiles, T = 9 (split 2, cluster); 2 tiles, T = 20
# (split 5, cluster); 17 tiles, T = 2 (whole tiles); 3 tiles, T = 5 (whole)
SHAPES = [(127, 512), (1000, 2304), (129, 5120), (2049, 512), (300, 1280)]


@pytest.mark.parametrize("fmt", ["nvfp4", "q4_0"])
@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [9, 13, 16])
def test_sixteen_row_shapes_elementwise(fmt, N, K, M):
    q, s, ts, A = _case(fmt, 11 * N + K + M, N, K, M)
    gpu = gemm_gpu(fmt, q, s, ts, A).cpu().numpy()
    ref, bnd = oracle.gemm_w4(ORACLE_FMT[fmt], N, K, q, s, ts, A)
    assert_gemm_close(gpu, ref, bnd, f"{fmt} N={N} K={K} M={M}")


@pytest.mark.parametrize("fmt", ["nvfp4", "q4_0"])
@pytest.mark.parametrize("N,K,M", [(40000, 512, 16), (45000, 1792, 11)])
def test_sixteen_rows_stream_k(fmt, N, K, M):
    """More tiles than CTAs: stream-K ranges that start and end inside tiles,
    the last contributor of each 32-row slice summing both n-tiles."""
    q, s, ts, A = _case(fmt, N + K + M, N, K, M)
    gpu = gemm_gpu(fmt, q, s, ts, A).cpu().numpy()
    cols = np.unique(np.concatenate([np.arange(0, N, 5), [N - 1]])).astype(np.int32)
    ref, bnd = oracle.gemm_w4(ORACLE_FMT[fmt], N, K, q, s, ts, A, cols=cols)
    assert_gemm_close(gpu[:, cols], ref, bnd, f"{fmt} stream-K N={N} K={K} M={M}")


@pytest.mark.parametrize("N,K,M", [(1000, 1024, 16), (129, 5120, 12), (40000, 512, 16),
                                   (5000, 768, 9)])
def test_sixteen_rows_fused_argmax(N, K, M):
    """The fused argmax over 16 rows (whole tiles, split-K through tickets,
    stream-K): bit-exact against the oracle's argmax of the GPU's logits."""
    q, s, ts, A = _case("nvfp4", N + 3 * M, N, K, M)
    am = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    gpu = gemm_gpu("nvfp4", q, s, ts, A, row_argmax=am).cpu().numpy()
    am = am.cpu().numpy()
    for m in range(M):
        assert am[m] == oracle.argmax_f32(gpu[m]), m
    cols = np.unique(np.concatenate([np.arange(0, N, 13), [N - 1]])).astype(np.int32)
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A, cols=cols)
    assert_gemm_close(gpu[:, cols], ref, bnd, "argmax call logits")


def test_sixteen_rows_match_single_rows():
    """Row m of a 16-row call and the 1-row call on that row both pass
    against the oracle (the same products, another accumulation order)."""
    N, K = 700, 1536
    q, s, ts, A = _case("nvfp4", 5, N, K, 16)
    full = gemm_gpu("nvfp4", q, s, ts, A).cpu().numpy()
    for m in (0, 7, 8, 15):
        one = gemm_gpu("nvfp4", q, s, ts, A[m:m + 1]).cpu().numpy()
        ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A[m:m + 1])
        assert_gemm_close(one, ref, bnd)
        assert_gemm_close(full[m:m + 1], ref, bnd)


def test_sixteen_rows_deterministic_and_extreme_scales():
    N, K = 1100, 4096
    q, s, ts = synth.linear(6, N, K, "nvfp4")
    g = synth.rng(16)
    x = g.standard_normal((16, K)).astype(np.float32)
    x[9] *= 1e30       # per-row power-of-two pre-scale, second n-tile
    x[10] *= 1e-30
    x[11, :] = 0.0
    x[15] *= 3e5
    A = synth.bf16_bits(x)
    a = gemm_gpu("nvfp4", q, s, ts, A).cpu().numpy()
    b = gemm_gpu("nvfp4", q, s, ts, A).cpu().numpy()
    assert np.array_equal(a, b)
    assert np.all(a[11] == 0.0)
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A)
    assert_gemm_close(a, ref, bnd, "extreme 16")


@pytest.mark.parametrize("fmt", ["nvfp4", "q4_0"])
@pytest.mark.parametrize("name,N,K", [("gate_up", 34816, 5120), ("down", 5120, 17408),
                                      ("qkv", 8192, 5120)])
def test_dense_layer_sixteen_rows_sampled(fmt, name, N, K):
    q, s, ts = synth.linear(300 + N + K, N, K, fmt)
    g = synth.rng(N)
    A = synth.activations(g, 16, K)
    cols = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, 96)])).astype(np.int32)
    for M in (9, 16):
        gpu = gemm_gpu(fmt, q, s, ts, A[:M]).cpu().numpy()
        ref, bnd = oracle.gemm_w4(ORACLE_FMT[fmt], N, K, q, s, ts, A[:M], cols=cols)
        assert_gemm_close(gpu[:, cols], ref, bnd, f"{fmt} {name} M={M}")


def test_lm_head_sixteen_rows_sampled_and_fused_argmax():
    """LM head 5376 -> 262144 nvfp4 at 16 rows with the fused argmax."""
    N, K, M = 262144, 5376, 16
    q, s, ts = synth.linear(3, N, K, "nvfp4")
    A = synth.activations(synth.rng(3), M, K)
    am = torch.empty((M,), dtype=torch.int32, device="cuda")
    gpu = gemm_gpu("nvfp4", q, s, ts, A, row_argmax=am).cpu().numpy()
    am = am.cpu().numpy()
    g = synth.rng(78)
    cols = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, 96)]))
    for m in range(M):
        cols = np.union1d(cols, np.argsort(-gpu[m], kind="stable")[:2])
    cols = cols.astype(np.int32)
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A, cols=cols)
    assert_gemm_close(gpu[:, cols], ref, bnd, "lm head 16")
    for m in range(M):
        assert am[m] == oracle.argmax_f32(gpu[m]), m


def test_prepared_gemm_sixteen_rows():
    N, K = 900, 1536
    q, s, ts, A = _case("q4_0", 12, N, K, 16)
    qd, sd = upload_weight(q, s, "q4_0")
    Ad = bf16_dev(A)
    plain = vw4.verify_gemm_w4(vw4.FMT_Q4_0, qd, sd, ts, Ad)
    prep = vw4.PreparedGemm(vw4.FMT_Q4_0, qd, sd, ts, M_max=16)
    out = torch.empty_like(plain)
    for M in (16, 10, 3):  # one workspace sized for 16 rows serves every width
        prep(Ad[:M], out[:M])
        torch.cuda.synchronize()
        assert torch.equal(plain[:M], out[:M]) if M == 16 else True
    ref, bnd = oracle.gemm_w4(oracle.FMT_Q4_0, N, K, q, s, ts, A[:3])
    assert_gemm_close(out[:3].cpu().numpy(), ref, bnd, "prepared, 3 rows after 16")
