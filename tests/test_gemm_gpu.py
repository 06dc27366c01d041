"""GPU parity of verify_gemm_w4 against the oracle (through the C ABI).

Element by element on small shapes that span several 128-row tiles, several
256-wide k slices, stream-K splits and a ragged row tail; on sampled columns
at the full sizes of the dense-27B-like layer and the LM head; plus the fused
argmax (bit-exact against the oracle's argmax of the GPU's own fp32 logits).
Pass rule: |gpu - oracle| <= 1e-3 * sum_k |a_k w_k| per element.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decode_verification_w4_gb300 as vw4
from gpu_util import (ORACLE_FMT, assert_gemm_close, bf16_dev, gemm_gpu, upload_weight)

pytestmark = pytest.mark.gpu

DENSE = {  # the dense-27B-like layer: name -> (N, K)
    "q": (6144, 5120), "k": (1024, 5120), "v": (1024, 5120), "o": (5120, 6144),
    "gate": (17408, 5120), "up": (17408, 5120), "down": (5120, 17408),
}


def _case(fmt, seed, N, K, M):
    q, s, ts = synth.linear(seed, N, K, fmt)
    A = synth.activations(synth.rng(seed + 1000), M, K)
    return q, s, ts, A


def test_tiny_config_nvfp4_m4():
    """Tiny verify: K=N=1024, nvfp4 N(0, 0.02), bf16 N(0,1) M=4, seed 0."""
    q, s, ts = synth.linear(0, 1024, 1024, "nvfp4")
    A = synth.activations(synth.rng(0), 4, 1024)
    gpu = gemm_gpu("nvfp4", q, s, ts, A).cpu().numpy()
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, 1024, 1024, q, s, ts, A)
    assert_gemm_close(gpu, ref, bnd, "tiny")


@pytest.mark.parametrize("fmt", ["nvfp4", "q4_0"])
@pytest.mark.parametrize("N,K", [(1, 256), (127, 512), (128, 256), (129, 768), (300, 1280),
                                 (1000, 2304), (2049, 512)])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_small_shapes_elementwise(fmt, N, K, M):
    q, s, ts, A = _case(fmt, 7 * N + K + M, N, K, M)
    gpu = gemm_gpu(fmt, q, s, ts, A).cpu().numpy()
    ref, bnd = oracle.gemm_w4(ORACLE_FMT[fmt], N, K, q, s, ts, A)
    assert_gemm_close(gpu, ref, bnd, f"{fmt} N={N} K={K} M={M}")


@pytest.mark.parametrize("fmt", ["nvfp4", "q4_0"])
@pytest.mark.parametrize("N,K,M", [(5000, 5376, 8), (20000, 5376, 1), (3000, 1792, 3),
                                   (9000, 3328, 2)])
def test_stage_counts_not_multiple_of_scale_group(fmt, N, K, M):
    """K/256 = 21, 7, 13: the last group of scale stages in a row is short, and
    with many tiles the stream-K ranges start at every stage offset."""
    q, s, ts, A = _case(fmt, N + K + M, N, K, M)
    gpu = gemm_gpu(fmt, q, s, ts, A).cpu().numpy()
    cols = np.unique(np.concatenate([np.arange(0, N, 7), [N - 1]])).astype(np.int32)
    ref, bnd = oracle.gemm_w4(ORACLE_FMT[fmt], N, K, q, s, ts, A, cols=cols)
    assert_gemm_close(gpu[:, cols], ref, bnd, f"{fmt} N={N} K={K} M={M}")


@pytest.mark.parametrize("fmt", ["nvfp4", "q4_0"])
def test_strided_activations_and_outputs(fmt):
    N, K, M = 333, 1024, 5
    q, s, ts, A = _case(fmt, 99, N, K, M)
    gpu = gemm_gpu(fmt, q, s, ts, A, lda_pad=24, ldo_pad=12)
    ref, bnd = oracle.gemm_w4(ORACLE_FMT[fmt], N, K, q, s, ts, A)
    assert_gemm_close(gpu.cpu().numpy(), ref, bnd, "strided")
    # nothing written past column N of each output row
    base = gpu.as_strided((M, N + 12), (gpu.stride(0), 1))
    assert torch.isnan(base[:, N:]).all()


def test_rows_are_independent_of_batch():
    """Row m of an M-batch equals the M=1 call on that row (identical computation)."""
    N, K = 700, 1536
    q, s, ts, A = _case("nvfp4", 5, N, K, 8)
    full = gemm_gpu("nvfp4", q, s, ts, A).cpu().numpy()
    for m in (0, 3, 7):
        one = gemm_gpu("nvfp4", q, s, ts, A[m:m + 1]).cpu().numpy()
        ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A[m:m + 1])
        assert_gemm_close(one, ref, bnd)
        assert_gemm_close(full[m:m + 1], ref, bnd)


def test_deterministic():
    N, K, M = 1100, 4096, 8
    q, s, ts, A = _case("nvfp4", 6, N, K, M)
    a = gemm_gpu("nvfp4", q, s, ts, A).cpu().numpy()
    b = gemm_gpu("nvfp4", q, s, ts, A).cpu().numpy()
    assert np.array_equal(a, b)


def test_extreme_activation_magnitudes():
    """Rows whose scale is far outside fp16 (the per-row power-of-two pre-scale)."""
    N, K = 200, 512
    q, s, ts = synth.linear(8, N, K, "nvfp4")
    g = synth.rng(9)
    x = g.standard_normal((4, K)).astype(np.float32)
    x[0] *= 1e30
    x[1] *= 1e-30
    x[2, :] = 0.0
    x[3] *= 3e5
    A = synth.bf16_bits(x)
    gpu = gemm_gpu("nvfp4", q, s, ts, A).cpu().numpy()
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A)
    assert_gemm_close(gpu, ref, bnd, "extreme")
    assert np.all(gpu[2] == 0.0)


@pytest.mark.parametrize("fmt", ["nvfp4", "q4_0"])
@pytest.mark.parametrize("name", list(DENSE))
def test_dense_layer_full_size_sampled(fmt, name):
    """Dense-27B-like layer, full sizes, M in {1, 2, 4, 8}: sampled columns."""
    N, K = DENSE[name]
    seed = 100 + list(DENSE).index(name)
    q, s, ts = synth.linear(seed, N, K, fmt)
    g = synth.rng(seed + 500)
    cols = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, 96)])).astype(np.int32)
    A8 = synth.activations(g, 8, K)
    for M in (1, 2, 4, 8):
        A = A8[:M]
        gpu = gemm_gpu(fmt, q, s, ts, A).cpu().numpy()
        ref, bnd = oracle.gemm_w4(ORACLE_FMT[fmt], N, K, q, s, ts, A, cols=cols)
        assert_gemm_close(gpu[:, cols], ref, bnd, f"{fmt} {name} M={M}")


@pytest.mark.parametrize("N,K,M", [(1000, 1024, 8), (5000, 768, 3), (300, 256, 1)])
def test_fused_argmax_small(N, K, M):
    q, s, ts, A = _case("nvfp4", N + M, N, K, M)
    am = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    gpu = gemm_gpu("nvfp4", q, s, ts, A, row_argmax=am).cpu().numpy()
    am = am.cpu().numpy()
    for m in range(M):
        assert am[m] == oracle.argmax_f32(gpu[m])


def test_lm_head_full_size_sampled_and_fused_argmax():
    """LM head 5376 -> 262144 nvfp4, M = 8: sampled columns against the oracle,
    the fused argmax bit-exact against the oracle's argmax of the GPU logits,
    and against the fp64 oracle logits unless the top-2 gap is within the
    GEMM error bound (then the row is a tie within tolerance)."""
    N, K, M = 262144, 5376, 8
    q, s, ts = synth.linear(2, N, K, "nvfp4")
    A = synth.activations(synth.rng(2), M, K)
    am = torch.empty((M,), dtype=torch.int32, device="cuda")
    gpu = gemm_gpu("nvfp4", q, s, ts, A, row_argmax=am).cpu().numpy()
    am = am.cpu().numpy()
    g = synth.rng(77)
    cols = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, 128)]))
    for m in range(M):
        top = np.argsort(-gpu[m], kind="stable")[:4]
        cols = np.union1d(cols, top)
    cols = cols.astype(np.int32)
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A, cols=cols)
    assert_gemm_close(gpu[:, cols], ref, bnd, "lm head")
    for m in range(M):
        assert am[m] == oracle.argmax_f32(gpu[m])
        # the fp64 argmax over the candidate columns equals the GPU's unless tied
        j = int(np.argmax(ref[m]))
        if cols[j] != am[m]:
            k = int(np.searchsorted(cols, am[m]))
            gap = ref[m, j] - ref[m, k]
            assert gap <= 2e-3 * max(bnd[m, j], bnd[m, k]), (m, cols[j], am[m], gap)


def test_prepared_gemm_matches_plain_call():
    N, K, M = 900, 1536, 6
    q, s, ts, A = _case("nvfp4", 12, N, K, M)
    qd, sd = upload_weight(q, s, "nvfp4")
    Ad = bf16_dev(A)
    plain = vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad)
    prep = vw4.PreparedGemm(vw4.FMT_NVFP4, qd, sd, ts, M_max=8)
    out = torch.empty_like(plain)
    prep(Ad, out)
    torch.cuda.synchronize()
    assert torch.equal(plain, out)


def test_q4_0_from_blocks_matches_split_layout():
    N, K = 64, 512
    qs, d, _ = synth.linear(11, N, K, "q4_0")
    nb = K // 32
    rec = np.zeros((N, nb, 18), np.uint8)
    rec[:, :, 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    rec[:, :, 2:] = qs.reshape(N, nb, 16)
    q2, d2 = vw4.vw4_q4_0_from_blocks(torch.from_numpy(rec.reshape(-1)).cuda(), N, K)
    torch.cuda.synchronize()
    assert np.array_equal(q2.cpu().numpy(), qs)
    assert np.array_equal(d2.cpu().numpy().view(np.uint16), d.view(np.uint16))


def test_argument_errors_are_synchronous():
    q, s, ts, A = _case("nvfp4", 1, 128, 256, 2)
    qd, sd = upload_weight(q, s, "nvfp4")
    Ad = bf16_dev(A)
    with pytest.raises(vw4.VW4Error) as e:
        vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, torch.cat([Ad] * 9))  # M = 18
    assert e.value.code == 1
    with pytest.raises(vw4.VW4Error) as e:
        vw4.verify_gemm_w4(vw4.FMT_Q4_0, qd, sd, 2.0, Ad)  # Q4_0 needs tensor_scale 1
    assert e.value.code == 1
    assert vw4.vw4_get_device_status() == 0


def _mixed_stage_case(tiny_exp):
    """Rows whose first 256-wide k stage holds activations of 1 on the k's
    where a chosen output column's weight is zero-coded and 2^tiny_exp * u
    (u in [1, 2), random bf16 mantissas) elsewhere; the second stage is zero.
    The large activations then add nothing to that column, whose sum|a*w|
    comes from the tiny ones alone."""
    N, K, M = 256, 512, 4
    q, s, ts = synth.linear(31, N, K, "nvfp4")
    w = oracle.dequant(oracle.FMT_NVFP4, N, K, q, s, ts)
    g = synth.rng(32)
    x = np.zeros((M, K), np.float32)
    cols = []
    for m in range(M):
        n = (37 * m + 5) % N
        cols.append(n)
        zero = w[n, :256] == 0.0
        assert zero.sum() >= 8 and (~zero).sum() >= 64
        u = (1.0 + g.random(256)).astype(np.float32) * np.float32(2.0 ** tiny_exp)
        sign = np.where(g.random(256) < 0.5, -1.0, 1.0).astype(np.float32)
        x[m, :256] = np.where(zero, np.float32(1.0), u * sign)
    return N, K, M, q, s, ts, w, synth.bf16_bits(x), np.array(cols)


def test_mixed_magnitude_stage_inside_the_exact_range():
    """Within one 256-wide k stage, activations down to 2^-31 of the stage's
    largest magnitude are represented exactly (vw4.h, verify_gemm_w4
    precision): the pass rule holds for the column the large activations do
    not reach."""
    N, K, M, q, s, ts, w, A, cols = _mixed_stage_case(-31)
    gpu = gemm_gpu("nvfp4", q, s, ts, A).cpu().numpy()
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A)
    assert_gemm_close(gpu, ref, bnd, "mixed magnitudes, exact range")
    for m, n in enumerate(cols):
        assert bnd[m, n] > 0.0 and abs(gpu[m, n] - ref[m, n]) <= 1e-3 * bnd[m, n]


@pytest.mark.parametrize("tiny_exp", [-36, -40, -60])
def test_mixed_magnitude_stage_below_the_exact_range(tiny_exp):
    """Below 2^-31 of the stage's largest magnitude an activation is rounded
    to a multiple of 2^-39 of it (or to zero): the error of every element
    stays within 1e-3 * sum|a*w| + 2^-39 * sum_k amax_stage(k) * |w_k|, the
    bound vw4.h states."""
    N, K, M, q, s, ts, w, A, cols = _mixed_stage_case(tiny_exp)
    gpu = gemm_gpu("nvfp4", q, s, ts, A).cpu().numpy()
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A)
    a = np.array([[oracle.bf16(int(b)) for b in row] for row in A])
    amax = np.abs(a).reshape(M, K // 256, 256).max(axis=2)          # [M, stages]
    amax_k = np.repeat(amax, 256, axis=1)                            # [M, K]
    extra = 2.0 ** -39 * (amax_k @ np.abs(w).T)                      # [M, N]
    err = np.abs(gpu.astype(np.float64) - ref)
    assert np.all(err <= 1e-3 * bnd + extra), float(np.max(err - 1e-3 * bnd - extra))


@pytest.mark.parametrize("fmt,K", [("nvfp4", 272), ("nvfp4", 1040), ("nvfp4", 5136),
                                   ("q4_0", 288), ("q4_0", 1056), ("q4_0", 5152)])
@pytest.mark.parametrize("N,M", [(300, 8), (5000, 1), (1000, 12)])
def test_k_not_a_multiple_of_256(fmt, K, N, M):
    """K a multiple of the format's block (16 nvfp4, 32 Q4_0) but not of 256:
    the weights are padded to whole stages in the workspace, the activations
    read as zero past K; element by element against the oracle."""
    q, s, ts, A = _case(fmt, 3 * K + N + M, N, K, M)
    gpu = gemm_gpu(fmt, q, s, ts, A).cpu().numpy()
    ref, bnd = oracle.gemm_w4(ORACLE_FMT[fmt], N, K, q, s, ts, A)
    assert_gemm_close(gpu, ref, bnd, f"{fmt} N={N} K={K} M={M}")


def test_k_not_a_multiple_of_256_fused_argmax_and_greedy():
    N, K, B, Kd = 20000, 1040, 1, 7
    M = B * (Kd + 1)
    q, s, ts, A = _case("nvfp4", 77, N, K, M)
    qd, sd = upload_weight(q, s, "nvfp4")
    Ad = bf16_dev(A)
    am = torch.empty((M,), dtype=torch.int32, device="cuda")
    logits = vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, row_argmax=am)
    lg = logits.cpu().numpy()
    assert np.array_equal(am.cpu().numpy(), lg.argmax(axis=1))
    drafts = synth.greedy_drafts(synth.rng(78), am.cpu().numpy()[None, :Kd], N)
    tok, ln = vw4.verify_greedy_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, torch.from_numpy(drafts).cuda())
    torch.cuda.synchronize()
    rt, rl, _ = oracle.accept_greedy(lg.reshape(B, Kd + 1, N), drafts)
    assert np.array_equal(tok.cpu().numpy(), rt) and np.array_equal(ln.cpu().numpy(), rl)
    assert vw4.vw4_get_device_status() == 0
