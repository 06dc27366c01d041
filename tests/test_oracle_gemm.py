"""Pins of the oracle GEMM and MoE against independent computations.

* brute force: an independent dequantizer (golden E2M1 table, torch's e4m3
  cast, numpy's fp16) and exact rational sums on tiny shapes;
* M = 1 equals a numpy fp64 GEMV on that independently dequantized matrix;
* each row of an M-batch equals its own single-row call ("identical
  computation": batching changes nothing);
* a one-hot activation returns the exact dequantized column;
* the result is linear in the tensor scale;
* MoE equals the dense oracle per routed pair, summed with the gates.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden_lines

E2M1 = {int(c, 16): float(v) for c, v in golden_lines("e2m1_ocp_mx_v1.txt")}


def indep_dequant(fmt, N, K, q, scales, ts):
    """Table/library based decoding, written apart from the oracle's formulas."""
    w = np.zeros((N, K), np.float64)
    if fmt == oracle.FMT_NVFP4:
        sv = torch.from_numpy(np.ascontiguousarray(scales, np.uint8)).view(
            torch.float8_e4m3fn).to(torch.float64).numpy()
        for n in range(N):
            for k in range(K):
                byte = int(q[n, k // 2])
                code = (byte >> 4) if (k % 2) else (byte & 15)
                w[n, k] = E2M1[code] * sv[n, k // 16] * ts
    else:
        dv = np.asarray(scales, np.float16).astype(np.float64)
        for n in range(N):
            for b in range(K // 32):
                for j in range(16):
                    byte = int(q[n, b * 16 + j])
                    w[n, b * 32 + j] = ((byte & 15) - 8) * dv[n, b]
                    w[n, b * 32 + j + 16] = ((byte >> 4) - 8) * dv[n, b]
    return w


def bits_to_f64(a_bits):
    return torch.from_numpy(a_bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def make(fmt, seed, N, K, M):
    g = synth.rng(seed)
    w = synth.normal_weights(g, N, K)
    if fmt == oracle.FMT_NVFP4:
        q, s, ts = synth.quantize_nvfp4(w)
    else:
        (q, s), ts = synth.quantize_q4_0(w), 1.0
    A = synth.activations(g, M, K)
    return q, s, ts, A


@pytest.mark.parametrize("fmt", [oracle.FMT_NVFP4, oracle.FMT_Q4_0])
@pytest.mark.parametrize("N,K,M", [(1, 32, 1), (3, 32, 8), (4, 64, 5), (2, 96, 3)])
def test_brute_force_exact_sum(fmt, N, K, M):
    q, s, ts, A = make(fmt, 10 + N + K + M, N, K, M)
    out, bound = oracle.gemm_w4(fmt, N, K, q, s, ts, A)
    w = indep_dequant(fmt, N, K, q, s, ts)
    a = bits_to_f64(A)
    for m in range(M):
        for n in range(N):
            exact = sum((Fraction(a[m, k]) * Fraction(w[n, k]) for k in range(K)), Fraction(0))
            mag = sum((abs(Fraction(a[m, k]) * Fraction(w[n, k])) for k in range(K)), Fraction(0))
            # fp64 sequential sum: error <= K * 2^-53 * sum|terms|
            tol = float(mag) * K * 2.0 ** -52 + 1e-300
            assert abs(out[m, n] - float(exact)) <= tol
            assert abs(bound[m, n] - float(mag)) <= tol


@pytest.mark.parametrize("fmt", [oracle.FMT_NVFP4, oracle.FMT_Q4_0])
def test_m1_equals_numpy_gemv(fmt):
    N, K = 40, 256
    q, s, ts, A = make(fmt, 21, N, K, 1)
    out, _ = oracle.gemm_w4(fmt, N, K, q, s, ts, A)
    w = indep_dequant(fmt, N, K, q, s, ts)
    ref = w @ bits_to_f64(A)[0]
    assert np.allclose(out[0], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", [oracle.FMT_NVFP4, oracle.FMT_Q4_0])
def test_rows_of_batch_equal_single_row_calls(fmt):
    N, K, M = 24, 512, 8
    q, s, ts, A = make(fmt, 22, N, K, M)
    out, bound = oracle.gemm_w4(fmt, N, K, q, s, ts, A)
    for m in range(M):
        o1, b1 = oracle.gemm_w4(fmt, N, K, q, s, ts, A[m:m + 1])
        assert np.array_equal(o1[0], out[m]) and np.array_equal(b1[0], bound[m])


@pytest.mark.parametrize("fmt", [oracle.FMT_NVFP4, oracle.FMT_Q4_0])
def test_one_hot_activation_returns_column(fmt):
    N, K = 12, 128
    q, s, ts, _ = make(fmt, 23, N, K, 1)
    w = indep_dequant(fmt, N, K, q, s, ts)
    for k in (0, 1, 15, 16, 77, K - 1):
        A = np.zeros((1, K), np.uint16)
        A[0, k] = 0x3F80  # bf16 1.0
        out, _ = oracle.gemm_w4(fmt, N, K, q, s, ts, A)
        assert np.array_equal(out[0], w[:, k])


def test_linear_in_tensor_scale():
    N, K, M = 16, 256, 4
    q, s, ts, A = make(oracle.FMT_NVFP4, 24, N, K, M)
    o1, _ = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A)
    o2, _ = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, 2.0 * ts, A)
    o3, _ = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, 3.0 * ts, A)
    assert np.array_equal(o2, 2.0 * o1)
    assert np.allclose(o3, 3.0 * o1, rtol=1e-13)


def test_column_subset_matches_full():
    N, K, M = 50, 256, 3
    q, s, ts, A = make(oracle.FMT_NVFP4, 25, N, K, M)
    full, fb = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A)
    cols = np.array([49, 0, 17, 17, 3], np.int32)
    sub, sb = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A, cols=cols)
    assert np.array_equal(sub, full[:, cols]) and np.array_equal(sb, fb[:, cols])


# ----------------------------------------------------------------------- MoE
@pytest.mark.parametrize("rows_are_pairs,combine", [(0, 0), (1, 1), (0, 1), (1, 0)])
def test_moe_equals_dense_per_pair(rows_are_pairs, combine):
    E, N, K, M, topk = 6, 20, 64, 3, 2
    g = synth.rng(30)
    w = synth.normal_weights(g, E * N, K)
    q, s, ts = synth.quantize_nvfp4(w)
    ids, gates = synth.routing(31, M, E, topk)
    A = synth.activations(g, M * topk if rows_are_pairs else M, K)
    out, bound = oracle.moe_w4(oracle.FMT_NVFP4, E, N, K, q, s, ts, A, rows_are_pairs, ids, gates,
                               M, topk, combine)
    wd = indep_dequant(oracle.FMT_NVFP4, E * N, K, q, s, ts)
    a = bits_to_f64(A)
    pair = np.zeros((M * topk, N))
    for p in range(M * topk):
        e = ids.reshape(-1)[p]
        arow = a[p] if rows_are_pairs else a[p // topk]
        pair[p] = wd[e * N:(e + 1) * N] @ arow
    if combine:
        ref = np.stack([sum(gates[m, j] * pair[m * topk + j] for j in range(topk))
                        for m in range(M)])
    else:
        ref = pair
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert np.all(bound >= np.abs(out) - 1e-12)


def test_route_sort_is_stable_counting_sort():
    ids, _ = synth.routing(32, 8, 128, 8)
    order, seg = oracle.route_sort(ids, 128)
    flat = ids.reshape(-1)
    ref = np.argsort(flat, kind="stable")
    assert np.array_equal(order, ref)
    counts = np.bincount(flat, minlength=128)
    assert np.array_equal(np.diff(seg), counts)
