"""Pins of the oracle's format decoders against sources other than itself.

E2M1 against the OCP MX v1.0 table (golden file), E4M3 against torch's
float8_e4m3fn cast, fp16 against numpy's float16, bf16 against torch's
bfloat16, and both 4-bit layouts against an independent encoder (the input
synthesizer) through the quantization error bound: a swapped nibble order,
a wrong block index or a dropped scale would blow the bound.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden_lines


def test_e2m1_all_codes_match_ocp_table():
    table = {int(c, 16): float(v) for c, v in golden_lines("e2m1_ocp_mx_v1.txt")}
    assert len(table) == 16
    for code, val in table.items():
        got = oracle.e2m1(code)
        assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val), code


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3(c)
        if np.isnan(ref[c]):
            assert np.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])
    assert np.isnan(oracle.e4m3(0x7F)) and np.isnan(oracle.e4m3(0xFF))
    assert oracle.e4m3(0x7E) == 448.0 and oracle.e4m3(0x01) == 2.0 ** -9


def test_f16_all_codes_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for b in range(0, 65536, 7):
        got = oracle.f16(b)
        if np.isnan(ref[b]):
            assert np.isnan(got)
        else:
            assert got == ref[b], b


def test_bf16_matches_torch():
    g = np.random.default_rng(1)
    bits = g.integers(0, 65536, 4000).astype(np.int64)
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b, r in zip(bits, ref):
        got = oracle.bf16(int(b))
        assert (np.isnan(got) and np.isnan(r)) or got == r


@pytest.mark.parametrize("N,K", [(7, 64), (33, 256), (5, 1024)])
def test_nvfp4_layout_round_trip_within_quantization_bound(N, K):
    g = synth.rng(3)
    w = synth.normal_weights(g, N, K)
    Wq, S, ts = synth.quantize_nvfp4(w)
    dq = oracle.dequant(oracle.FMT_NVFP4, N, K, Wq, S, ts)
    # each block's step is at most 2 * scale (E2M1 spacing at the top is 2)
    scale = np.array([[oracle.e4m3(int(c)) for c in row] for row in S]) * ts
    step = np.repeat(scale, 16, axis=1)
    err = np.abs(dq - w.astype(np.float64))
    assert np.all(err <= step * 1.0 + 1e-12), float(np.max(err / step))
    # the codes really are used: dequantized values correlate with the input
    assert np.corrcoef(dq.ravel(), w.ravel())[0, 1] > 0.95


def test_nvfp4_nibble_order_and_block_index():
    # row 0: byte i = (code_hi << 4) | code_lo; element 2i is the low nibble
    K = 32
    Wq = np.zeros((1, K // 2), np.uint8)
    Wq[0, 0] = 0x71   # elements 0 -> 0.5, 1 -> 6.0
    Wq[0, 8] = 0x0A   # element 16 -> -1.0 (second scale block)
    S = np.zeros((1, K // 16), np.uint8)
    S[0, 0] = 0x38    # e4m3 1.0
    S[0, 1] = 0x40    # e4m3 2.0
    dq = oracle.dequant(oracle.FMT_NVFP4, 1, K, Wq, S, 0.5)
    expect = np.zeros(K)
    expect[0], expect[1], expect[16] = 0.25, 3.0, -1.0
    assert np.array_equal(dq[0], expect)


@pytest.mark.parametrize("N,K", [(9, 64), (16, 512)])
def test_q4_0_layout_round_trip_within_quantization_bound(N, K):
    g = synth.rng(4)
    w = synth.normal_weights(g, N, K)
    qs, d = synth.quantize_q4_0(w)
    dq = oracle.dequant(oracle.FMT_Q4_0, N, K, qs, d)
    dv = np.repeat(np.abs(d.astype(np.float64)), 32, axis=1)
    err = np.abs(dq - w.astype(np.float64))
    # rounding to the grid is within d/2 except at the clipped end (q = 15
    # stands for +8d), which is within d; plus the fp16 rounding of d
    assert np.all(err <= dv * (1.0 + 8 * 2.0 ** -10) + 1e-12)
    assert np.mean(err <= dv * (0.5 + 8 * 2.0 ** -10) + 1e-12) > 0.95
    assert np.corrcoef(dq.ravel(), w.ravel())[0, 1] > 0.95


def test_q4_0_in_block_order():
    K = 64
    qs = np.full((1, K // 2), 0x88, np.uint8)  # all zero weights
    qs[0, 0] = 0xF0 | 0x09   # element 0 -> (9-8), element 16 -> (15-8)
    qs[0, 16 + 3] = 0x0A | 0x30  # block 1: element 32+3 -> 2, element 32+19 -> -5
    d = np.array([[0.5, 2.0]], np.float16)
    dq = oracle.dequant(oracle.FMT_Q4_0, 1, K, qs, d)
    expect = np.zeros(K)
    expect[0], expect[16], expect[35], expect[51] = 0.5, 3.5, 4.0, -10.0
    assert np.array_equal(dq[0], expect)
