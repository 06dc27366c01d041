"""GPU parity of verify_moe_w4 (segmented expert gather) against the oracle.

MoE head: 128 experts, top-8, d = 2048; each expert's gate and up projections
(2048 -> 768 each) are stored stacked as one 1536-row matrix, the down
projection is 768 -> 2048; nvfp4; M = 8 tokens with seeded top-8 routing, and
1-16 tokens (up to 128 routed pairs).
The activation between the two GEMMs (silu(gate) * up, rounded to bf16) is
computed by the test harness and fed to both sides.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decode_verification_w4_gb300 as vw4
from gpu_util import assert_gemm_close, bf16_dev

pytestmark = pytest.mark.gpu


def moe_gpu(q, s, ts, E, A_bits, rows_are_pairs, ids, gates, combine):
    out = vw4.verify_moe_w4(vw4.FMT_NVFP4, torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(),
                            ts, E, bf16_dev(A_bits), rows_are_pairs,
                            torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda(),
                            torch.from_numpy(np.ascontiguousarray(gates, np.float32)).cuda(),
                            combine)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.fixture(scope="module")
def moe_head():
    E, d, f = 128, 2048, 768
    gu = synth.linear(200, E * 2 * f, d, "nvfp4")
    dn = synth.linear(201, E * d, f, "nvfp4")
    return E, d, f, gu, dn


@pytest.mark.parametrize("M", [8, 1, 3, 16, 12, 9])
def test_moe_head_full_config(moe_head, M):
    E, d, f, (qg, sg, tg), (qd, sd, tdn) = moe_head
    ids, gates = synth.routing(300 + M, M, E, 8)
    A = synth.activations(synth.rng(301 + M), M, d)
    pair = moe_gpu(qg, sg, tg, E, A, 0, ids, gates, 0)           # [M*8, 1536]
    ref, bnd = oracle.moe_w4(oracle.FMT_NVFP4, E, 2 * f, d, qg, sg, tg, A, 0, ids, gates, M, 8, 0)
    assert_gemm_close(pair, ref, bnd, "gate/up pairs")
    g, u = pair[:, :f].astype(np.float64), pair[:, f:].astype(np.float64)
    h = synth.bf16_bits((g / (1.0 + np.exp(-g)) * u).astype(np.float32))
    out = moe_gpu(qd, sd, tdn, E, h, 1, ids, gates, 1)           # [M, 2048]
    ref, bnd = oracle.moe_w4(oracle.FMT_NVFP4, E, d, f, qd, sd, tdn, h, 1, ids, gates, M, 8, 1)
    assert_gemm_close(out, ref, bnd, "down combine")


@pytest.mark.parametrize("rows_are_pairs,combine", [(0, 0), (1, 1), (0, 1), (1, 0)])
def test_moe_small_modes(rows_are_pairs, combine):
    E, N, K, M, topk = 5, 300, 512, 4, 3
    q, s, ts = synth.linear(210, E * N, K, "nvfp4")
    ids, gates = synth.routing(211, M, E, topk)
    A = synth.activations(synth.rng(212), M * topk if rows_are_pairs else M, K)
    out = moe_gpu(q, s, ts, E, A, rows_are_pairs, ids, gates, combine)
    ref, bnd = oracle.moe_w4(oracle.FMT_NVFP4, E, N, K, q, s, ts, A, rows_are_pairs, ids, gates, M,
                             topk, combine)
    assert_gemm_close(out, ref, bnd, "moe small")


def test_moe_same_expert_for_every_token_and_bad_ids():
    """Nine pairs on one expert split into two segments; an invalid expert id
    contributes zeros and sets the status bit."""
    E, N, K, M, topk = 3, 256, 256, 8, 2
    q, s, ts = synth.linear(220, E * N, K, "nvfp4")
    ids = np.zeros((M, topk), np.int32)
    ids[:, 1] = 1
    ids[3, 1] = 0   # token 3 routes to expert 0 twice (still a valid pair)
    ids[5, 0] = 7   # invalid
    gates = np.full((M, topk), 0.5, np.float32)
    A = synth.activations(synth.rng(221), M, K)
    vw4.vw4_get_device_status()
    out = moe_gpu(q, s, ts, E, A, 0, ids, gates, 0)
    assert vw4.vw4_get_device_status() & vw4.DEV_BAD_EXPERT_ID
    ref, bnd = oracle.moe_w4(oracle.FMT_NVFP4, E, N, K, q, s, ts, A, 0, ids, gates, M, topk, 0)
    assert_gemm_close(out, ref, bnd, "moe shared expert")
    assert np.all(out[5 * topk] == 0.0)


def test_moe_sixteen_tokens_crowded_expert():
    """16 tokens x top-8 = 128 pairs, a third of them on one expert: that
    expert's pairs fill several 8-row segments (each streams its weights),
    the rest spread over the others; the combine sums the gates in order."""
    E, N, K, M, topk = 16, 384, 512, 16, 8
    q, s, ts = synth.linear(230, E * N, K, "nvfp4")
    g = synth.rng(231)
    ids = np.stack([g.permutation(E)[:topk] for _ in range(M)]).astype(np.int32)
    ids[:6, 0] = 5
    ids[6:12, 2] = 5
    for m in range(M):   # keep each token's experts distinct
        row = list(dict.fromkeys(ids[m].tolist()))
        rest = [e for e in g.permutation(E).tolist() if e not in row]
        ids[m] = (row + rest)[:topk]
    gates = g.random((M, topk)).astype(np.float32)
    A = synth.activations(synth.rng(232), M * topk, K)
    out = moe_gpu(q, s, ts, E, A, 1, ids, gates, 1)
    ref, bnd = oracle.moe_w4(oracle.FMT_NVFP4, E, N, K, q, s, ts, A, 1, ids, gates, M, topk, 1)
    assert_gemm_close(out, ref, bnd, "moe 16 tokens, crowded expert")
    assert vw4.vw4_get_device_status() == 0
