"""GPU parity of accept_greedy against the oracle (bit-exact ids and lengths)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decode_verification_w4_gb300 as vw4

pytestmark = pytest.mark.gpu


def run(target, drafts, argmax=None):
    t = torch.from_numpy(np.ascontiguousarray(target)).cuda()
    d = torch.from_numpy(np.ascontiguousarray(drafts, np.int32)).cuda()
    am = None if argmax is None else torch.from_numpy(np.ascontiguousarray(argmax, np.int32)).cuda()
    tok, ln = vw4.accept_greedy(None if argmax is not None else t, d, target_argmax=am,
                                B=target.shape[0], V=target.shape[2])
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ln.cpu().numpy()


def test_tiny_config_greedy():
    """Greedy accept of K=3 drafts on fp32 N(0,1) logits, vocab 1024, seed 0."""
    g = synth.rng(0)
    target = synth.logits(g, (1, 4, 1024), 1.0)
    am = np.array([[oracle.argmax_f32(target[0, i]) for i in range(3)]])
    drafts = synth.greedy_drafts(g, am, 1024)
    tok, ln = run(target, drafts)
    rt, rl, _ = oracle.accept_greedy(target, drafts)
    assert np.array_equal(tok, rt) and np.array_equal(ln, rl)


@pytest.mark.parametrize("B,Kd,V", [(1, 0, 5), (7, 1, 1000), (33, 4, 4097), (256, 8, 151936),
                                    (3, 8, 7)])
def test_random_cases(B, Kd, V):
    g = synth.rng(B * 100 + Kd)
    target = synth.logits(g, (B, Kd + 1, V), 1.0)
    am = np.array([[oracle.argmax_f32(target[b, i]) for i in range(Kd)] for b in range(B)],
                  np.int32).reshape(B, Kd)
    drafts = synth.greedy_drafts(g, am, V) if Kd else np.zeros((B, 0), np.int32)
    tok, ln = run(target, drafts)
    rt, rl, _ = oracle.accept_greedy(target, drafts)
    assert np.array_equal(tok, rt) and np.array_equal(ln, rl)


def test_ties_nan_and_bad_ids():
    V = 64
    target = np.zeros((4, 3, V), np.float32)
    target[0, :, 5] = 1.0
    target[0, :, 9] = 1.0          # tie -> 5
    target[1, :, :] = np.nan       # all NaN -> 0
    target[2, :, 3] = np.nan
    target[2, :, 7] = -1.0         # NaN never wins; zeros elsewhere -> 0
    target[2, :, 0] = -2.0         # now index 1 is the first zero
    target[3, :, 60] = np.inf
    drafts = np.array([[5, 5], [0, 1], [1, 99], [60, -3]], np.int32)
    vw4.vw4_get_device_status()
    tok, ln = run(target, drafts)
    rt, rl, bad = oracle.accept_greedy(target, drafts)
    assert np.array_equal(tok, rt) and np.array_equal(ln, rl)
    assert bad == 2
    assert vw4.vw4_get_device_status() & vw4.DEV_BAD_DRAFT_ID


def test_precomputed_argmax_path():
    g = synth.rng(4)
    B, Kd, V = 9, 5, 300
    target = synth.logits(g, (B, Kd + 1, V), 1.0)
    am = np.array([[oracle.argmax_f32(target[b, i]) for i in range(Kd + 1)] for b in range(B)],
                  np.int32)
    drafts = synth.greedy_drafts(g, am[:, :Kd], V)
    tok, ln = run(target, drafts, argmax=am)
    rt, rl, _ = oracle.accept_greedy(target, drafts)
    assert np.array_equal(tok, rt) and np.array_equal(ln, rl)


def test_lm_head_fused_path_end_to_end():
    """LM-head verify + fused accept, at a reduced vocabulary: GEMM with fused
    argmax feeding accept_greedy, against the oracle applied to the GPU logits."""
    N, K, M = 20000, 1024, 8
    q, s, ts = synth.linear(3, N, K, "nvfp4")
    A = synth.activations(synth.rng(3), M, K)
    qd = torch.from_numpy(q).cuda()
    sd = torch.from_numpy(s).cuda()
    Ad = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
    am = torch.empty((M,), dtype=torch.int32, device="cuda")
    logits = vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, row_argmax=am)
    amh = am.cpu().numpy()
    drafts = synth.greedy_drafts(synth.rng(31), amh[None, :M - 1], N)
    d = torch.from_numpy(drafts).cuda()
    tok, ln = vw4.accept_greedy(None, d, target_argmax=am.view(1, M), B=1, V=N)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()[None]
    rt, rl, _ = oracle.accept_greedy(lg, drafts)
    assert np.array_equal(tok.cpu().numpy(), rt) and np.array_equal(ln.cpu().numpy(), rl)


@pytest.mark.parametrize("N,K,B,Kd", [(20000, 1024, 1, 7), (20000, 1024, 2, 3), (5000, 2048, 4, 1),
                                      (3000, 512, 3, 0), (70000, 768, 1, 7),
                                      # 9..16 verify rows: two n-tiles per weight fragment
                                      (20000, 1024, 2, 7), (5000, 2048, 4, 3), (70000, 768, 8, 1),
                                      (3000, 512, 5, 2)])
def test_verify_greedy_one_launch(N, K, B, Kd):
    """GEMM, row argmax and greedy accept in one launch: the committed run
    equals the oracle's greedy accept over the GPU's own fp32 logits (which
    the same call writes when asked), and the call without logits commits the
    same run."""
    M = B * (Kd + 1)
    q, s, ts = synth.linear(N + K, N, K, "nvfp4")
    A = synth.activations(synth.rng(K), M, K)
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    Ad = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
    am = torch.empty((M,), dtype=torch.int32, device="cuda")
    vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, row_argmax=am)
    amh = am.cpu().numpy().reshape(B, Kd + 1)
    drafts = synth.greedy_drafts(synth.rng(N), amh[:, :Kd], N) if Kd else \
        np.zeros((B, 0), np.int32)
    d = torch.from_numpy(np.ascontiguousarray(drafts, np.int32)).cuda()
    logits = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    tok, ln = vw4.verify_greedy_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, d, out=logits)
    tok2, ln2 = vw4.verify_greedy_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, d)
    torch.cuda.synchronize()
    assert vw4.vw4_get_device_status() == 0
    lg = logits.cpu().numpy().reshape(B, Kd + 1, N)
    rt, rl, _ = oracle.accept_greedy(lg, drafts)
    assert np.array_equal(tok.cpu().numpy(), rt) and np.array_equal(ln.cpu().numpy(), rl)
    assert np.array_equal(tok2.cpu().numpy(), rt) and np.array_equal(ln2.cpu().numpy(), rl)
    # the logits it wrote are the verify GEMM's
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A,
                              cols=np.arange(0, N, 97, dtype=np.int32))
    assert np.all(np.abs(lg.reshape(M, N)[:, ::97] - ref) <= 1e-3 * bnd)


def test_verify_greedy_bad_draft_ids():
    N, K, B, Kd = 4000, 512, 2, 3
    q, s, ts = synth.linear(9, N, K, "nvfp4")
    A = synth.activations(synth.rng(9), B * (Kd + 1), K)
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    Ad = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
    logits = vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad)
    lg = logits.cpu().numpy().reshape(B, Kd + 1, N)
    am = lg.argmax(axis=-1).astype(np.int32)
    drafts = am[:, :Kd].copy()
    drafts[0, 1] = N          # out of range after one agreeing position
    drafts[1, 0] = -5
    vw4.vw4_get_device_status()
    tok, ln = vw4.verify_greedy_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad,
                                   torch.from_numpy(drafts).cuda())
    torch.cuda.synchronize()
    assert vw4.vw4_get_device_status() & vw4.DEV_BAD_DRAFT_ID
    rt, rl, _ = oracle.accept_greedy(lg, drafts)
    assert np.array_equal(tok.cpu().numpy(), rt) and np.array_equal(ln.cpu().numpy(), rl)


def test_verify_greedy_lm_head_full_size():
    """LM-head verify + fused accept at its full size, through the timed path:
    W 5376 -> 262144 nvfp4 N(0, 0.02), M = 8 bf16 hidden rows (B = 1, 7
    drafts), drafts agreeing with the oracle's fp64 argmax with probability
    0.8 (seeded).  verify_greedy_w4 runs the GEMM, the row argmax and the
    greedy accept in one launch; the committed run must equal the oracle's
    greedy accept over the GPU's own fp32 logits (which the same call writes),
    every logit must be within 1e-3 * sum|a*w| of the oracle's fp64 value, and
    the GPU argmax of each row must be the fp64 one unless the two lie within
    the GEMM error bound of each other (a tie within tolerance)."""
    N, K, B, Kd = 262144, 5376, 1, 7
    M = B * (Kd + 1)
    q, s, ts = synth.linear(2, N, K, "nvfp4")
    A = synth.activations(synth.rng(2), M, K)
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A)   # fp64, every column
    ref_am = np.array([int(np.argmax(ref[m])) for m in range(M)])
    drafts = synth.greedy_drafts(synth.rng(333), ref_am[None, :Kd], N)
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    Ad = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
    d = torch.from_numpy(np.ascontiguousarray(drafts, np.int32)).cuda()
    logits = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    tok, ln = vw4.verify_greedy_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, d, out=logits)
    tok2, ln2 = vw4.verify_greedy_w4(vw4.FMT_NVFP4, qd, sd, ts, Ad, d)   # no logits written
    torch.cuda.synchronize()
    assert vw4.vw4_get_device_status() == 0
    lg = logits.cpu().numpy()
    tok, ln = tok.cpu().numpy(), ln.cpu().numpy()
    rt, rl, _ = oracle.accept_greedy(lg.reshape(B, Kd + 1, N), drafts)
    assert np.array_equal(tok, rt) and np.array_equal(ln, rl), (tok, rt, ln, rl)
    assert np.array_equal(tok2.cpu().numpy(), rt) and np.array_equal(ln2.cpu().numpy(), rl)
    err = np.abs(lg.astype(np.float64) - ref)
    assert np.all(err <= 1e-3 * bnd), float(np.max(err / bnd))
    for m in range(M):
        g = oracle.argmax_f32(lg[m])
        if g != ref_am[m]:
            gap = ref[m, ref_am[m]] - ref[m, g]
            assert gap <= 2e-3 * max(bnd[m, ref_am[m]], bnd[m, g]), (m, g, ref_am[m], gap)
    # the accept agreed with at least the drafts that match the GPU argmax
    assert 1 <= ln[0] <= Kd + 1
