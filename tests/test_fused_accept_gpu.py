"""The sampled accept fed by the verify GEMM (LM-head verify + fused accept).

The pages' engine runs drafting, sampling and verification on the GPU in one
pass ("Faster Gemma 4 on MLX with multi-token prediction"), and sampled MTP
reuses the target distribution for the acceptance, residual and bonus draws
(Ollama's mtp.go commit log, "rework the MLX sampler").  Here the verify
GEMM writes, next to the logits, the largest of every 16 consecutive outputs
of each row, and accept_rejection_blockmax takes the accept's row maxima and
segment maxima from them instead of reading the rows for them.

Checked against the oracle on the GPU's own logits: the block maxima element
by element (exact), the logits within 1e-3 * sum|a*w|, and the committed ids
and lengths bit for bit; and against accept_rejection on the same logits
(identical ids, identical row records)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decode_verification_w4_gb300 as vw4

pytestmark = pytest.mark.gpu


def block_max_ref(x):
    """Largest of every 16 consecutive entries of each row (NaN as -inf)."""
    M, N = x.shape
    nb = (N + 15) // 16
    pad = np.full((M, nb * 16), -np.inf, np.float32)
    pad[:, :N] = np.where(np.isnan(x), -np.inf, x)
    return pad.reshape(M, nb, 16).max(axis=2)


def head_logits(q, sd_q, ts, A):
    """Logits and block maxima of hidden rows A through the shared head."""
    qd, sd = sd_q
    Ad = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
    out, bm = vw4.verify_gemm_w4_blockmax(vw4.FMT_NVFP4, qd, sd, ts, Ad)
    torch.cuda.synchronize()
    return out, bm


@pytest.mark.parametrize("N,K,B,Kd,top_k,min_p", [
    (20000, 1024, 2, 3, 0, 0.0), (20001, 768, 1, 7, 0, 0.0), (5000, 2048, 4, 1, 40, 0.05),
    (70000, 512, 2, 7, 0, 0.0), (3000, 256, 5, 2, 0, 0.1)])
def test_fused_sampled_accept_matches_oracle(N, K, B, Kd, top_k, min_p):
    M = B * (Kd + 1)
    q, s, ts = synth.linear(N + K, N, K, "nvfp4")
    wd = (torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda())
    A_t = synth.activations(synth.rng(K + 1), M, K)            # verify rows
    A_d = synth.activations(synth.rng(K + 2), B * Kd, K) if Kd else None   # drafter rows
    tl, tbm = head_logits(q, wd, ts, A_t)
    lg = tl.cpu().numpy()
    # the block maxima are exact maxima of the logits the same launch wrote
    assert np.array_equal(tbm.cpu().numpy(), block_max_ref(lg))
    cols = np.unique(np.concatenate([[0, N - 1], synth.rng(3).integers(0, N, 64)])).astype(
        np.int32)
    ref, bnd = oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A_t, cols=cols)
    assert np.all(np.abs(lg[:, cols] - ref) <= 1e-3 * bnd)
    if Kd:
        dl, dbm = head_logits(q, wd, ts, A_d)
        dlg = dl.cpu().numpy()
        assert np.array_equal(dbm.cpu().numpy(), block_max_ref(dlg))
    else:
        dl = dbm = None
        dlg = np.zeros((B * 0, N), np.float32)
    target = lg.reshape(B, Kd + 1, N)
    draft = dlg.reshape(B, Kd, N)
    kw = dict(top_k=top_k, min_p=min_p)
    drafts = oracle.sample_drafts(draft, 0.6, 0.95, 9, 1 << 32, **kw) if Kd else \
        np.zeros((B, 0), np.int32)
    x = torch.from_numpy(np.ascontiguousarray(drafts, np.int32)).cuda()
    t3 = tl.view(B, Kd + 1, N)
    d3 = dl.view(B, Kd, N) if Kd else None
    ws = vw4.Workspace()
    tok, ln = vw4.accept_rejection_blockmax(t3, tbm, d3, dbm, x, 0.6, 0.95, 9, 0, workspace=ws, **kw)
    rec_fused = vw4.vw4_rejection_row_records(ws, B, Kd, N).cpu().numpy().copy()
    tok2, ln2 = vw4.accept_rejection(t3, d3, x, 0.6, 0.95, 9, 0, workspace=ws, **kw)
    rec_plain = vw4.vw4_rejection_row_records(ws, B, Kd, N).cpu().numpy()
    torch.cuda.synchronize()
    assert vw4.vw4_get_device_status() == 0
    rt, rl, _ = oracle.accept_rejection(target, draft, drafts, 0.6, 0.95, 9, 0, **kw)
    assert np.array_equal(ln.cpu().numpy(), rl) and np.array_equal(tok.cpu().numpy(), rt)
    assert np.array_equal(ln2.cpu().numpy(), rl) and np.array_equal(tok2.cpu().numpy(), rt)
    # every row record equal, the row max up to the sign of a zero
    f = rec_fused.reshape(-1).view(np.dtype(vw4.ROW_RECORD_DTYPE))
    p = rec_plain.reshape(-1).view(np.dtype(vw4.ROW_RECORD_DTYPE))
    assert np.array_equal(f["max"], p["max"])
    for name in ("cut", "tau", "kept_sum", "topk_key", "topk_idx"):
        assert np.array_equal(f[name], p[name]), name


def test_fused_sampled_accept_lm_head_full_size():
    """W 5376 -> 262144 nvfp4, B = 1 sequence with 7 drafts: the 8 verify rows
    through verify_gemm_w4_blockmax, the 7 draft rows through the same head,
    drafts sampled from the draft rows; the fused accept against the oracle
    on the GPU logits (T = 0.6, top_p = 0.95)."""
    N, K, B, Kd = 262144, 5376, 1, 7
    q, s, ts = synth.linear(2, N, K, "nvfp4")
    wd = (torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda())
    tl, tbm = head_logits(q, wd, ts, synth.activations(synth.rng(2), B * (Kd + 1), K))
    dl, dbm = head_logits(q, wd, ts, synth.activations(synth.rng(22), B * Kd, K))
    lg, dlg = tl.cpu().numpy(), dl.cpu().numpy()
    assert np.array_equal(tbm.cpu().numpy(), block_max_ref(lg))
    assert np.array_equal(dbm.cpu().numpy(), block_max_ref(dlg))
    target, draft = lg.reshape(B, Kd + 1, N), dlg.reshape(B, Kd, N)
    for seed in (4, 5, 6):
        drafts = oracle.sample_drafts(draft, 0.6, 0.95, seed, 1 << 32)
        x = torch.from_numpy(drafts).cuda()
        tok, ln = vw4.accept_rejection_blockmax(tl.view(B, Kd + 1, N), tbm, dl.view(B, Kd, N), dbm,
                                                x, 0.6, 0.95, seed, 0)
        torch.cuda.synchronize()
        rt, rl, _ = oracle.accept_rejection(target, draft, drafts, 0.6, 0.95, seed, 0)
        assert np.array_equal(ln.cpu().numpy(), rl) and np.array_equal(tok.cpu().numpy(), rt)
    assert vw4.vw4_get_device_status() == 0


def test_fused_block_max_sixteen_rows_and_split_tiles():
    """16 verify rows (two mma n-tiles) and a stream-K shape whose tiles are
    split across CTAs: the block maxima are finished by the last contributor
    of each 16-row slice."""
    for N, K, M in ((40000, 512, 16), (50000, 1024, 3), (1000, 4096, 12)):
        q, s, ts = synth.linear(N, N, K, "nvfp4")
        out, bm = head_logits(q, (torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()), ts,
                              synth.activations(synth.rng(M), M, K))
        assert np.array_equal(bm.cpu().numpy(), block_max_ref(out.cpu().numpy()))
    assert vw4.vw4_get_device_status() == 0


def test_blockmax_argument_errors():
    q, s, ts = synth.linear(1, 128, 256, "nvfp4")
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    W = vw4.make_weight(vw4.FMT_NVFP4, qd, sd, ts, 128, 256)
    lib = vw4.load_library()
    A = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((2, 128), device="cuda")
    assert lib.verify_gemm_w4_blockmax(__import__("ctypes").byref(W), A.data_ptr(), 2, 256,
                                       out.data_ptr(), 128, None, None, 0, None) == 1
