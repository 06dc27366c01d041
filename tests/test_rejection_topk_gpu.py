"""GPU parity of accept_rejection_topk (rows given as top-k lists) against
the oracle: committed ids and lengths bit-exact.  The oracle's reading of a
list is the dense row holding the listed logits and -inf elsewhere; the
lists come from dense synthetic rows (their top Kt, shuffled) or are drawn
directly (synth.topk_lists_case), at small sizes and at the full sweep size
(vocabulary 151936, 256 sequences, sampled sequences checked)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decode_verification_w4_gb300 as vw4

pytestmark = pytest.mark.gpu


def _dev(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x, dtype)).cuda()


def gpu_accept(t_ids, t_vals, d_ids, d_vals, drafts, V, T, top_p, seed, offset, **kw):
    Kd = t_ids.shape[1] - 1
    tok, ln = vw4.accept_rejection_topk(
        _dev(t_ids, np.int32), _dev(t_vals, np.float32),
        _dev(d_ids, np.int32) if Kd else None, _dev(d_vals, np.float32) if Kd else None,
        _dev(drafts, np.int32), V, T, top_p, seed, offset, **kw)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ln.cpu().numpy()


def _top_lists(rows, Kt, g):
    B, R, V = rows.shape
    ids = np.empty((B, R, Kt), np.int32)
    vals = np.empty((B, R, Kt), np.float32)
    for b in range(B):
        for r in range(R):
            o = np.lexsort((np.arange(V), -rows[b, r].astype(np.float64)))[:Kt]
            o = o[g.permutation(Kt)]
            ids[b, r], vals[b, r] = o, rows[b, r, o]
    return ids, vals


@pytest.mark.parametrize("B,Kd,V,Kt,top_p,top_k,min_p", [
    (16, 3, 300, 16, 0.95, 0, 0.0), (32, 2, 5000, 50, 0.95, 0, 0.0),
    (12, 4, 2000, 64, 0.9, 20, 0.05), (8, 8, 20000, 256, 0.95, 0, 0.0),
    (9, 1, 1000, 1, 0.95, 0, 0.0), (5, 0, 700, 40, 0.8, 0, 0.0),
    (10, 5, 40000, 1024, 0.95, 100, 0.1), (6, 2, 3000, 100, 1.0, 0, 1.0),
    (7, 3, 500, 33, 0.5, 0, 0.0)])
def test_lists_from_dense_rows_match_oracle(B, Kd, V, Kt, top_p, top_k, min_p):
    g = synth.rng(B * 13 + Kt)
    target, draft, _ = synth.stochastic_case(B + V + Kt, B, Kd, V)
    kk = min(top_k, Kt) if top_k else Kt
    drafts = oracle.sample_drafts(draft, 0.6, top_p, 3, 1 << 32, top_k=kk, min_p=min_p) if Kd \
        else np.zeros((B, 0), np.int32)
    t_ids, t_vals = _top_lists(target, Kt, g)
    d_ids, d_vals = _top_lists(draft, Kt, g) if Kd else (None, None)
    kw = dict(top_k=top_k, min_p=min_p)
    tok, ln = gpu_accept(t_ids, t_vals, d_ids, d_vals, drafts, V, 0.6, top_p, 3, 7, **kw)
    rt, rl, _ = oracle.accept_rejection_topk(t_ids, t_vals, d_ids, d_vals, drafts, V, 0.6, top_p,
                                             3, 7, **kw)
    assert np.array_equal(ln, rl), (ln, rl)
    assert np.array_equal(tok, rt)
    # and the dense accept with the top-k stage at Kt gives the same run
    dt, dl, _ = oracle.accept_rejection(target, draft, drafts, 0.6, top_p, 3, 7, top_k=kk,
                                        min_p=min_p)
    assert np.array_equal(ln, dl) and np.array_equal(tok, dt)


@pytest.mark.parametrize("B,Kd,Kt,V", [(24, 4, 64, 151936), (16, 8, 200, 50000),
                                       (40, 1, 8, 1000)])
def test_drawn_lists_match_oracle(B, Kd, Kt, V):
    """Lists that overlap only in part (draft ids swapped out), in any order."""
    t_ids, t_vals, d_ids, d_vals, drafts = synth.topk_lists_case(B + Kt, B, Kd, Kt, V)
    g = synth.rng(Kt)  # shuffle every list together with its logits
    perm_t = np.argsort(g.random(t_ids.shape), axis=-1)
    t_ids, t_vals = np.take_along_axis(t_ids, perm_t, -1), np.take_along_axis(t_vals, perm_t, -1)
    perm_d = np.argsort(g.random(d_ids.shape), axis=-1)
    d_ids, d_vals = np.take_along_axis(d_ids, perm_d, -1), np.take_along_axis(d_vals, perm_d, -1)
    tok, ln = gpu_accept(t_ids, t_vals, d_ids, d_vals, drafts, V, 0.6, 0.95, 11, 0)
    for b in range(B):
        rt, rl, _ = oracle.accept_rejection_topk(t_ids[b:b + 1], t_vals[b:b + 1], d_ids[b:b + 1],
                                                 d_vals[b:b + 1], drafts[b:b + 1], V, 0.6, 0.95,
                                                 11, 0, b_base=b)
        assert rl[0] == ln[b] and np.array_equal(rt[0], tok[b]), b


def test_degenerate_entries_and_bad_ids():
    """-inf and NaN logits in the lists, a NaN at id 0 (the dense row's max is
    then NaN and every mass 0: the draw returns V - 1), a target row with
    every logit -inf, an out-of-range list id (dropped, flagged) and
    out-of-range draft ids (rejections, flagged)."""
    B, Kd, Kt, V = 8, 3, 32, 4000
    t_ids, t_vals, d_ids, d_vals, drafts = synth.topk_lists_case(5, B, Kd, Kt, V)
    t_vals[0, 0, 3] = -np.inf
    t_vals[0, 1, 5] = np.nan
    d_vals[1, 0, 2] = np.nan
    z = np.flatnonzero(t_ids[2, 0] == 0)    # id 0 listed with NaN: all masses 0
    k0 = int(z[0]) if z.size else 0
    t_ids[2, 0, k0] = 0
    t_vals[2, 0, k0] = np.nan
    t_vals[3, 1, :] = -np.inf               # an empty row
    t_ids[4, 2, 7] = V + 5                  # out of range: dropped
    drafts[5, 0] = -1
    drafts[6, 0] = V                        # position 0: always tested
    vw4.vw4_get_device_status()
    tok, ln = gpu_accept(t_ids, t_vals, d_ids, d_vals, drafts, V, 0.6, 0.95, 2, 9)
    st = vw4.vw4_get_device_status()
    rt, rl, bad = oracle.accept_rejection_topk(t_ids, t_vals, d_ids, d_vals, drafts, V, 0.6, 0.95,
                                               2, 9)
    assert np.array_equal(ln, rl), (ln, rl)
    assert np.array_equal(tok, rt)
    assert bad == 2 and st & vw4.DEV_BAD_DRAFT_ID and st & vw4.DEV_BAD_LIST_ID


def test_p_equals_q_lists_accept_everything():
    B, Kd, Kt, V = 16, 6, 128, 30000
    t_ids, t_vals, _, _, _ = synth.topk_lists_case(8, B, Kd, Kt, V)
    d_ids, d_vals = t_ids[:, :Kd].copy(), t_vals[:, :Kd].copy()
    rows = oracle.lists_to_rows(d_ids, d_vals, V)
    drafts = oracle.sample_drafts(rows, 0.6, 0.95, 4, 1 << 32)
    tok, ln = gpu_accept(t_ids, t_vals, d_ids, d_vals, drafts, V, 0.6, 0.95, 4, 0)
    assert np.all(ln == Kd + 1)
    rt, rl, _ = oracle.accept_rejection_topk(t_ids, t_vals, d_ids, d_vals, drafts, V, 0.6, 0.95,
                                             4, 0)
    assert np.array_equal(tok, rt)


@pytest.mark.parametrize("Kd", [1, 8])
def test_full_size_sampled(Kd):
    """256 sequences, vocabulary 151936, 64-entry lists: every sequence on the
    GPU, a sample through the oracle (same counter indices)."""
    B, Kt, V = 256, 64, 151936
    t_ids, t_vals, d_ids, d_vals, drafts = synth.topk_lists_case(60 + Kd, B, Kd, Kt, V)
    tok, ln = gpu_accept(t_ids, t_vals, d_ids, d_vals, drafts, V, 0.6, 0.95, 4, 0, top_k=50,
                         min_p=0.05)
    for b in (0, 1, 100, 255):
        rt, rl, _ = oracle.accept_rejection_topk(t_ids[b:b + 1], t_vals[b:b + 1], d_ids[b:b + 1],
                                                 d_vals[b:b + 1], drafts[b:b + 1], V, 0.6, 0.95,
                                                 4, 0, b_base=b, top_k=50, min_p=0.05)
        assert rl[0] == ln[b] and np.array_equal(rt[0], tok[b]), b
    assert vw4.vw4_get_device_status() == 0
