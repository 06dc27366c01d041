"""Guard canaries around every output of every entry point.

Each call writes into views carved out of larger buffers filled with a
sentinel bit pattern: guard regions before and after every output, the
padding columns of strided outputs, and a guard after the workspace, whose
own bytes are filled with the same garbage (a workspace needs no
initialization).  The call must leave every sentinel as it was, leave its
inputs unchanged, and give results bit-identical to the same call on plain
buffers and a fresh zeroed workspace: a device-side write out of bounds or a
half-written output shows up here as a changed sentinel or a mismatch, not
as a silent corruption of a neighbour.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import speculative_decode_verification_w4_gb300 as vw4
from gpu_util import FMT, bf16_dev, upload_weight

pytestmark = pytest.mark.gpu

SENT32 = -0x5A5A5A5B   # 0xA5A5A5A5 as int32 (a NaN pattern as fp32)
SENT8 = 0xA5
G = 1024               # guard elements on each side (4 KB: keeps 256-byte alignment)


class Guarded:
    """A [rows, cols] view (row stride ld) of 4-byte elements inside a flat
    buffer of sentinels, with G sentinel elements before and after."""

    def __init__(self, rows, cols, ld, dtype):
        self.rows, self.cols, self.ld = rows, cols, ld
        self.flat = torch.full((G + rows * ld + G,), SENT32, dtype=torch.int32, device="cuda")
        body = self.flat[G:G + rows * ld].view(dtype)
        self.view = body.view(rows, ld)[:, :cols]

    def check(self, what):
        f = self.flat.cpu().numpy()
        body = f[G:G + self.rows * self.ld].reshape(self.rows, self.ld)
        assert (f[:G] == SENT32).all(), f"{what}: guard before the output written"
        assert (f[G + self.rows * self.ld:] == SENT32).all(), f"{what}: guard after the output written"
        assert (body[:, self.cols:] == SENT32).all(), f"{what}: padding between rows written"


class GuardedWorkspace:
    """need bytes of garbage followed by a guard of sentinel bytes."""

    def __init__(self, need):
        self.need = need
        self.buf = torch.full((need + 4 * G,), SENT8, dtype=torch.uint8, device="cuda")
        self.ws = self.buf[:need]

    def check(self, what):
        tail = self.buf[self.need:].cpu().numpy()
        assert (tail == SENT8).all(), f"{what}: written past the workspace"


def same_bits(a, b, what):
    a = a.contiguous().view(torch.int32) if a.element_size() == 4 else a.contiguous()
    b = b.contiguous().view(torch.int32) if b.element_size() == 4 else b.contiguous()
    assert torch.equal(a, b), f"{what}: result differs from the call on plain buffers"


def status_ok(what):
    torch.cuda.synchronize()
    st = vw4.vw4_get_device_status()
    assert st == 0, f"{what}: device status {st:#x}"


def weight(fmt, N, K, seed):
    q, s, ts = synth.linear(seed, N, K, fmt)
    qd, sd = upload_weight(q, s, fmt)
    return qd, sd, ts


@pytest.mark.parametrize("fmt,N,K,M,argmax", [
    ("nvfp4", 1000, 768, 3, True),      # ragged last tile, few rows
    ("q4_0", 1000, 768, 3, True),
    ("nvfp4", 300, 8192, 8, False),     # few tiles, long K: split-K parts
    ("nvfp4", 40000, 512, 8, True),     # many tiles: stream-K finish
    ("nvfp4", 5000, 2304, 16, True),    # two n-tiles
    ("q4_0", 700, 1056, 12, False),     # ragged K: the padded-weights path
    ("nvfp4", 900, 1040, 8, True),
])
def test_verify_gemm_canaries(fmt, N, K, M, argmax):
    qd, sd, ts = weight(fmt, N, K, 700 + N + K)
    A = bf16_dev(synth.activations(synth.rng(M + K), M, K))
    A0 = A.clone()
    ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ref_am = torch.empty((M,), dtype=torch.int32, device="cuda") if argmax else None
    vw4.verify_gemm_w4(FMT[fmt], qd, sd, ts, A, out=ref, row_argmax=ref_am,
                       workspace=vw4.Workspace())
    status_ok("reference call")
    out = Guarded(M, N, N + 37, torch.float32)
    am = Guarded(1, M, M, torch.int32) if argmax else None
    ws = GuardedWorkspace(vw4.vw4_workspace_bytes(vw4.OP_GEMM, M, N, K))
    for rep in range(2):  # the second call starts from the first call's workspace
        vw4.verify_gemm_w4(FMT[fmt], qd, sd, ts, A, out=out.view,
                           row_argmax=am.view[0] if argmax else None, workspace=ws.ws)
        status_ok("guarded call")
        out.check("out")
        same_bits(out.view, ref, "out")
        if argmax:
            am.check("row_argmax")
            same_bits(am.view[0], ref_am, "row_argmax")
        ws.check("workspace")
    assert torch.equal(A.view(torch.int16), A0.view(torch.int16)), "activations changed"


def test_verify_gemm_noalloc_canaries():
    N, K, M = 3000, 1024, 8
    qd, sd, ts = weight("nvfp4", N, K, 77)
    A = bf16_dev(synth.activations(synth.rng(78), M, K))
    ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ref_am = torch.empty((M,), dtype=torch.int32, device="cuda")
    vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, A, out=ref, row_argmax=ref_am,
                       workspace=vw4.Workspace())
    status_ok("reference call")
    out = Guarded(M, N, N + 5, torch.float32)
    am = Guarded(1, M, M, torch.int32)
    W = vw4.make_weight(vw4.FMT_NVFP4, qd, sd, ts, N, K)
    lib = vw4.load_library()
    code = lib.verify_gemm_w4_noalloc(ctypes.byref(W), ctypes.c_void_p(A.data_ptr()), M,
                                      A.stride(0), ctypes.c_void_p(out.view.data_ptr()), N + 5,
                                      ctypes.c_void_p(am.view.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    status_ok("noalloc call")
    out.check("out")
    am.check("row_argmax")
    # the fused argmax is bit-exact; the outputs are the same GEMM
    same_bits(am.view[0], ref_am, "row_argmax")
    same_bits(out.view, ref, "out")


def test_verify_gemm_blockmax_canaries():
    N, K, M = 2000, 768, 5
    qd, sd, ts = weight("nvfp4", N, K, 91)
    A = bf16_dev(synth.activations(synth.rng(92), M, K))
    nb = (N + 15) // 16
    ref, ref_bm = vw4.verify_gemm_w4_blockmax(vw4.FMT_NVFP4, qd, sd, ts, A,
                                              workspace=vw4.Workspace())
    status_ok("reference call")
    out = Guarded(M, N, N + 11, torch.float32)
    bm = Guarded(M, nb, nb, torch.float32)
    ws = GuardedWorkspace(vw4.vw4_workspace_bytes(vw4.OP_GEMM, M, N, K))
    vw4.verify_gemm_w4_blockmax(vw4.FMT_NVFP4, qd, sd, ts, A, out=out.view, block_max=bm.view,
                                workspace=ws.ws)
    status_ok("guarded call")
    out.check("out")
    bm.check("block_max")
    ws.check("workspace")
    same_bits(out.view, ref, "out")
    same_bits(bm.view, ref_bm, "block_max")


@pytest.mark.parametrize("with_logits", [False, True])
def test_verify_greedy_canaries(with_logits):
    N, K, B, Kd = 6000, 1024, 2, 5
    M = B * (Kd + 1)
    qd, sd, ts = weight("nvfp4", N, K, 93)
    A = bf16_dev(synth.activations(synth.rng(94), M, K))
    drafts = torch.from_numpy(synth.rng(95).integers(0, N, (B, Kd), dtype=np.int32)).cuda()
    d0 = drafts.clone()
    ref_out = torch.empty((M, N), dtype=torch.float32, device="cuda") if with_logits else None
    ref_t, ref_l = vw4.verify_greedy_w4(vw4.FMT_NVFP4, qd, sd, ts, A, drafts, out=ref_out,
                                        workspace=vw4.Workspace())
    status_ok("reference call")
    tok = Guarded(B, Kd + 1, Kd + 1, torch.int32)
    ln = Guarded(1, B, B, torch.int32)
    out = Guarded(M, N, N + 3, torch.float32) if with_logits else None
    ws = GuardedWorkspace(vw4.vw4_workspace_bytes(vw4.OP_GEMM, M, N, K))
    vw4.verify_greedy_w4(vw4.FMT_NVFP4, qd, sd, ts, A, drafts,
                         out=out.view if with_logits else None, tokens=tok.view,
                         length=ln.view[0], workspace=ws.ws)
    status_ok("guarded call")
    tok.check("tokens")
    ln.check("len")
    ws.check("workspace")
    same_bits(tok.view, ref_t, "tokens")
    same_bits(ln.view[0], ref_l, "len")
    if with_logits:
        out.check("logits")
        same_bits(out.view, ref_out, "logits")
    assert torch.equal(drafts, d0), "drafts changed"


@pytest.mark.parametrize("M,rows_are_pairs,combine", [(8, 0, 0), (8, 1, 1), (16, 0, 1)])
def test_verify_moe_canaries(M, rows_are_pairs, combine):
    E, N, K, topk = 16, 512, 512, 4
    q, s, ts = synth.linear(96, E * N, K, "nvfp4")
    qd, sd = upload_weight(q, s, "nvfp4")
    ids, gates = synth.routing(97 + M, M, E, topk)
    ids_d = torch.from_numpy(ids).cuda()
    gates_d = torch.from_numpy(gates).cuda()
    rows_in = M * topk if rows_are_pairs else M
    A = bf16_dev(synth.activations(synth.rng(98), rows_in, K))
    rows_out = M if combine else M * topk
    ref = vw4.verify_moe_w4(vw4.FMT_NVFP4, qd, sd, ts, E, A, rows_are_pairs, ids_d, gates_d,
                            combine, workspace=vw4.Workspace())
    status_ok("reference call")
    out = Guarded(rows_out, N, N + 9, torch.float32)
    ws = GuardedWorkspace(vw4.vw4_workspace_bytes(vw4.OP_MOE, M * topk, N, K))
    vw4.verify_moe_w4(vw4.FMT_NVFP4, qd, sd, ts, E, A, rows_are_pairs, ids_d, gates_d, combine,
                      out=out.view, workspace=ws.ws)
    status_ok("guarded call")
    out.check("out")
    ws.check("workspace")
    same_bits(out.view, ref, "out")


def test_accept_greedy_canaries():
    B, Kd, V = 5, 6, 30000
    g = synth.rng(99)
    logits = torch.from_numpy(synth.logits(g, (B, Kd + 1, V), 2.0)).cuda()
    l0 = logits.clone()
    am = logits.argmax(-1).cpu().numpy()
    drafts = torch.from_numpy(synth.greedy_drafts(g, am[:, :Kd], V)).cuda()
    ref_t, ref_l = vw4.accept_greedy(logits, drafts)
    status_ok("reference call")
    tok = Guarded(B, Kd + 1, Kd + 1, torch.int32)
    ln = Guarded(1, B, B, torch.int32)
    vw4.accept_greedy(logits, drafts, tokens=tok.view, length=ln.view[0])
    status_ok("guarded call")
    tok.check("tokens")
    ln.check("len")
    same_bits(tok.view, ref_t, "tokens")
    same_bits(ln.view[0], ref_l, "len")
    assert torch.equal(logits, l0), "logits changed"


@pytest.mark.parametrize("B,Kd,V,top_k,min_p", [
    (40, 4, 5000, 0, 0.0),      # one CTA per row
    (1, 3, 40000, 0, 0.0),      # few rows of a wide vocabulary: rows split over CTAs
    (6, 2, 20000, 50, 0.05),    # top-k and min-p stages
])
def test_accept_rejection_canaries(B, Kd, V, top_k, min_p):
    tgt, drf, drafts = synth.stochastic_case(101 + B, B, Kd, V)
    tgt_d, drf_d, dr_d = (torch.from_numpy(x).cuda() for x in (tgt, drf, drafts))
    t0, f0 = tgt_d.clone(), drf_d.clone()
    ref_t, ref_l = vw4.accept_rejection(tgt_d, drf_d, dr_d, 0.6, 0.95, 4, 7, top_k=top_k,
                                        min_p=min_p, workspace=vw4.Workspace())
    status_ok("reference call")
    tok = Guarded(B, Kd + 1, Kd + 1, torch.int32)
    ln = Guarded(1, B, B, torch.int32)
    ws = GuardedWorkspace(vw4.vw4_workspace_bytes(vw4.OP_REJECTION, B, Kd, V))
    vw4.accept_rejection(tgt_d, drf_d, dr_d, 0.6, 0.95, 4, 7, top_k=top_k, min_p=min_p,
                         tokens=tok.view, length=ln.view[0], workspace=ws.ws)
    status_ok("guarded call")
    tok.check("tokens")
    ln.check("len")
    ws.check("workspace")
    same_bits(tok.view, ref_t, "tokens")
    same_bits(ln.view[0], ref_l, "len")
    assert torch.equal(tgt_d, t0) and torch.equal(drf_d, f0), "logits changed"


def test_accept_rejection_blockmax_canaries():
    B, Kd, V = 3, 3, 20000
    tgt, drf, drafts = synth.stochastic_case(111, B, Kd, V)
    tgt_d, drf_d, dr_d = (torch.from_numpy(x).cuda() for x in (tgt, drf, drafts))
    nb = (V + 15) // 16

    def bmax(x):
        pad = torch.full((*x.shape[:-1], nb * 16), float("-inf"), device="cuda")
        pad[..., :V] = x
        return pad.view(*x.shape[:-1], nb, 16).amax(-1).contiguous()
    tb, db = bmax(tgt_d), bmax(drf_d)
    ref_t, ref_l = vw4.accept_rejection_blockmax(tgt_d, tb, drf_d, db, dr_d, 0.6, 0.95, 4, 3,
                                                 workspace=vw4.Workspace())
    status_ok("reference call")
    tok = Guarded(B, Kd + 1, Kd + 1, torch.int32)
    ln = Guarded(1, B, B, torch.int32)
    ws = GuardedWorkspace(vw4.vw4_workspace_bytes(vw4.OP_REJECTION, B, Kd, V))
    vw4.accept_rejection_blockmax(tgt_d, tb, drf_d, db, dr_d, 0.6, 0.95, 4, 3, tokens=tok.view,
                                  length=ln.view[0], workspace=ws.ws)
    status_ok("guarded call")
    tok.check("tokens")
    ln.check("len")
    ws.check("workspace")
    same_bits(tok.view, ref_t, "tokens")
    same_bits(ln.view[0], ref_l, "len")


@pytest.mark.parametrize("Kt", [64, 300])
def test_accept_rejection_topk_canaries(Kt):
    B, Kd, V = 8, 4, 151936
    ti, tv, di, dv, drafts = synth.topk_lists_case(121 + Kt, B, Kd, Kt, V)
    ti_d, tv_d, di_d, dv_d, dr_d = (torch.from_numpy(x).cuda() for x in (ti, tv, di, dv, drafts))
    ref_t, ref_l = vw4.accept_rejection_topk(ti_d, tv_d, di_d, dv_d, dr_d, V, 0.6, 0.95, 4, 1,
                                             workspace=vw4.Workspace())
    status_ok("reference call")
    tok = Guarded(B, Kd + 1, Kd + 1, torch.int32)
    ln = Guarded(1, B, B, torch.int32)
    ws = GuardedWorkspace(vw4.vw4_workspace_bytes(vw4.OP_REJECTION_TOPK, B, Kd, Kt))
    vw4.accept_rejection_topk(ti_d, tv_d, di_d, dv_d, dr_d, V, 0.6, 0.95, 4, 1, tokens=tok.view,
                              length=ln.view[0], workspace=ws.ws)
    status_ok("guarded call")
    tok.check("tokens")
    ln.check("len")
    ws.check("workspace")
    same_bits(tok.view, ref_t, "tokens")
    same_bits(ln.view[0], ref_l, "len")
