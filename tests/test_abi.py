"""The C-ABI library loads and exports every symbol include/vw4.h declares, and
rejects bad arguments on the host before touching the GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

import speculative_decode_verification_w4_gb300 as vw4
from speculative_decode_verification_w4_gb300 import build as vbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    vbuild.build()
    return vw4.load_library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "vw4.h")).read()
    return sorted(set(re.findall(r"VW4_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    names = declared_symbols()
    assert set(names) == set(vw4.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(vw4.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(raw, name), name


def test_checks_build_exports_every_declared_symbol_and_says_so(lib):
    """The checks build (-DVW4_CHECKS: in-kernel bounds checks) compiles for
    sm_103a, exports every declared symbol, and reports its flag; the plain
    build reports none."""
    path = vbuild.build(checks=True)
    raw = ctypes.CDLL(path)
    for name in declared_symbols():
        assert hasattr(raw, name), name
    raw.vw4_build_flags.restype = ctypes.c_int
    assert raw.vw4_build_flags() == vw4.BUILD_CHECKS
    plain = ctypes.CDLL(vbuild.LIB)
    plain.vw4_build_flags.restype = ctypes.c_int
    assert plain.vw4_build_flags() == 0


def test_vw4_lib_selects_the_library_the_binding_opens(lib):
    """VW4_LIB names the library load_library() opens by default: the checks
    build when it points there, the plain build otherwise (host calls only)."""
    import subprocess
    import sys
    checks = vbuild.build(checks=True)
    code = ("import speculative_decode_verification_w4_gb300 as v; "
            "print(v.LIB_PATH, v.vw4_build_flags())")
    env = {k: val for k, val in os.environ.items() if k != "VW4_LIB"}
    plain = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env,
                           capture_output=True, text=True, timeout=300)
    assert plain.returncode == 0, plain.stderr[-2000:]
    assert plain.stdout.split() == [vbuild.LIB, "0"], plain.stdout
    chk = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=dict(env, VW4_LIB=checks),
                         capture_output=True, text=True, timeout=300)
    assert chk.returncode == 0, chk.stderr[-2000:]
    assert chk.stdout.split() == [checks, str(vw4.BUILD_CHECKS)], chk.stdout


def test_status_strings(lib):
    assert lib.vw4_status_str(0) == b"ok"
    assert lib.vw4_status_str(6) == b"workspace too small"
    assert lib.vw4_version() >= 100


def test_workspace_sizes(lib):
    assert vw4.vw4_workspace_bytes(vw4.OP_GEMM, 8, 262144, 5376) > 0
    # 9..16 rows take 16-row activation blocks and partial tiles: more bytes
    w8 = vw4.vw4_workspace_bytes(vw4.OP_GEMM, 8, 262144, 5376)
    assert vw4.vw4_workspace_bytes(vw4.OP_GEMM, 9, 262144, 5376) > w8
    # the rest grows only by the room to repack unaligned activation rows
    w9 = vw4.vw4_workspace_bytes(vw4.OP_GEMM, 9, 262144, 5376)
    w16 = vw4.vw4_workspace_bytes(vw4.OP_GEMM, 16, 262144, 5376)
    assert w9 <= w16 <= w9 + 7 * 5376 * 2 + 256
    assert vw4.vw4_workspace_bytes(vw4.OP_GEMM, 17, 1024, 1024) == 0
    assert vw4.vw4_workspace_bytes(vw4.OP_GEMM, 4, 1024, 1000) == 0
    assert vw4.vw4_workspace_bytes(vw4.OP_MOE, 64, 1536, 2048) > 0
    assert vw4.vw4_workspace_bytes(99, 1, 1, 1) == 0


def _weight(fmt=1, N=128, K=256, ts=1.0, q=0x1000, s=0x2000):
    return vw4.Weight(fmt, N, K, 0, q, s, ts, 0.0)


@pytest.mark.parametrize("kw,code", [
    (dict(M=0), 1), (dict(M=17), 1), (dict(lda=100), 1), (dict(ldo=10), 1),
    (dict(A=0), 1), (dict(out=0), 1), (dict(A=0x3001), 3), (dict(out=0x4002), 3),
    (dict(ws=0), 6), (dict(ws_bytes=16), 6),
])
def test_gemm_argument_checks_on_host(lib, kw, code):
    W = _weight()
    args = dict(A=0x3000, M=2, lda=256, out=0x4000, ldo=128, am=0, ws=0x10000,
                ws_bytes=1 << 30)
    args.update(kw)
    r = lib.verify_gemm_w4(ctypes.byref(W), args["A"], args["M"], args["lda"], args["out"],
                           args["ldo"], args["am"], args["ws"], args["ws_bytes"], None)
    assert r == code


@pytest.mark.parametrize("W,code", [
    (_weight(fmt=3), 1), (_weight(K=24), 1), (_weight(fmt=2, ts=2.0), 1),
    (_weight(q=0x1001), 3), (_weight(N=0), 1),
])
def test_weight_checks_on_host(lib, W, code):
    r = lib.verify_gemm_w4(ctypes.byref(W), 0x3000, 2, 512, 0x4000, 128, None, 0x10000,
                           1 << 30, None)
    assert r == code


def test_accept_argument_checks_on_host(lib):
    assert lib.accept_greedy(None, None, None, 1, 2, 10, 0x100, 0x200, None) == 1
    assert lib.accept_greedy(0x100, 0x100, None, 0, 2, 10, 0x100, 0x200, None) == 1
    assert lib.accept_greedy(0x100, 0x100, None, 1, 9, 10, 0x100, 0x200, None) == 1
    for bad in (vw4.Sampling(0.6, 0.95, -1, 0.0), vw4.Sampling(0.6, 0.95, 5, 1.5),
                vw4.Sampling(0.6, 0.95, 5, float("nan"))):
        assert lib.accept_rejection(0x100, 0x100, 0x100, 1, 2, 10, ctypes.byref(bad), 0, 0,
                                    0x100, 0x200, 0x1000, 1 << 20, None) == 1
    prm = vw4.Sampling(-1.0, 0.95, 0, 0.0)
    assert lib.accept_rejection(0x100, 0x100, 0x100, 1, 2, 10, ctypes.byref(prm), 0, 0, 0x100,
                                0x200, 0x1000, 1 << 20, None) == 1
    prm = vw4.Sampling(0.6, 0.0, 0, 0.0)
    assert lib.accept_rejection(0x100, 0x100, 0x100, 1, 2, 10, ctypes.byref(prm), 0, 0, 0x100,
                                0x200, 0x1000, 1 << 20, None) == 1


def test_accept_rejection_topk_argument_checks_on_host(lib):
    assert vw4.vw4_workspace_bytes(vw4.OP_REJECTION_TOPK, 256, 8, 64) > 0
    assert vw4.vw4_workspace_bytes(vw4.OP_REJECTION_TOPK, 256, 8, 1025) == 0
    prm = vw4.Sampling(0.6, 0.95, 0, 0.0)

    def call(Kt=16, B=2, Kd=2, V=100, p=prm, ws=0x1000, ws_bytes=1 << 24, t_ids=0x100):
        return lib.accept_rejection_topk(t_ids, 0x200, 0x300, 0x400, 0x500, B, Kd, Kt, V,
                                         ctypes.byref(p), 0, 0, 0x600, 0x700, ws, ws_bytes, None)
    assert call(Kt=0) == 1
    assert call(B=0) == 1
    assert call(Kd=9) == 1
    assert call(V=0) == 1
    assert call(t_ids=None) == 1
    assert call(Kt=1025) == 2                                 # longer lists: unsupported
    assert call(p=vw4.Sampling(0.0, 0.95, 0, 0.0)) == 2       # greedy: accept_greedy instead
    assert call(p=vw4.Sampling(0.6, 0.95, -1, 0.0)) == 1
    assert call(p=vw4.Sampling(0.6, 0.95, 0, 2.0)) == 1
    assert call(ws=None) == 6
    assert call(ws_bytes=64) == 6
    assert call(ws=0x1001) == 3


def test_verify_greedy_argument_checks_on_host(lib):
    W = _weight()
    # B * (Kd + 1) above 16, B < 1, Kd < 0, null tokens / lengths, null drafts with Kd > 0
    assert lib.verify_greedy_w4(ctypes.byref(W), 0x3000, 512, 0x100, 3, 5, 0x200, 0x300, None, 0,
                                0x10000, 1 << 30, None) == 1
    assert lib.verify_greedy_w4(ctypes.byref(W), 0x3000, 512, 0x100, 0, 3, 0x200, 0x300, None, 0,
                                0x10000, 1 << 30, None) == 1
    assert lib.verify_greedy_w4(ctypes.byref(W), 0x3000, 512, 0x100, 1, -1, 0x200, 0x300, None,
                                0, 0x10000, 1 << 30, None) == 1
    assert lib.verify_greedy_w4(ctypes.byref(W), 0x3000, 512, 0x100, 1, 3, None, 0x300, None, 0,
                                0x10000, 1 << 30, None) == 1
    assert lib.verify_greedy_w4(ctypes.byref(W), 0x3000, 512, None, 1, 3, 0x200, 0x300, None, 0,
                                0x10000, 1 << 30, None) == 1


def test_ragged_k_sizes_and_moe_rule(lib):
    """K a multiple of the block but not of 256: the dense GEMM sizes room for
    the weights padded to whole stages; the MoE call (its experts streamed in
    place) returns VW4_ERR_UNSUPPORTED on the host."""
    w256 = vw4.vw4_workspace_bytes(vw4.OP_GEMM, 8, 1000, 256)
    w272 = vw4.vw4_workspace_bytes(vw4.OP_GEMM, 8, 1000, 272)
    assert w272 >= w256 + 1000 * (512 // 2) + 1000 * (512 // 16)
    assert vw4.vw4_workspace_bytes(vw4.OP_GEMM, 8, 1000, 24) == 0
    assert vw4.vw4_workspace_bytes(vw4.OP_MOE, 8, 1000, 272) == 0
    W = _weight(K=272, N=64)
    r = lib.verify_moe_w4(ctypes.byref(W), 4, 0x3000, 512, 0, 0x5000, 0x6000, 2, 2, 1, 0x4000,
                          64, 0x10000, 1 << 30, None)
    assert r == 2
