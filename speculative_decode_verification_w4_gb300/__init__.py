"""speculative_decode_verification_w4_gb300 -- Python binding of the vw4 C ABI.

A thin ctypes layer over ``libvw4.so`` (see ``include/vw4.h``): it marshals
torch tensors into device pointers and sizes, and turns status codes into
exceptions.  Every step of the computation runs in the library's CUDA kernels;
there is no fallback.  If the library is missing or cannot be loaded, every
call raises.

Entry points (same names as the C ABI):
  verify_gemm_w4, verify_moe_w4, accept_greedy, accept_rejection,
  accept_rejection_topk,
  vw4_workspace_bytes, vw4_get_device_status, vw4_q4_0_from_blocks,
  vw4_set_wait_limit_ns.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# the plain build; the checks build (in-kernel bounds checks, see vw4.h) sits
# beside it.  VW4_LIB, when set, names the library that load_library() opens
# by default (e.g. the checks build for a test run).
LIB_CHECKS_PATH = os.path.join(_HERE, "libvw4_checks.so")
LIB_PATH = os.environ.get("VW4_LIB") or os.path.join(_HERE, "libvw4.so")

FMT_NVFP4 = 1
FMT_Q4_0 = 2
OP_GEMM = 1
OP_MOE = 2
OP_REJECTION = 3
OP_REJECTION_TOPK = 4

DEV_BAD_DRAFT_ID = 0x1
DEV_BAD_EXPERT_ID = 0x2
DEV_WAIT_TIMEOUT = 0x4
DEV_ZERO_RESIDUAL = 0x8
DEV_BAD_LIST_ID = 0x10
DEV_BOUNDS = 0x20          # checks build only: an in-kernel bounds check failed
BUILD_CHECKS = 0x1         # vw4_build_flags(): the checks build

STATUS_NAMES = {0: "VW4_OK", 1: "VW4_ERR_INVALID_ARG", 2: "VW4_ERR_UNSUPPORTED",
                3: "VW4_ERR_ALIGN", 4: "VW4_ERR_CUDA", 5: "VW4_ERR_TIMEOUT",
                6: "VW4_ERR_WORKSPACE"}

# the exported C symbols (checked against include/vw4.h by the tests)
EXPORTS = ("verify_gemm_w4", "verify_moe_w4", "accept_greedy", "accept_rejection",
           "vw4_workspace_bytes", "vw4_get_device_status", "vw4_q4_0_from_blocks",
           "vw4_status_str", "vw4_last_error_string", "vw4_version", "vw4_set_wait_limit_ns",
           "vw4_own_exp", "vw4_own_mass_pairs", "verify_gemm_w4_noalloc", "verify_greedy_w4",
           "vw4_depth_ctl_init",
           "vw4_depth_ctl_observe", "vw4_depth_ctl_expected", "vw4_depth_ctl_choose",
           "accept_rejection_topk", "vw4_rejection_row_records",
           "vw4_test_inject_stall", "verify_gemm_w4_blockmax", "accept_rejection_blockmax",
           "vw4_build_flags")


class VW4Error(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        msg = f"{where}: {STATUS_NAMES.get(code, code)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class DepthCtl(ctypes.Structure):
    """vw4_depth_ctl (see vw4.h): the draft-depth controller's state."""
    _fields_ = [("att", ctypes.c_double * 16), ("acc", ctypes.c_double * 16),
                ("verify_us", ctypes.c_float * 17), ("draft_us_fixed", ctypes.c_float),
                ("draft_us_per_token", ctypes.c_float), ("k_max", ctypes.c_int32),
                ("decay", ctypes.c_float)]


class Weight(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("q_dev", ctypes.c_void_p),
                ("scales_dev", ctypes.c_void_p), ("tensor_scale", ctypes.c_float),
                ("reserved_f", ctypes.c_float)]


class Sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_p", ctypes.c_float),
                ("top_k", ctypes.c_int32), ("min_p", ctypes.c_float)]


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH):
    """Loads libvw4.so and declares the C signatures.  Raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"the vw4 library is not built at {path}: run "
                              "`python -m speculative_decode_verification_w4_gb300.build`")
        lib = ctypes.CDLL(path)
        P, I, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
        sigs = {
            "verify_gemm_w4": (I, [ctypes.POINTER(Weight), P, I, I, P, I, P, P, ctypes.c_size_t, P]),
            "verify_moe_w4": (I, [ctypes.POINTER(Weight), I, P, I, I, P, P, I, I, I, P, I, P,
                                  ctypes.c_size_t, P]),
            "accept_greedy": (I, [P, P, P, I, I, I, P, P, P]),
            "accept_rejection": (I, [P, P, P, I, I, I, ctypes.POINTER(Sampling), U64, U64, P, P,
                                     P, ctypes.c_size_t, P]),
            "accept_rejection_topk": (I, [P, P, P, P, P, I, I, I, I, ctypes.POINTER(Sampling),
                                          U64, U64, P, P, P, ctypes.c_size_t, P]),
            "vw4_workspace_bytes": (ctypes.c_size_t, [I, I, I, I]),
            "vw4_get_device_status": (I, [ctypes.POINTER(ctypes.c_uint32), P]),
            "vw4_q4_0_from_blocks": (I, [P, I, I, P, P, P]),
            "vw4_status_str": (ctypes.c_char_p, [I]),
            "vw4_last_error_string": (ctypes.c_char_p, []),
            "vw4_version": (I, []),
            "vw4_build_flags": (I, []),
            "vw4_set_wait_limit_ns": (None, [U64]),
            "vw4_own_exp": (I, [P, P, ctypes.c_int64, P]),
            "vw4_own_mass_pairs": (I, [P, P, ctypes.c_int64, P]),
            "verify_gemm_w4_noalloc": (I, [ctypes.POINTER(Weight), P, I, I, P, I, P, P]),
            "vw4_depth_ctl_init": (I, [ctypes.POINTER(DepthCtl), I, ctypes.c_float]),
            "vw4_depth_ctl_observe": (I, [ctypes.POINTER(DepthCtl), I, I]),
            "vw4_depth_ctl_expected": (I, [ctypes.POINTER(DepthCtl), I,
                                           ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_double)]),
            "vw4_depth_ctl_choose": (I, [ctypes.POINTER(DepthCtl)]),
            "verify_greedy_w4": (I, [ctypes.POINTER(Weight), P, I, P, I, I, P, P, P, I, P,
                                     ctypes.c_size_t, P]),
            "vw4_rejection_row_records": (I, [P, ctypes.c_size_t, I, I, I, P, P]),
            "vw4_test_inject_stall": (None, [I]),
            "verify_gemm_w4_blockmax": (I, [ctypes.POINTER(Weight), P, I, I, P, I, P, P,
                                            ctypes.c_size_t, P]),
            "accept_rejection_blockmax": (I, [P, P, P, P, P, I, I, I, ctypes.POINTER(Sampling),
                                              U64, U64, P, P, P, ctypes.c_size_t, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(code: int, where: str):
    if code != 0:
        detail = ""
        if code == 4:
            detail = load_library().vw4_last_error_string().decode(errors="replace")
        raise VW4Error(code, where, detail)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def vw4_workspace_bytes(op: int, a: int, b: int, c: int) -> int:
    return int(load_library().vw4_workspace_bytes(op, a, b, c))


class Workspace:
    """A growable device scratch buffer (256-byte aligned torch allocation),
    zero-filled when allocated as the library requires of a fresh workspace
    (every call leaves it that way)."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def _workspace(ws, nbytes, device):
    if ws is None:
        key = (device.index, threading.get_ident())
        ws = _default_ws.setdefault(key, Workspace(device))
    if isinstance(ws, Workspace):
        return ws.get(nbytes)
    if ws.numel() * ws.element_size() < nbytes:
        raise VW4Error(6, "workspace", f"need {nbytes} bytes")
    return ws


def make_weight(fmt: int, q: torch.Tensor, scales: torch.Tensor, tensor_scale: float = 1.0,
                N: int | None = None, K: int | None = None) -> Weight:
    if N is None:
        N = q.shape[-2] if q.dim() >= 2 else 1
    if K is None:
        K = q.shape[-1] * 2
    return Weight(fmt, int(N), int(K), 0, q.data_ptr(), scales.data_ptr(), float(tensor_scale), 0.0)


def verify_gemm_w4(fmt: int, q: torch.Tensor, scales: torch.Tensor, tensor_scale: float,
                   A: torch.Tensor, out: torch.Tensor | None = None,
                   row_argmax: torch.Tensor | None = None, workspace=None, stream=None):
    """out[M, N] (fp32) = A[M, K] (bf16) x w[N, K]^T; q u8 [N, K/2]; see vw4.h."""
    N, K = q.shape[0], q.shape[1] * 2
    M = A.shape[0]
    if A.dtype != torch.bfloat16:
        raise ValueError("A must be bfloat16")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    W = make_weight(fmt, q, scales, tensor_scale, N, K)
    need = vw4_workspace_bytes(OP_GEMM, M, N, K)
    ws = _workspace(workspace, need, A.device)
    code = load_library().verify_gemm_w4(ctypes.byref(W), _ptr(A), M, A.stride(0), _ptr(out),
                                         out.stride(0), _ptr(row_argmax), _ptr(ws),
                                         ws.numel(), _stream(stream))
    _check(code, "verify_gemm_w4")
    return out


def verify_gemm_w4_blockmax(fmt: int, q: torch.Tensor, scales: torch.Tensor,
                            tensor_scale: float, A: torch.Tensor, out: torch.Tensor | None = None,
                            block_max: torch.Tensor | None = None, workspace=None, stream=None):
    """verify_gemm_w4 that also writes block_max fp32 [M, ceil(N/16)], the
    largest of every 16 consecutive outputs of each row -> (out, block_max)."""
    N, K = q.shape[0], q.shape[1] * 2
    M = A.shape[0]
    if A.dtype != torch.bfloat16:
        raise ValueError("A must be bfloat16")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    nb = (N + 15) // 16
    if block_max is None:
        block_max = torch.empty((M, nb), dtype=torch.float32, device=A.device)
    if block_max.stride(0) != nb or block_max.stride(1) != 1:
        raise ValueError("block_max must be a contiguous [M, ceil(N/16)] tensor")
    W = make_weight(fmt, q, scales, tensor_scale, N, K)
    ws = _workspace(workspace, vw4_workspace_bytes(OP_GEMM, M, N, K), A.device)
    code = load_library().verify_gemm_w4_blockmax(ctypes.byref(W), _ptr(A), M, A.stride(0),
                                                  _ptr(out), out.stride(0), _ptr(block_max),
                                                  _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "verify_gemm_w4_blockmax")
    return out, block_max


def verify_greedy_w4(fmt: int, q: torch.Tensor, scales: torch.Tensor, tensor_scale: float,
                     A: torch.Tensor, drafts: torch.Tensor, out: torch.Tensor | None = None,
                     tokens=None, length=None, workspace=None, stream=None):
    """The verify GEMM over A [B*(Kd+1), K] (sequence b's rows together), its
    row argmax and the greedy accept of drafts int32 [B, Kd], in one launch ->
    (tokens [B, Kd+1], len [B]).  out: optional fp32 [B*(Kd+1), N] logits (not
    written when None); see vw4.h."""
    N, K = q.shape[0], q.shape[1] * 2
    B, Kd = drafts.shape
    M = B * (Kd + 1)
    if A.dtype != torch.bfloat16 or A.shape[0] != M:
        raise ValueError("A must be bfloat16 [B*(Kd+1), K]")
    if tokens is None:
        tokens = torch.empty((B, Kd + 1), dtype=torch.int32, device=A.device)
    if length is None:
        length = torch.empty((B,), dtype=torch.int32, device=A.device)
    W = make_weight(fmt, q, scales, tensor_scale, N, K)
    ws = _workspace(workspace, vw4_workspace_bytes(OP_GEMM, M, N, K), A.device)
    code = load_library().verify_greedy_w4(
        ctypes.byref(W), _ptr(A), A.stride(0), _ptr(drafts), B, Kd, _ptr(tokens), _ptr(length),
        _ptr(out), out.stride(0) if out is not None else 0, _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "verify_greedy_w4")
    return tokens, length


class DepthController:
    """The draft-depth controller of vw4.h on a caller-owned state: verify
    costs per width (us, for 1..k_max+1 rows), the drafting cost, live
    per-position acceptance from observed verify steps."""

    def __init__(self, k_max: int = 7, decay: float = 0.98, verify_us=None,
                 draft_us_fixed: float = 0.0, draft_us_per_token: float = 0.0):
        self.state = DepthCtl()
        _check(load_library().vw4_depth_ctl_init(ctypes.byref(self.state), k_max, decay),
               "vw4_depth_ctl_init")
        if verify_us is not None:
            for w, us in verify_us.items():
                self.state.verify_us[w] = us
        self.state.draft_us_fixed = draft_us_fixed
        self.state.draft_us_per_token = draft_us_per_token

    def observe(self, depth: int, accepted: int) -> None:
        _check(load_library().vw4_depth_ctl_observe(ctypes.byref(self.state), depth, accepted),
               "vw4_depth_ctl_observe")

    def expected(self, depth: int):
        t, us = ctypes.c_double(), ctypes.c_double()
        _check(load_library().vw4_depth_ctl_expected(ctypes.byref(self.state), depth,
                                                     ctypes.byref(t), ctypes.byref(us)),
               "vw4_depth_ctl_expected")
        return t.value, us.value

    def choose(self) -> int:
        k = load_library().vw4_depth_ctl_choose(ctypes.byref(self.state))
        if k < 0:
            raise VW4Error(1, "vw4_depth_ctl_choose", "invalid controller state")
        return k


class PreparedGemm:
    """One weight matrix bound to the C ABI once: the vw4_weight descriptor,
    a workspace sized for up to M_max verify rows and the stream handle are
    kept, so every call is a single ctypes call with integer pointers.  The
    computation is verify_gemm_w4 (same entry point, same kernels)."""

    def __init__(self, fmt: int, q: torch.Tensor, scales: torch.Tensor, tensor_scale: float,
                 M_max: int = 8, stream=None):
        self._keep = (q, scales)
        self.N, self.K = q.shape[0], q.shape[1] * 2
        self.W = make_weight(fmt, q, scales, tensor_scale, self.N, self.K)
        need = vw4_workspace_bytes(OP_GEMM, M_max, self.N, self.K)
        self.ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=q.device)
        self.ws_ptr, self.ws_bytes = self.ws.data_ptr(), self.ws.numel()
        self.stream = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        self._fn = load_library().verify_gemm_w4
        self._Wref = ctypes.byref(self.W)

    def __call__(self, A: torch.Tensor, out: torch.Tensor, row_argmax: torch.Tensor | None = None):
        code = self._fn(self._Wref, A.data_ptr(), A.shape[0], A.stride(0), out.data_ptr(),
                        out.stride(0), None if row_argmax is None else row_argmax.data_ptr(),
                        self.ws_ptr, self.ws_bytes, self.stream)
        if code:
            _check(code, "verify_gemm_w4")
        return out


def verify_gemm_w4_noalloc(fmt: int, q: torch.Tensor, scales: torch.Tensor, tensor_scale: float,
                           A: torch.Tensor, out: torch.Tensor | None = None,
                           row_argmax: torch.Tensor | None = None, stream=None):
    """verify_gemm_w4 without a workspace: for callers that cannot allocate
    device memory.  The library's fixed device scratch array is used instead;
    calls that may overlap on the GPU must be serialized by the caller."""
    N, K = q.shape[0], q.shape[1] * 2
    M = A.shape[0]
    if A.dtype != torch.bfloat16:
        raise ValueError("A must be bfloat16")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    W = make_weight(fmt, q, scales, tensor_scale, N, K)
    code = load_library().verify_gemm_w4_noalloc(ctypes.byref(W), _ptr(A), M, A.stride(0),
                                                 _ptr(out), out.stride(0), _ptr(row_argmax),
                                                 _stream(stream))
    _check(code, "verify_gemm_w4_noalloc")
    return out


def verify_moe_w4(fmt: int, q: torch.Tensor, scales: torch.Tensor, tensor_scale: float, E: int,
                  A: torch.Tensor, rows_are_pairs: int, expert_ids: torch.Tensor,
                  gates: torch.Tensor | None, combine: int, out: torch.Tensor | None = None,
                  workspace=None, stream=None):
    """q u8 [E, N, K/2] (or [E*N, K/2]); expert_ids int32 [M, topk]; see vw4.h."""
    K = q.shape[-1] * 2
    N = q.numel() // (K // 2) // E
    M, topk = expert_ids.shape
    rows = M if combine else M * topk
    if out is None:
        out = torch.empty((rows, N), dtype=torch.float32, device=A.device)
    W = make_weight(fmt, q, scales, tensor_scale, N, K)
    need = vw4_workspace_bytes(OP_MOE, M * topk, N, K)
    ws = _workspace(workspace, need, A.device)
    code = load_library().verify_moe_w4(ctypes.byref(W), E, _ptr(A), A.stride(0), rows_are_pairs,
                                        _ptr(expert_ids), _ptr(gates), M, topk, combine,
                                        _ptr(out), out.stride(0), _ptr(ws), ws.numel(),
                                        _stream(stream))
    _check(code, "verify_moe_w4")
    return out


def accept_greedy(target_logits: torch.Tensor | None, drafts: torch.Tensor,
                  target_argmax: torch.Tensor | None = None, B: int | None = None,
                  V: int | None = None, tokens=None, length=None, stream=None):
    """target_logits f32 [B, Kd+1, V]; drafts int32 [B, Kd] -> (tokens [B, Kd+1], len [B])."""
    if target_logits is not None:
        B, R, V = target_logits.shape
    Kd = drafts.shape[1]
    dev = drafts.device
    if tokens is None:
        tokens = torch.empty((B, Kd + 1), dtype=torch.int32, device=dev)
    if length is None:
        length = torch.empty((B,), dtype=torch.int32, device=dev)
    code = load_library().accept_greedy(_ptr(target_logits), _ptr(drafts), _ptr(target_argmax), B,
                                        Kd, V, _ptr(tokens), _ptr(length), _stream(stream))
    _check(code, "accept_greedy")
    return tokens, length


def accept_rejection(target_logits: torch.Tensor, draft_logits: torch.Tensor | None,
                     drafts: torch.Tensor, temperature: float, top_p: float, seed: int,
                     offset: int = 0, top_k: int = 0, min_p: float = 0.0, tokens=None,
                     length=None, workspace=None, stream=None):
    """Leviathan/Chen rejection accept; returns (tokens [B, Kd+1], len [B])."""
    B, R, V = target_logits.shape
    Kd = R - 1
    dev = target_logits.device
    if tokens is None:
        tokens = torch.empty((B, Kd + 1), dtype=torch.int32, device=dev)
    if length is None:
        length = torch.empty((B,), dtype=torch.int32, device=dev)
    prm = Sampling(float(temperature), float(top_p), int(top_k), float(min_p))
    need = vw4_workspace_bytes(OP_REJECTION, B, Kd, V)
    ws = _workspace(workspace, need, dev)
    code = load_library().accept_rejection(_ptr(target_logits), _ptr(draft_logits), _ptr(drafts),
                                           B, Kd, V, ctypes.byref(prm), int(seed), int(offset),
                                           _ptr(tokens), _ptr(length), _ptr(ws), ws.numel(),
                                           _stream(stream))
    _check(code, "accept_rejection")
    return tokens, length


def accept_rejection_blockmax(target_logits: torch.Tensor, target_bmax: torch.Tensor,
                              draft_logits: torch.Tensor | None, draft_bmax: torch.Tensor | None,
                              drafts: torch.Tensor, temperature: float, top_p: float, seed: int,
                              offset: int = 0, top_k: int = 0, min_p: float = 0.0, tokens=None,
                              length=None, workspace=None, stream=None):
    """accept_rejection with the block maxima of every logits row (as
    verify_gemm_w4_blockmax writes them) -> (tokens [B, Kd+1], len [B])."""
    B, R, V = target_logits.shape
    Kd = R - 1
    nb = (V + 15) // 16
    if target_bmax.numel() != B * R * nb or (Kd and draft_bmax.numel() != B * Kd * nb):
        raise ValueError("block maxima must be [B, rows, ceil(V/16)]")
    dev = target_logits.device
    if tokens is None:
        tokens = torch.empty((B, Kd + 1), dtype=torch.int32, device=dev)
    if length is None:
        length = torch.empty((B,), dtype=torch.int32, device=dev)
    prm = Sampling(float(temperature), float(top_p), int(top_k), float(min_p))
    ws = _workspace(workspace, vw4_workspace_bytes(OP_REJECTION, B, Kd, V), dev)
    code = load_library().accept_rejection_blockmax(
        _ptr(target_logits), _ptr(target_bmax), _ptr(draft_logits), _ptr(draft_bmax),
        _ptr(drafts), B, Kd, V, ctypes.byref(prm), int(seed), int(offset), _ptr(tokens),
        _ptr(length), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "accept_rejection_blockmax")
    return tokens, length


def accept_rejection_topk(target_ids: torch.Tensor, target_vals: torch.Tensor,
                          draft_ids: torch.Tensor | None, draft_vals: torch.Tensor | None,
                          drafts: torch.Tensor, V: int, temperature: float, top_p: float,
                          seed: int, offset: int = 0, top_k: int = 0, min_p: float = 0.0,
                          tokens=None, length=None, workspace=None, stream=None):
    """accept_rejection over rows given as top-k lists: target ids/logits
    int32/fp32 [B, Kd+1, Kt], draft ids/logits [B, Kd, Kt], vocabulary size V;
    returns (tokens [B, Kd+1], len [B])."""
    B, R, Kt = target_ids.shape
    Kd = R - 1
    dev = target_ids.device
    if tokens is None:
        tokens = torch.empty((B, Kd + 1), dtype=torch.int32, device=dev)
    if length is None:
        length = torch.empty((B,), dtype=torch.int32, device=dev)
    prm = Sampling(float(temperature), float(top_p), int(top_k), float(min_p))
    need = vw4_workspace_bytes(OP_REJECTION_TOPK, B, Kd, Kt)
    ws = _workspace(workspace, need, dev)
    code = load_library().accept_rejection_topk(
        _ptr(target_ids), _ptr(target_vals), _ptr(draft_ids), _ptr(draft_vals), _ptr(drafts), B,
        Kd, Kt, int(V), ctypes.byref(prm), int(seed), int(offset), _ptr(tokens), _ptr(length),
        _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "accept_rejection_topk")
    return tokens, length


# vw4_row_record (see vw4.h): 32 bytes per row
ROW_RECORD_DTYPE = [("max", "<f4"), ("cut", "<i4"), ("tau", "<u8"), ("kept_sum", "<u8"),
                    ("topk_key", "<u4"), ("topk_idx", "<i4")]


def vw4_rejection_row_records(workspace, B: int, Kd: int, V: int, stream=None):
    """The row records of the accept_rejection call that last used `workspace`
    (a Workspace or a uint8 tensor) with the same B, Kd, V: a CUDA uint8
    tensor [rows, 32]; view it on the host with ROW_RECORD_DTYPE.  Rows: the
    target rows (b, i <= Kd) in order, then the draft rows (b, i < Kd)."""
    buf = workspace.buf if isinstance(workspace, Workspace) else workspace
    rows = B * (2 * Kd + 1)
    rec = torch.empty((rows, 32), dtype=torch.uint8, device=buf.device)
    _check(load_library().vw4_rejection_row_records(_ptr(buf), buf.numel(), B, Kd, V, _ptr(rec),
                                                    _stream(stream)),
           "vw4_rejection_row_records")
    return rec


def vw4_get_device_status(stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check(load_library().vw4_get_device_status(ctypes.byref(bits), _stream(stream)),
           "vw4_get_device_status")
    return int(bits.value)


def vw4_q4_0_from_blocks(blocks: torch.Tensor, N: int, K: int, stream=None):
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=blocks.device)
    d = torch.empty((N, K // 32), dtype=torch.float16, device=blocks.device)
    _check(load_library().vw4_q4_0_from_blocks(_ptr(blocks), N, K, _ptr(q), _ptr(d),
                                               _stream(stream)), "vw4_q4_0_from_blocks")
    return q, d


def vw4_own_exp(x: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    """The accept step's own fp32 exp, elementwise on a float32 CUDA tensor."""
    if out is None:
        out = torch.empty_like(x)
    _check(load_library().vw4_own_exp(_ptr(x), _ptr(out), x.numel(), _stream(stream)),
           "vw4_own_exp")
    return out


def vw4_own_mass_pairs(x: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    """The accept step's integer masses floor(own_exp(x) 2^40) by its packed
    fp32-pair path, elementwise on a float32 CUDA tensor (int64 result)."""
    if out is None:
        out = torch.empty(x.shape, dtype=torch.int64, device=x.device)
    _check(load_library().vw4_own_mass_pairs(_ptr(x), _ptr(out), x.numel(), _stream(stream)),
           "vw4_own_mass_pairs")
    return out


def vw4_build_flags() -> int:
    """BUILD_CHECKS when the loaded library is the checks build."""
    return int(load_library().vw4_build_flags())


def vw4_set_wait_limit_ns(ns: int):
    load_library().vw4_set_wait_limit_ns(int(ns))


def vw4_test_inject_stall(calls: int):
    """Test hook: the next `calls` GEMM launches wait on a barrier nothing
    completes until their bounded wait runs out (see vw4.h)."""
    load_library().vw4_test_inject_stall(int(calls))
