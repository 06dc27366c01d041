"""CPU oracle for speculative-decoding verification with 4-bit weights.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` do.  The arithmetic lives in ``vw4_oracle.c`` (plain C, fp64,
``-ffp-contract=off``); this file only builds it with gcc and marshals numpy
arrays through ctypes.  It shares no code with the CUDA path.

Every function states which page and section of the source material it
follows in ``vw4_oracle.c``.  Parity pins live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vw4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_NVFP4 = 1
FMT_Q4_0 = 2


def build(force: bool = False) -> str:
    """Compile vw4_oracle.c into liboracle.so with gcc (OpenMP over outputs)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
               "-shared", "-std=gnu11", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i32, i64, u32, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
    f32, f64 = ctypes.c_float, ctypes.c_double
    sig = {
        "oracle_e2m1": (f64, [u32]),
        "oracle_e4m3": (f64, [u32]),
        "oracle_f16": (f64, [u32]),
        "oracle_bf16": (f64, [u32]),
        "oracle_dequant": (None, [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, f64, P]),
        "oracle_gemm_w4": (None, [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, f64, P,
                                  ctypes.c_int, ctypes.c_int, P, ctypes.c_int, P, P]),
        "oracle_moe_w4": (None, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                 f64, P, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, P, P]),
        "oracle_route_sort": (ctypes.c_int, [P, ctypes.c_int, ctypes.c_int, P, P]),
        "oracle_argmax_f32": (i32, [P, i64]),
        "oracle_accept_greedy": (ctypes.c_int, [P, i64, P, ctypes.c_int, ctypes.c_int, i64, P, P]),
        "oracle_philox4x32_10": (None, [P, P, P]),
        "oracle_own_exp": (f32, [f32]),
        "oracle_row_mass": (u64, [P, i64, f32, u64, P]),
        "oracle_accept_rejection": (ctypes.c_int, [P, i64, P, i64, P, ctypes.c_int, ctypes.c_int,
                                                   i64, f32, f32, u64, u64, u32, P, P]),
        "oracle_sample_drafts": (None, [P, i64, ctypes.c_int, ctypes.c_int, i64, f32, f32, u64,
                                        u64, u32, P]),
        "oracle_own_exp_array": (None, [P, P, i64]),
        "oracle_row_mass_ex": (u64, [P, i64, f32, u64, i64, u64, P]),
        "oracle_accept_rejection_ex": (ctypes.c_int, [P, i64, P, i64, P, ctypes.c_int,
                                                      ctypes.c_int, i64, f32, f32, i64, f32, u64,
                                                      u64, u32, P, P]),
        "oracle_sample_drafts_ex": (None, [P, i64, ctypes.c_int, ctypes.c_int, i64, f32, f32,
                                           i64, f32, u64, u64, u32, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- formats
def e2m1(code: int) -> float:
    return _load().oracle_e2m1(code)


def e4m3(code: int) -> float:
    return _load().oracle_e4m3(code)


def f16(bits: int) -> float:
    return _load().oracle_f16(bits)


def bf16(bits: int) -> float:
    return _load().oracle_bf16(bits)


def dequant(fmt: int, N: int, K: int, q: np.ndarray, scales: np.ndarray,
            tensor_scale: float = 1.0) -> np.ndarray:
    """Dense fp64 [N, K] matrix of the dequantized weights."""
    q = _c(q, np.uint8)
    scales = np.ascontiguousarray(scales)
    w = np.empty((N, K), np.float64)
    _load().oracle_dequant(fmt, N, K, _ptr(q), _ptr(scales), float(tensor_scale), _ptr(w))
    return w


# -------------------------------------------------------------------- GEMM
def gemm_w4(fmt: int, N: int, K: int, q: np.ndarray, scales: np.ndarray, tensor_scale: float,
            A_bits: np.ndarray, cols=None):
    """out[m, j], bound[m, j] (fp64) for A given as raw bf16 bits uint16 [M, lda]."""
    q = _c(q, np.uint8)
    scales = np.ascontiguousarray(scales)
    A_bits = np.ascontiguousarray(A_bits, dtype=np.uint16)
    M, lda = A_bits.shape
    colv = None if cols is None else _c(cols, np.int32)
    nc = N if colv is None else len(colv)
    out = np.empty((M, nc), np.float64)
    bound = np.empty((M, nc), np.float64)
    _load().oracle_gemm_w4(fmt, N, K, _ptr(q), _ptr(scales), float(tensor_scale), _ptr(A_bits),
                           M, lda, _ptr(colv), nc, _ptr(out), _ptr(bound))
    return out, bound


def moe_w4(fmt: int, E: int, N: int, K: int, q, scales, tensor_scale: float, A_bits,
           rows_are_pairs: int, expert_ids, gates, M: int, topk: int, combine: int):
    q = _c(q, np.uint8)
    scales = np.ascontiguousarray(scales)
    A_bits = np.ascontiguousarray(A_bits, dtype=np.uint16)
    ids = _c(expert_ids, np.int32)
    g = _c(gates, np.float32)
    rows = M if combine else M * topk
    out = np.empty((rows, N), np.float64)
    bound = np.empty((rows, N), np.float64)
    _load().oracle_moe_w4(fmt, E, N, K, _ptr(q), _ptr(scales), float(tensor_scale), _ptr(A_bits),
                          A_bits.shape[1], rows_are_pairs, _ptr(ids), _ptr(g), M, topk, combine,
                          _ptr(out), _ptr(bound))
    return out, bound


def route_sort(expert_ids, E: int):
    ids = _c(expert_ids, np.int32).reshape(-1)
    order = np.empty(len(ids), np.int32)
    seg = np.empty(E + 1, np.int32)
    n = _load().oracle_route_sort(_ptr(ids), len(ids), E, _ptr(order), _ptr(seg))
    return order[:n], seg


# ------------------------------------------------------------------ accept
def argmax_f32(row) -> int:
    row = _c(row, np.float32)
    return int(_load().oracle_argmax_f32(_ptr(row), row.size))


def accept_greedy(target, drafts):
    """target f32 [B, Kd+1, V], drafts i32 [B, Kd] -> tokens [B, Kd+1], len [B], n_bad."""
    target = _c(target, np.float32)
    B, R, V = target.shape
    Kd = R - 1
    drafts = _c(drafts, np.int32).reshape(B, Kd)
    tokens = np.empty((B, Kd + 1), np.int32)
    ln = np.empty(B, np.int32)
    bad = _load().oracle_accept_greedy(_ptr(target), R * V, _ptr(drafts), B, Kd, V,
                                       _ptr(tokens), _ptr(ln))
    return tokens, ln, bad


def philox4x32_10(ctr, key):
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.empty(4, np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def own_exp(x: float) -> float:
    return float(_load().oracle_own_exp(float(x)))


def own_exp_array(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    y = np.empty_like(x)
    _load().oracle_own_exp_array(_ptr(x), _ptr(y), x.size)
    return y


def top_p_fixed(top_p: float) -> int:
    """P = round(top_p * 2^32), saturating at 2^32 (keep everything)."""
    pd = float(np.float32(top_p)) * 4294967296.0
    return (1 << 32) if pd >= 4294967296.0 else int(np.floor(pd + 0.5))


def row_mass(logits, temperature: float, top_p: float, top_k: int = 0, min_p: float = 0.0):
    """Integer masses W (uint64 [V]) after top-k / temperature+softmax / top-p /
    min-p, and their kept sum."""
    logits = _c(logits, np.float32)
    invT = float(np.float32(1.0 / float(np.float32(temperature))))
    W = np.empty(logits.size, np.uint64)
    mp = top_p_fixed(min_p) if min_p > 0 else 0
    S = _load().oracle_row_mass_ex(_ptr(logits), logits.size, invT, top_p_fixed(top_p),
                                   int(top_k), mp, _ptr(W))
    return W, int(S)


def accept_rejection(target, draft, drafts, temperature: float, top_p: float, seed: int,
                     offset: int, broadcast_rows: bool = False, B: int | None = None,
                     b_base: int = 0, top_k: int = 0, min_p: float = 0.0):
    """target f32 [B, Kd+1, V], draft f32 [B, Kd, V] (or one shared [Kd+1, V] / [Kd, V]
    pair reused by every sequence when broadcast_rows=True, with B given).  Sequence b
    draws from Philox counter index b_base + b."""
    target = _c(target, np.float32)
    draft = _c(draft, np.float32)
    if broadcast_rows:
        R, V = target.shape
        Kd = R - 1
        ld_tb = ld_db = 0
        assert B is not None
    else:
        B, R, V = target.shape
        Kd = R - 1
        ld_tb, ld_db = R * V, Kd * V
    drafts = _c(drafts, np.int32).reshape(B, Kd)
    if Kd == 0 and draft.size == 0:
        draft = np.zeros(1, np.float32)
    tokens = np.empty((B, Kd + 1), np.int32)
    ln = np.empty(B, np.int32)
    bad = _load().oracle_accept_rejection_ex(_ptr(target), ld_tb, _ptr(draft), ld_db,
                                             _ptr(drafts), B, Kd, V, float(temperature),
                                             float(top_p), int(top_k), float(min_p), int(seed),
                                             int(offset), int(b_base), _ptr(tokens), _ptr(ln))
    return tokens, ln, bad


def lists_to_rows(ids, vals, V: int):
    """Dense rows [B, R, V] of top-k lists ids / logits [B, R, Kt]: each listed
    logit at its id, -inf at every id not listed (ids outside [0, V) are
    dropped).  The reading of the sampler's sparse [B, K] representation in
    Ollama's mtp.go commit log ("rework the MLX sampler"): the entries a
    top-k stage did not keep have no probability."""
    ids = np.asarray(ids, np.int64)
    vals = np.asarray(vals, np.float32)
    B, R, Kt = ids.shape
    rows = np.full((B, R, V), -np.inf, np.float32)
    for b in range(B):
        for r in range(R):
            for t in range(Kt):
                v = ids[b, r, t]
                if 0 <= v < V:
                    rows[b, r, v] = vals[b, r, t]
    return rows


def accept_rejection_topk(t_ids, t_vals, d_ids, d_vals, drafts, V: int, temperature: float,
                          top_p: float, seed: int, offset: int, b_base: int = 0,
                          top_k: int = 0, min_p: float = 0.0):
    """The accept over top-k lists, by its definition: accept_rejection on the
    dense rows of the lists (lists_to_rows)."""
    target = lists_to_rows(t_ids, t_vals, V)
    B, R, _ = target.shape
    Kd = R - 1
    draft = lists_to_rows(d_ids, d_vals, V) if Kd else np.zeros((B, 0, V), np.float32)
    return accept_rejection(target, draft, drafts, temperature, top_p, seed, offset,
                            b_base=b_base, top_k=top_k, min_p=min_p)


def sample_drafts(draft, temperature: float, top_p: float, seed: int, offset: int,
                  broadcast_rows: bool = False, B: int | None = None, b_base: int = 0,
                  top_k: int = 0, min_p: float = 0.0):
    draft = _c(draft, np.float32)
    if broadcast_rows:
        Kd, V = draft.shape
        ld = 0
        assert B is not None
    else:
        B, Kd, V = draft.shape
        ld = Kd * V
    out = np.empty((B, Kd), np.int32)
    _load().oracle_sample_drafts_ex(_ptr(draft), ld, B, Kd, V, float(temperature),
                                    float(top_p), int(top_k), float(min_p), int(seed),
                                    int(offset), int(b_base), _ptr(out))
    return out
