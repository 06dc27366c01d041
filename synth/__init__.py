"""Seeded synthetic inputs for the verify GEMM and the accept step.

Shared by the tests, the benchmark and the oracle checks.  This module holds
none of the verification arithmetic: it only draws random numbers and packs
them into the storage formats the library consumes (the quantizers below are
input synthesis -- both sides of every parity check read the same packed
bytes, so nothing depends on how these round).

Recipes (the sizes are the ones the pages' workloads use):
  * weights  ~ N(0, 0.02), quantized to nvfp4 (E2M1 values, one E4M3 scale per
    16 k, one fp32 tensor scale) or to Q4_0 (32-element blocks, fp16 scale).
  * activations: bf16 rounding of N(0, 1).
  * greedy drafts: agree with a given argmax with probability 0.8, otherwise a
    uniform id different from it.
  * MoE routing: router logits N(0, 1) [M, E], softmax in fp64, top-k by
    descending probability (ties to the lower expert), gates = the kept
    probabilities renormalized to sum 1.
  * stochastic accept: target logits N(0, 3), draft logits = target + N(0, 1),
    drafts sampled from softmax(draft / T) with Gumbel-max (a float stand-in
    for the draft model's own sampler).
"""
from __future__ import annotations

import numpy as np

E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float32)
_E2M1_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
_E2M1_ODD_MIDS = np.array([0.75, 1.75, 3.5], np.float32)  # ties that round up to an even code


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ dense
def normal_weights(g: np.random.Generator, N: int, K: int, std: float = 0.02) -> np.ndarray:
    return (g.standard_normal((N, K), dtype=np.float32) * np.float32(std))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even) and return the raw uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def activations(g: np.random.Generator, M: int, K: int) -> np.ndarray:
    """bf16 bits [M, K] of N(0, 1) samples."""
    return bf16_bits(g.standard_normal((M, K), dtype=np.float32))


def _e4m3_encode(x: np.ndarray) -> np.ndarray:
    import torch  # the library cast is the encoder; torch is plumbing here
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_values(codes: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy()


def _e2m1_encode(y: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code (ties to the even code), saturating at +-6."""
    a = np.abs(y)
    code = np.searchsorted(_E2M1_MIDS, a, side="left").astype(np.uint8)
    code += np.isin(a, _E2M1_ODD_MIDS).astype(np.uint8)
    code = np.minimum(code, 7).astype(np.uint8)
    sign = (np.signbit(y) & (code != 0)).astype(np.uint8) << np.uint8(3)
    return code | sign


def quantize_nvfp4(w: np.ndarray, rows_per_chunk: int = 4096):
    """w fp32 [N, K] (K % 16 == 0) -> (Wq u8 [N, K/2], S u8(e4m3) [N, K/16], tensor_scale)."""
    N, K = w.shape
    assert K % 16 == 0
    amax = float(np.max(np.abs(w))) if w.size else 0.0
    ts = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    Wq = np.empty((N, K // 2), np.uint8)
    S = np.empty((N, K // 16), np.uint8)
    for r0 in range(0, N, rows_per_chunk):
        blk = w[r0:r0 + rows_per_chunk].reshape(-1, K // 16, 16)
        bamax = np.max(np.abs(blk), axis=2)
        s_codes = _e4m3_encode(bamax / np.float32(6.0) / ts)
        s_vals = _e4m3_values(s_codes)
        denom = (s_vals * ts)[..., None]
        with np.errstate(divide="ignore", invalid="ignore"):
            y = np.where(denom > 0, blk / denom, np.float32(0.0)).astype(np.float32)
        codes = _e2m1_encode(y).reshape(blk.shape[0], K)
        Wq[r0:r0 + rows_per_chunk] = codes[:, 0::2] | (codes[:, 1::2] << np.uint8(4))
        S[r0:r0 + rows_per_chunk] = s_codes
    return Wq, S, float(ts)


def quantize_q4_0(w: np.ndarray, rows_per_chunk: int = 4096):
    """w fp32 [N, K] (K % 32 == 0) -> (qs u8 [N, K/2], d f16 [N, K/32]); byte j of a
    block holds element j (low nibble) and element j+16 (high nibble)."""
    N, K = w.shape
    assert K % 32 == 0
    qs = np.empty((N, K // 2), np.uint8)
    d = np.empty((N, K // 32), np.float16)
    for r0 in range(0, N, rows_per_chunk):
        blk = w[r0:r0 + rows_per_chunk].reshape(-1, K // 32, 32)
        idx = np.argmax(np.abs(blk), axis=2)
        mx = np.take_along_axis(blk, idx[..., None], axis=2)[..., 0]
        dd = (mx / np.float32(-8.0)).astype(np.float16)
        dv = dd.astype(np.float32)[..., None]
        with np.errstate(divide="ignore", invalid="ignore"):
            y = np.where(dv != 0, blk / dv, np.float32(0.0))
        q = np.clip(np.rint(y) + 8, 0, 15).astype(np.uint8)
        packed = q[..., :16] | (q[..., 16:] << np.uint8(4))
        qs[r0:r0 + rows_per_chunk] = packed.reshape(-1, K // 2)
        d[r0:r0 + rows_per_chunk] = dd
    return qs, d


def linear(seed: int, N: int, K: int, fmt: str = "nvfp4", std: float = 0.02):
    """A quantized N(0, std) linear layer [N, K] of the given format."""
    g = rng(seed)
    w = normal_weights(g, N, K, std)
    if fmt == "nvfp4":
        Wq, S, ts = quantize_nvfp4(w)
        return Wq, S, ts
    qs, d = quantize_q4_0(w)
    return qs, d, 1.0


# ----------------------------------------------------------- accept inputs
def greedy_drafts(g: np.random.Generator, argmax: np.ndarray, V: int, p_agree: float = 0.8):
    """argmax int [B, Kd] -> drafts int32 [B, Kd]."""
    argmax = np.asarray(argmax, np.int64)
    agree = g.random(argmax.shape) < p_agree
    other = (argmax + 1 + g.integers(0, V - 1, size=argmax.shape)) % V
    return np.where(agree, argmax, other).astype(np.int32)


def logits(g: np.random.Generator, shape, std: float) -> np.ndarray:
    return g.standard_normal(shape, dtype=np.float32) * np.float32(std)


def stochastic_case(seed: int, B: int, Kd: int, V: int, temperature: float = 0.6,
                    target_std: float = 3.0, noise_std: float = 1.0):
    """target f32 [B, Kd+1, V], draft f32 [B, Kd, V], drafts int32 [B, Kd]."""
    g = rng(seed)
    target = logits(g, (B, Kd + 1, V), target_std)
    draft = target[:, :Kd, :] + logits(g, (B, Kd, V), noise_std)
    drafts = np.empty((B, Kd), np.int32)
    for b in range(B):
        for i in range(Kd):
            gum = -np.log(-np.log(g.random(V)))
            drafts[b, i] = int(np.argmax(draft[b, i].astype(np.float64) / temperature + gum))
    return target, np.ascontiguousarray(draft), drafts


# --------------------------------------------------------------------- MoE
def routing(seed: int, M: int, E: int, topk: int):
    """expert_ids int32 [M, topk], gates f32 [M, topk]."""
    g = rng(seed)
    lg = g.standard_normal((M, E)).astype(np.float64)
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :topk]
    gp = np.take_along_axis(p, order, axis=1)
    gates = (gp / gp.sum(axis=1, keepdims=True)).astype(np.float32)
    return order.astype(np.int32), gates
