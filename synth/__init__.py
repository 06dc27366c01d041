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


def _e2m1_codes(y):
    """Nearest E2M1 code of a float tensor (ties to the even code), saturating
    at +-6.  The thresholds are the midpoints of 0, .5, 1, 1.5, 2, 3, 4, 6;
    at a midpoint the comparison picks the even code."""
    import torch
    a = y.abs()
    code = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8) + (a > 1.25).to(torch.uint8)
            + (a >= 1.75).to(torch.uint8) + (a > 2.5).to(torch.uint8)
            + (a >= 3.5).to(torch.uint8) + (a > 5.0).to(torch.uint8))
    sign = ((y < 0) & (code != 0)).to(torch.uint8)
    return code | (sign << 3)


def quantize_nvfp4(w: np.ndarray, amax: float | None = None):
    """w fp32 [N, K] (K % 16 == 0) -> (Wq u8 [N, K/2], S u8(e4m3) [N, K/16], tensor_scale).
    amax (the whole matrix's max |w|) may be given when w is one chunk of a larger
    matrix.  torch CPU ops are used as multithreaded plumbing; the e4m3 encoder is
    torch's float8_e4m3fn cast."""
    import torch
    N, K = w.shape
    assert K % 16 == 0
    t = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32))
    if amax is None:
        amax = float(t.abs().max()) if t.numel() else 0.0
    ts = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    blk = t.view(N, K // 16, 16)
    bamax = blk.abs().amax(dim=2)
    s8 = (bamax / 6.0 / float(ts)).to(torch.float8_e4m3fn)
    sv = s8.to(torch.float32) * float(ts)
    y = torch.where(sv[..., None] > 0, blk / sv[..., None].clamp_min(1e-38),
                    torch.zeros((), dtype=torch.float32))
    codes = _e2m1_codes(y).view(N, K)
    Wq = (codes[:, 0::2] | (codes[:, 1::2] << 4)).numpy()
    return np.ascontiguousarray(Wq), s8.view(torch.uint8).numpy().copy(), float(ts)


def quantize_q4_0(w: np.ndarray):
    """w fp32 [N, K] (K % 32 == 0) -> (qs u8 [N, K/2], d f16 [N, K/32]); byte j of a
    block holds element j (low nibble) and element j+16 (high nibble).
    d = (the block's largest-magnitude value) / -8, q = clamp(round(w/d) + 8)."""
    import torch
    N, K = w.shape
    assert K % 32 == 0
    t = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32))
    blk = t.view(N, K // 32, 32)
    idx = blk.abs().argmax(dim=2, keepdim=True)
    mx = torch.gather(blk, 2, idx)[..., 0]
    dd = (mx / -8.0).to(torch.float16)
    dv = dd.to(torch.float32)[..., None]
    y = torch.where(dv != 0, blk / torch.where(dv != 0, dv, torch.ones_like(dv)),
                    torch.zeros((), dtype=torch.float32))
    q = (torch.round(y) + 8).clamp(0, 15).to(torch.uint8)
    packed = q[..., :16] | (q[..., 16:] << 4)
    return packed.reshape(N, K // 2).numpy().copy(), dd.numpy().copy()


LINEAR_CHUNK_ROWS = 2048


def _chunk_weights(seed: int, j: int, n: int, K: int, std: float) -> np.ndarray:
    """Rows [j*2048, j*2048 + n) of a synthetic linear: chunk j has its own
    child stream of the seed, so chunks can be drawn in any order or in
    parallel and the matrix is the same."""
    return normal_weights(rng([seed, j]), n, K, std)


def linear(seed: int, N: int, K: int, fmt: str = "nvfp4", std: float = 0.02, threads: int = 8):
    """A quantized N(0, std) linear layer [N, K] of the given format.  Rows are
    drawn in 2048-row chunks (a first pass finds the global max for the nvfp4
    tensor scale), so large matrices never exist in fp32 all at once."""
    from concurrent.futures import ThreadPoolExecutor
    C = LINEAR_CHUNK_ROWS
    chunks = [(j, min(C, N - j * C)) for j in range((N + C - 1) // C)]
    with ThreadPoolExecutor(threads) as ex:
        if fmt == "nvfp4":
            amax = max(ex.map(lambda jc: float(np.max(np.abs(_chunk_weights(seed, jc[0], jc[1],
                                                                              K, std)))), chunks))
            Wq = np.empty((N, K // 2), np.uint8)
            S = np.empty((N, K // 16), np.uint8)
            ts = [1.0]

            def quant(jc):
                j, n = jc
                Wq[j * C:j * C + n], S[j * C:j * C + n], ts[0] = quantize_nvfp4(
                    _chunk_weights(seed, j, n, K, std), amax=amax)
            list(ex.map(quant, chunks))
            return Wq, S, ts[0]
        qs = np.empty((N, K // 2), np.uint8)
        d = np.empty((N, K // 32), np.float16)

        def quant4(jc):
            j, n = jc
            qs[j * C:j * C + n], d[j * C:j * C + n] = quantize_q4_0(
                _chunk_weights(seed, j, n, K, std))
        list(ex.map(quant4, chunks))
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


def topk_lists_case(seed: int, B: int, Kd: int, Kt: int, V: int, temperature: float = 0.6,
                    target_std: float = 3.0, noise_std: float = 1.0, swap: float = 0.2):
    """Rows given as top-Kt lists, as a top-k stage would hand them on: target
    ids int32 [B, Kd+1, Kt] (distinct per row, uniform over the vocabulary)
    with logits fp32 sorted descending; draft lists [B, Kd, Kt] holding the
    target row's ids, a fraction `swap` of them replaced by other ids, with
    the target logits plus N(0, noise_std); drafts int32 [B, Kd] picked from
    the draft lists by the Gumbel-max rule at `temperature`."""
    g = rng(seed)
    t_ids = np.empty((B, Kd + 1, Kt), np.int32)
    t_vals = np.empty((B, Kd + 1, Kt), np.float32)
    d_ids = np.empty((B, Kd, Kt), np.int32)
    d_vals = np.empty((B, Kd, Kt), np.float32)
    drafts = np.empty((B, Kd), np.int32)
    for b in range(B):
        for r in range(Kd + 1):
            ids = g.choice(V, size=Kt, replace=False).astype(np.int32)
            vals = np.sort(g.standard_normal(Kt).astype(np.float32) * np.float32(target_std))[::-1]
            t_ids[b, r], t_vals[b, r] = ids, vals
            if r < Kd:
                di = ids.copy()
                sw = g.random(Kt) < swap
                if sw.any():
                    pool = np.setdiff1d(np.arange(V, dtype=np.int32), ids)
                    di[sw] = g.choice(pool, size=int(sw.sum()), replace=False)
                dv = vals + g.standard_normal(Kt).astype(np.float32) * np.float32(noise_std)
                d_ids[b, r], d_vals[b, r] = di, dv
                gum = -np.log(-np.log(g.random(Kt)))
                drafts[b, r] = di[int(np.argmax(dv.astype(np.float64) / temperature + gum))]
    return t_ids, t_vals, d_ids, d_vals, drafts

