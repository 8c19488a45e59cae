"""Independent double-precision brute force for pinning the oracle on tiny inputs.

Written from the closed forms, not from the oracle's code:
  * E2M1 value of a 4-bit code c = (s, e1 e0, m): (-1)^s * 2^(e-1) * (1 + m/2)
    for e > 0 and (-1)^s * m/2 for e = 0 (the subnormal);
  * E8M0 value of a byte b: 2^(b - 127), b = 255 is NaN;
  * routing: a full stable sort of all E logits (descending, lower index on
    ties) and a double-precision softmax;
  * the expert MLP as dense float64 matrix products (numpy), with the SwiGLU
    intermediate rounded to bf16.
"""
from __future__ import annotations

import numpy as np


def e2m1_closed_form(code: int) -> float:
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = (2.0 ** (e - 1)) * (1.0 + m / 2.0) if e > 0 else m * 0.5
    return -mag if s else mag


def e8m0_closed_form(b: int) -> float:
    return float("nan") if b == 255 else 2.0 ** (b - 127)


def decode_mxfp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes uint8 [..., R, K/2], scales uint8 [..., R, K/32] -> float64 [..., R, K]."""
    lo = codes & 0x0F
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    table = np.array([e2m1_closed_form(c) for c in range(16)], np.float64)
    vals = table[nib]
    sc = np.array([e8m0_closed_form(b) for b in range(256)], np.float64)[scales]
    return vals * np.repeat(sc, 32, axis=-1)


def bf16_round(a) -> np.ndarray:
    """Round float64/float32 values to bf16 (nearest even, via float32) -> float64."""
    f = np.asarray(a, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint32) << 16
    return r.view(np.float32).astype(np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def route(logits: np.ndarray, K: int, with_shared: bool, renormalize: bool = True):
    T, E = logits.shape
    l64 = logits.astype(np.float64)
    ids = np.empty((T, K + int(with_shared)), np.int64)
    w = np.empty((T, K + int(with_shared)), np.float64)
    for t in range(T):
        finite = np.isfinite(l64[t])
        m = l64[t][finite].max() if finite.any() else 0.0
        ex = np.where(np.isneginf(l64[t]), 0.0, np.exp(l64[t] - m))
        p = ex / ex.sum()
        order = np.lexsort((np.arange(E), -l64[t]))  # by -logit, then by index
        sel = order[:K]
        ids[t, :K] = sel
        w[t, :K] = p[sel] / p[sel].sum() if renormalize else p[sel]
        if with_shared:
            ids[t, K] = E
            w[t, K] = 1.0
    return ids, w


def permute(ids: np.ndarray, Et: int, tile_m: int):
    T, Kt = ids.shape
    flat = ids.reshape(-1).astype(np.int64)
    P = flat.size
    counts = np.bincount(flat, minlength=Et)
    padded = (counts + tile_m - 1) // tile_m * tile_m
    offsets = np.concatenate([[0], np.cumsum(padded)])
    cap = P + Et * (tile_m - 1)
    order = np.lexsort((np.arange(P), flat))  # by expert, then by pair index
    sorted_pairs = np.full(cap, -1, np.int64)
    inv = np.empty(P, np.int64)
    starts = offsets[:-1]
    rank = np.arange(P) - np.concatenate([[0], np.cumsum(counts)])[:-1][flat[order]]
    pos = starts[flat[order]] + rank
    sorted_pairs[pos] = order
    inv[order] = pos
    num_tiles = int(offsets[-1] // tile_m)
    tile_expert = np.full(cap // tile_m, -1, np.int64)
    rows = np.arange(num_tiles) * tile_m
    tile_expert[:num_tiles] = np.searchsorted(offsets, rows, side="right") - 1
    return dict(sorted_pairs=sorted_pairs, offsets=offsets, inv=inv, tile_expert=tile_expert,
                num_tiles=num_tiles)


def silu64(g):
    return g / (1.0 + np.exp(-g))


def expert_mlp(x64: np.ndarray, w13: np.ndarray, s13: np.ndarray, w2: np.ndarray, s2: np.ndarray):
    """x64 [n, H] float64 -> y [n, H] float64 for one expert (h rounded to bf16)."""
    W13 = decode_mxfp4(w13, s13)  # [2I, H]
    W2 = decode_mxfp4(w2, s2)     # [H, I]
    I = W13.shape[0] // 2
    g = x64 @ W13[:I].T
    u = x64 @ W13[I:].T
    h = bf16_round(silu64(g) * u)
    return h @ W2.T


def ffn(x_bits, w13, s13, w2, s2, ids, w):
    x64 = bf16_bits_to_f64(x_bits)
    T, H = x64.shape
    out = np.zeros((T, H), np.float64)
    for t in range(T):
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            out[t] += float(w[t, j]) * expert_mlp(x64[t:t + 1], w13[e], s13[e], w2[e], s2[e])[0]
    return out


# ------------------------------------------------ MXFP4-quantised activations
# Written from the E2M1 format (1 sign, 2 exponent, 1 mantissa bit, bias 1) and
# the OCP Microscaling v1.0 scale rule, not from the oracle's search over the
# value table: rounding to nearest-even within each binade, where the spacing
# is fixed, and the shared exponent found by a search on its defining
# inequality 2^(e+2) <= amax < 2^(e+3).

def e2m1_round_binade(v: float) -> int:
    """E2M1 code of v: round to the binade's grid (spacing 0.5 below 2, 1 in
    [2, 4), 2 in [4, 8)) with Python's round-half-even, saturate at 6."""
    a = abs(float(v))
    if a < 2.0:
        q = round(a * 2.0) / 2.0      # multiples of 0.5; even multiple = even code
    elif a < 4.0:
        q = float(round(a))
    else:
        q = round(a / 2.0) * 2.0
    q = min(q, 6.0)
    mags = [e2m1_closed_form(c) for c in range(8)]
    code = mags.index(q)
    return code | (8 if np.signbit(v) else 0)


def mx_shared_exponent(amax: float) -> int:
    """Smallest e in [-127, 127] with amax < 2^(e+3), i.e. 2^(e+2) <= amax
    unless clamped."""
    e = -127
    while e < 127 and not (amax < 2.0 ** (e + 3)):
        e += 1
    return e


def quantize_mxfp4(v: np.ndarray):
    """float [..., n] -> (codes uint8 [..., n/2], scales uint8 [..., n/32])."""
    v = np.asarray(v, np.float64)
    n = v.shape[-1]
    rows = v.reshape(-1, n)
    codes = np.zeros((rows.shape[0], n // 2), np.uint8)
    scales = np.zeros((rows.shape[0], n // 32), np.uint8)
    for r in range(rows.shape[0]):
        for b in range(n // 32):
            blk = rows[r, 32 * b:32 * b + 32]
            amax = float(np.abs(blk).max())
            if amax == 0.0:
                continue
            e = mx_shared_exponent(amax)
            scales[r, b] = e + 127
            cs = [e2m1_round_binade(x / 2.0 ** e) for x in blk]
            for i in range(16):
                codes[r, 16 * b + i] = cs[2 * i] | (cs[2 * i + 1] << 4)
    return codes.reshape(*v.shape[:-1], n // 2), scales.reshape(*v.shape[:-1], n // 32)
