"""Helpers for the GPU parity tests: device upload and the parity bar.

The bar for the FFN output (bf16 [T, H]) against the oracle:
  per element |gpu - ref| <= 1e-2 * (|ref| + rms(ref)), rms over the whole
  compared tensor, and relative L2 error ||gpu - ref|| / ||ref|| <= 2e-3.
Routing ids, the permutation and every index output are compared bit for bit.
"""
from __future__ import annotations

import numpy as np

FFN_ELEM_TOL = 1e-2
FFN_REL_L2 = 2e-3
ROUTE_W_ATOL = 2e-6


def to_dev(a: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.cuda()


def bf16_dev_to_f64(t) -> np.ndarray:
    import torch
    bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ffn_parity(gpu: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    """Assert the parity bar; return the observed statistics."""
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite GPU output"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = np.abs(gpu - ref)
    bound = FFN_ELEM_TOL * (np.abs(ref) + rms)
    # where the bound is 0 (an all-zero reference) only an exact 0 passes
    ratio = np.divide(err, bound, out=np.where(err > 0, np.inf, 0.0), where=bound > 0)
    worst = float(ratio.max()) if err.size else 0.0
    rel_l2 = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300))
    stats = dict(worst_elem_ratio=worst, rel_l2=rel_l2, identical=float((gpu == ref).mean()))
    assert worst <= 1.0, f"{what}: element error {worst:.3g} x bound {stats}"
    assert rel_l2 <= FFN_REL_L2, f"{what}: rel L2 {rel_l2:.3g} {stats}"
    return stats


def staged_close(a: np.ndarray, b: np.ndarray, what: str = "") -> float:
    """Two GPU results that differ only in the prefill combine's f16 staging
    of y (each term rounded to 11 significant bits before the fp32 sum, then
    both sums rounded to bf16): per element |a - b| <= 2^-7 * (|a| + rms(a)),
    with 2^-11 per term and two bf16 roundings (2^-9 each) well inside.
    Returns the worst ratio."""
    assert a.shape == b.shape and np.isfinite(a).all() and np.isfinite(b).all(), what
    bound = 2.0 ** -7 * (np.abs(a) + float(np.sqrt(np.mean(a ** 2))))
    err = np.abs(a - b)
    ratio = np.divide(err, bound, out=np.where(err > 0, np.inf, 0.0), where=bound > 0)
    worst = float(ratio.max()) if err.size else 0.0
    assert worst <= 1.0, f"{what}: {worst:.3g} x bound"
    return worst


def upload_weights(d: dict) -> dict:
    return {k: to_dev(d[k]) for k in ("w13", "s13", "w2", "s2")}


def edge_tokens(ids: np.ndarray, tile_m: int, n_total: int, seed: int) -> np.ndarray:
    """Tokens whose pairs sit at the edges of the grouped GEMMs' tiles, for a
    sampled comparison at full size: the first and last row in use (the
    first and last work items), then, expert by expert in descending order of
    load, the first and last row of the expert's last (usually partial) tile,
    until three quarters of the budget; random tokens fill the rest.  Rows
    follow the stable grouping by expert, as moe_permute lays them out."""
    T, Kt = ids.shape
    flat = ids.ravel()
    order = np.argsort(flat, kind="stable")  # pair indices grouped by expert, ascending within
    _, starts, counts = np.unique(flat[order], return_index=True, return_counts=True)
    picks = {int(order[0]) // Kt, int(order[-1]) // Kt}
    for i in np.argsort(-counts, kind="stable"):
        if len(picks) >= max(2, n_total * 3 // 4):
            break
        c, s0 = int(counts[i]), int(starts[i])
        last0 = s0 + ((c - 1) // tile_m) * tile_m
        picks.add(int(order[last0]) // Kt)
        picks.add(int(order[s0 + c - 1]) // Kt)
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(T), np.fromiter(picks, int))
    n_more = max(0, min(n_total - len(picks), rest.size))
    tokens = np.concatenate([np.fromiter(picks, int), rng.choice(rest, n_more, replace=False)])
    return np.unique(tokens).astype(np.int32)
