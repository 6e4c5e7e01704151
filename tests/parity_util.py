"""Helpers shared by the GPU parity tests: run the oracle on the exact stored
inputs and compare element by element within the stated tolerances."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

# Tolerances: O max |diff| 1e-2 (bf16 storage) / 4e-3 (fp16 storage); LSE max |diff| 1e-3;
# rows that see no key must be exactly O = 0 and LSE = -inf.
TOL_O = {torch.bfloat16: 1e-2, torch.float16: 4e-3}
TOL_LSE = 1e-3


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact conversion of bf16/fp16 storage to fp64 (CPU)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def oracle_rows(q, k, v, *, causal, q_pos_offset, scale, rows):
    return oracle.attention(f64(q), f64(k), f64(v), causal=causal, q_pos_offset=q_pos_offset, scale=scale,
                            rows=rows)


def gather(o: torch.Tensor, lse: torch.Tensor, rows: np.ndarray):
    """Pick rows (b, h, i) from GPU outputs O [b, sq, hq, d] and LSE [b, hq, sq] as fp64."""
    r = torch.from_numpy(rows).to(o.device)
    og = o[r[:, 0], r[:, 2], r[:, 1]].to(torch.float64).cpu().numpy()
    lg = lse[r[:, 0], r[:, 1], r[:, 2]].to(torch.float64).cpu().numpy()
    return og, lg


def sample_rows(b, hq, sq, n_random=96, seed=0):
    """Deterministic row sample: tile edges, first/last rows, and random rows, over all (b, h) corners."""
    rng = np.random.default_rng(seed)
    edges = {0, 1, sq - 1, sq - 2}
    for t in (63, 64, 127, 128, 129, 255, 256, 257, 383, 384, 511, 512):
        if t < sq:
            edges.add(t)
    rows = set()
    for bi in {0, b - 1}:
        for hi in {0, hq - 1, hq // 2}:
            for i in edges:
                if 0 <= i < sq:
                    rows.add((bi, hi, i))
    for _ in range(n_random):
        rows.add((int(rng.integers(b)), int(rng.integers(hq)), int(rng.integers(sq))))
    return np.array(sorted(rows), dtype=np.int64)


def assert_parity(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    tol_o = TOL_O[dtype]
    masked = np.isneginf(lse_ref)
    if masked.any():
        assert np.all(np.isneginf(lse_gpu[masked])), f"{what}: fully masked rows must have LSE = -inf"
        assert np.all(o_gpu[masked] == 0.0), f"{what}: fully masked rows must have O = 0"
    vis = ~masked
    if vis.any():
        assert np.all(np.isfinite(o_gpu[vis])), f"{what}: non-finite O"
        do = np.abs(o_gpu[vis] - o_ref[vis]).max()
        dl = np.abs(lse_gpu[vis] - lse_ref[vis]).max()
        assert do <= tol_o, f"{what}: O max|diff| {do:.3e} > {tol_o}"
        assert dl <= TOL_LSE, f"{what}: LSE max|diff| {dl:.3e} > {TOL_LSE}"
        return float(do), float(dl)
    return 0.0, 0.0


def default_scale(d):
    return 1.0 / math.sqrt(d)


def e4m3_rounding_bound(qx, kx, vx, causal, off, window, o_ref, l_ref, rows, scale):
    """Per-element bound of what rounding P to e4m3 (and O to bf16) may change in the
    8-bit forward pass, every term from the oracle on the dequantised inputs:

      |O_ic - O_ref,ic| <= 2^-4 * sum_j P_ij |V_jc|               (normal e4m3 codes)
                         + 2^-10 * Pmax_i * sum_{j visible} |V_jc|  (subnormal codes)
                         + 2^-8 * |O_ref,ic| + 1e-6                (bf16 O, fp32 sums)

    The kernel forms p_j = 2^(x_j - m_ref) with a reference maximum no larger than
    the row's maximum, so its largest p is at least 1 and its row sum l at least
    1 / Pmax_i, Pmax_i = exp(m_i - LSE_i); a normal code (p >= 2^-6) is off by at most
    2^-4 of p, a subnormal one by at most 2^-10.  sum_j P_ij |V_jc| is the oracle with
    |V| in place of V; the visible sum of |V| is the oracle at scale 0 (uniform weights
    1 / n_i, LSE = ln n_i) times n_i; m_i is bounded above by LSE at 1000 times the
    scale, divided by 1000."""
    win = window if window else (-1, -1)
    kw = dict(causal=causal, q_pos_offset=off, rows=rows, window=win)
    a_abs, _ = oracle.attention(qx, kx, np.abs(vx), scale=scale, **kw)
    mean_abs, l0 = oracle.attention(qx, kx, np.abs(vx), scale=0.0, **kw)
    _, l_big = oracle.attention(qx, kx, vx, scale=1000.0 * scale, **kw)
    vis = ~np.isneginf(l_ref)
    b_abs = np.zeros_like(mean_abs)
    b_abs[vis] = mean_abs[vis] * np.exp(l0[vis])[:, None]
    pmax = np.zeros_like(l_ref)
    pmax[vis] = np.minimum(1.0, np.exp(l_big[vis] / 1000.0 - l_ref[vis]))
    return 2.0 ** -4 * a_abs + 2.0 ** -10 * pmax[:, None] * b_abs + 2.0 ** -8 * np.abs(o_ref) + 1e-6
