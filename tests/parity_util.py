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
