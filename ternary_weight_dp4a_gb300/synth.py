"""Seeded synthetic inputs for the ternary FFN decode path.

This module only draws random inputs.  It holds none of the method's arithmetic
(no packing, rotation, quantisation or GEMV); the library and the oracle both
take its outputs as given.

Recipe (the shapes and distributions of the workloads the pages describe: a 27B
ternary model's dense FFN, hidden 5120, intermediate 17408):

* 2-bit weight codes: i.i.d. per weight, code 0 (value 0) with p = 0.4, code 1
  (+1) with p = 0.3, code 2 (-1) with p = 0.3.
* 1-bit weight bits: i.i.d. per weight, 1 (+1) or 0 (-1) with p = 0.5 each.
* Weight scales: one fp16 per 128-weight block per row, fp16(U[0.01, 0.05]).
* Activations: bf16(N(0, 1)); with outliers, exactly round(frac * k) positions
  per row, drawn uniformly without replacement, are multiplied by 10 before the
  bf16 rounding.

Seeds name one stream per device kind: ``device="cpu"`` draws with numpy's
PCG64 (``default_rng(seed)``), ``device="cuda"`` with torch's CUDA generator
seeded with the same number.  The two kinds give different values for the same
seed; each test states which it uses.  Within one kind, a weight matrix is one
stream (codes first, then scales) and activation row r is the stream
``seed + r``.
"""
from __future__ import annotations

import numpy as np

P_ZERO = 0.4
P_PLUS = 0.3
SCALE_LO = 0.01
SCALE_HI = 0.05
OUTLIER_GAIN = 10.0
BLOCK = 128

# seed scheme used by the tests and the benchmark
SEED_TINY_WEIGHT = 0
SEED_ACT_BASE = 1_000_000


def ffn_weight_seed(layer: int, which: int) -> int:
    """Seed of FFN layer ``layer``'s matrix ``which`` (0 gate, 1 up, 2 down)."""
    return 1000 + 3 * layer + which


def _bf16_bits_from_f32(x32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def weight(n: int, k: int, fmt: int, seed: int, device: str = "cpu"):
    """Codes [n][k] (uint8: 0/1/2 for 2-bit, 0/1 for 1-bit) and fp16 scales
    [n][k/128].  Returns numpy arrays (cpu) or torch tensors (cuda)."""
    if k % BLOCK:
        raise ValueError("k must be a multiple of 128")
    nb = k // BLOCK
    if device == "cpu":
        rng = np.random.default_rng(seed)
        codes = np.empty((n, k), dtype=np.uint8)
        chunk = max(1, (1 << 24) // max(k, 1))
        for r0 in range(0, n, chunk):
            u = rng.random((min(chunk, n - r0), k), dtype=np.float32)
            if fmt == 0:
                c = np.where(u < P_ZERO, 0, np.where(u < P_ZERO + P_PLUS, 1, 2))
            else:
                c = (u < 0.5).astype(np.uint8)
            codes[r0:r0 + c.shape[0]] = c
        scales = rng.uniform(SCALE_LO, SCALE_HI, size=(n, nb)).astype(np.float16)
        return codes, scales
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    codes = torch.empty((n, k), dtype=torch.uint8, device=device)
    chunk = max(1, (1 << 26) // max(k, 1))
    for r0 in range(0, n, chunk):
        rows = min(chunk, n - r0)
        u = torch.rand((rows, k), generator=g, device=device, dtype=torch.float32)
        if fmt == 0:
            c = torch.where(u < P_ZERO, 0, torch.where(u < P_ZERO + P_PLUS, 1, 2))
        else:
            c = (u < 0.5)
        codes[r0:r0 + rows] = c.to(torch.uint8)
        del u, c
    scales = (torch.rand((n, nb), generator=g, device=device, dtype=torch.float32)
              * (SCALE_HI - SCALE_LO) + SCALE_LO).to(torch.float16)
    return codes, scales


def activation(m: int, k: int, seed: int, outlier_frac: float = 0.0,
               device: str = "cpu"):
    """bf16 activations as uint16 bits [m][k] (numpy) or a torch bf16 tensor
    (cuda).  Row r draws from stream ``seed + r``."""
    n_out = int(round(outlier_frac * k))
    if device == "cpu":
        rows = []
        for r in range(m):
            rng = np.random.default_rng(seed + r)
            v = rng.standard_normal(k).astype(np.float32)
            if n_out:
                idx = rng.choice(k, size=n_out, replace=False)
                v[idx] *= np.float32(OUTLIER_GAIN)
            rows.append(v)
        x32 = np.stack(rows) if rows else np.zeros((0, k), np.float32)
        return _bf16_bits_from_f32(x32)
    import torch
    out = torch.empty((m, k), dtype=torch.bfloat16, device=device)
    for r in range(m):
        g = torch.Generator(device=device)
        g.manual_seed(seed + r)
        v = torch.randn(k, generator=g, device=device, dtype=torch.float32)
        if n_out:
            idx = torch.randperm(k, generator=g, device=device)[:n_out]
            v[idx] *= OUTLIER_GAIN
        out[r] = v.to(torch.bfloat16)
    return out

