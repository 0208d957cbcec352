"""Seeded synthetic inputs shaped like the pages' long-context workloads.

This module only draws and arranges input tensors; it holds none of the
attention arithmetic.  Both the CUDA path (tests, benchmark, smoke check) and
the oracle (which receives the very same tensors, copied to the host) take
their inputs from here.

The pages run no public benchmark or dataset; their workloads are "long
contexts, millions of tokens" with blocks of thousands of tokens ("Ring
attention, explained", step 7 and "At the extremes"; "Ring Attention: the
math", section "Communication vs compute").  The five workloads below are
synthetic stand-ins of that shape.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    key: int
    name: str
    dtype: torch.dtype
    B: int
    H: int
    N: int
    d: int
    P: int
    recipe: str  # "normal", "shift_every_4th", "offset_mean_dir"
    scale: float = 1.0
    G: int = 1  # partial segments merged by ra_merge (1 = plain forward)

    @property
    def c(self) -> int:
        return self.N // self.P

    @property
    def rows(self) -> int:
        return self.B * self.H * self.N

    @property
    def flops(self) -> float:
        """Attention work 4 B H N^2 d (two matmuls, 2 flops per multiply-add)."""
        return 4.0 * self.B * self.H * self.N * self.N * self.d

    def describe(self) -> dict:
        return {"workload": self.name, "dtype": str(self.dtype).replace("torch.", ""),
                "B": self.B, "H": self.H, "N": self.N, "d": self.d, "P": self.P, "c": self.c,
                "G": self.G, "values": self.recipe}


WORKLOADS = {
    1: Workload(1, "fp32_B1_H1_N256_d64_P4", torch.float32, 1, 1, 256, 64, 4, "normal"),
    2: Workload(2, "bf16_B1_H8_N4096_d64_P8_shifted", torch.bfloat16, 1, 8, 4096, 64, 8,
                "shift_every_4th"),
    3: Workload(3, "bf16_B1_H32_N32768_d128_P16_offset", torch.bfloat16, 1, 32, 32768, 128, 16,
                "offset_mean_dir", scale=1.0 / math.sqrt(2.0)),
    4: Workload(4, "bf16_B1_H8_N131072_d128_P32", torch.bfloat16, 1, 8, 131072, 128, 32,
                "normal"),
    5: Workload(5, "bf16_B1_H8_N1048576_d128_P64_G4", torch.bfloat16, 1, 8, 1048576, 128, 64,
                "normal", G=4),
}


def seed_of(w: Workload) -> int:
    return 20260000 + w.key


def _normal(shape, seed: int, device, scale: float) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x


def make_inputs(w: Workload, device="cuda", seed: int | None = None, shape=None):
    """Draw (q, k, v) for workload `w` ([B, H, N, d], dtype w.dtype).

    shape=(B, H, N, d) overrides the workload's sizes (same recipe), for
    small test cases.  Q, K and V each come from their own seeded stream.

    Recipes:
      normal           i.i.d. N(0, scale^2)
      shift_every_4th  K blocks j with j % 4 == 3 get + 3 * qbar, qbar the mean
                       of that (b, h)'s fp32 Q rows; so later blocks raise the
                       running max
      offset_mean_dir  K block j gets + 0.25 * j * u, u = qbar / |qbar|; the max
                       grows at every ring step
    Shifts are applied in fp32 before rounding to the workload's dtype.
    """
    B, H, N, d = shape if shape is not None else (w.B, w.H, w.N, w.d)
    base = seed_of(w) if seed is None else seed
    q = _normal((B, H, N, d), 3 * base + 0, device, w.scale)
    k = _normal((B, H, N, d), 3 * base + 1, device, w.scale)
    v = _normal((B, H, N, d), 3 * base + 2, device, w.scale)
    c = N // w.P
    if w.recipe == "shift_every_4th":
        qbar = q.mean(dim=2)  # [B, H, d]
        for j in range(3, w.P, 4):
            k[:, :, j * c:(j + 1) * c, :] += 3.0 * qbar[:, :, None, :]
    elif w.recipe == "offset_mean_dir":
        qbar = q.mean(dim=2)
        u = qbar / qbar.norm(dim=-1, keepdim=True)
        for j in range(1, w.P):
            k[:, :, j * c:(j + 1) * c, :] += 0.25 * j * u[:, :, None, :]
    elif w.recipe != "normal":
        raise ValueError(f"unknown recipe {w.recipe}")
    return q.to(w.dtype), k.to(w.dtype), v.to(w.dtype)


def sample_rows(w: Workload, count: int, seed: int = 7, shape=None) -> torch.Tensor:
    """Flat query-row indices into [B*H*N] for sampled parity checks (CPU
    int64 tensor, sorted, unique, `count` of them when there are enough rows).

    Strata, in order: the first and last row of every (b, h, query block);
    then, up to half of the remaining count, the first and last row of seeded
    128-row query tiles (every head in turn, the tiles of a head drawn without
    replacement), which are the lanes 0 and 127 of the kernel's tiles; then
    seeded uniform rows.  If the block boundaries alone exceed `count`, a
    seeded subset of them is returned."""
    B, H, N, d = shape if shape is not None else (w.B, w.H, w.N, w.d)
    c = N // w.P
    g = torch.Generator().manual_seed(seed)
    rows = []
    for bh in range(B * H):
        for i in range(w.P):
            rows.append(bh * N + i * c)
            rows.append(bh * N + i * c + c - 1)
    allr = torch.unique(torch.tensor(rows, dtype=torch.int64))
    if allr.numel() > count:
        keep = torch.randperm(allr.numel(), generator=g)[:count]
        return torch.unique(allr[keep])
    count = min(count, B * H * N)
    tiles = N // 128
    want_tiles = (count - allr.numel()) // 2
    if tiles > 0 and want_tiles > 0:
        orders = [torch.randperm(tiles, generator=g) for _ in range(B * H)]
        picked, r = [], 0
        while len(picked) < want_tiles and r < tiles:
            for bh in range(B * H):
                t = int(orders[bh][r])
                picked += [bh * N + t * 128, bh * N + t * 128 + 127]
            r += 1
        picked = torch.tensor(picked[:want_tiles], dtype=torch.int64)
        allr = torch.unique(torch.cat([allr, picked]))
    while allr.numel() < count:
        extra = torch.randint(0, B * H * N, (count - allr.numel(),), generator=g)
        allr = torch.unique(torch.cat([allr, extra]))
    return allr
