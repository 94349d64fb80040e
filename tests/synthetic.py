"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

Holds no arithmetic of the method: only random draws, dtype conversion and
layout.  Everything is seeded through ``torch.Generator`` so the CUDA path and
the oracle always see identical inputs.

Distributions (standard deviations):
  router  x ~ N(0,1), W[N,K] ~ N(0, 1/sqrt(K)) (= 1/64 at K=4096), b ~ N(0, 0.01)
  MoE     x, W13, W2 ~ N(0, 0.02) in bf16; MoE router W ~ N(0, 0.02) fp32
  unit    x ~ N(0,1), W13 ~ N(0, 1/sqrt(H)), W2 ~ N(0, 1/sqrt(I))
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


def gen(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std, seed, dtype=torch.float32, device="cpu"):
    t = torch.randn(*shape, generator=gen(seed, device), device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(dtype)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 tensor (as numpy, on the host)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16)


# ----------------------------------------------------------------- router --
@dataclass
class RouterInputs:
    x: torch.Tensor      # [M_max, K] fp32
    w: torch.Tensor      # [N, K] fp32
    b: torch.Tensor      # [N] fp32


def router_inputs(M=4096, K=4096, N=256, seeds=(1, 2, 3)) -> RouterInputs:
    """DSv4 router shape: x ~ N(0,1), W ~ N(0, 1/sqrt(K)), b ~ N(0, 0.01)."""
    return RouterInputs(
        x=normal((M, K), 1.0, seeds[0]),
        w=normal((N, K), 1.0 / math.sqrt(K), seeds[1]),
        b=normal((N,), 0.01, seeds[2]),
    )


def router_tie_inputs(M=4096, K=4096, N=256, n_groups=16, copies=3, frac=0.3, seed=5):
    """Router inputs with exact-tie plateaus.

    ``n_groups`` source experts are each copied into ``copies`` other expert
    rows of W (and their bias entries), so every score row holds n_groups
    plateaus of width copies+1; in a seeded ``frac`` of the rows x is rounded
    to multiples of 1/8 and clamped to [-4, 4].  Returns (inputs, tie_rows).
    """
    base = router_inputs(M, K, N)
    g = gen(seed)
    perm = torch.randperm(N, generator=g)
    src = perm[:n_groups]
    dst = perm[n_groups:n_groups * (1 + copies)].view(n_groups, copies)
    w = base.w.clone()
    b = base.b.clone()
    for i in range(n_groups):
        w[dst[i]] = w[src[i]].clone()
        b[dst[i]] = b[src[i]].clone()
    rows = torch.rand(M, generator=g) < frac
    x = base.x.clone()
    x[rows] = torch.clamp(torch.round(x[rows] * 8.0) / 8.0, -4.0, 4.0)
    return RouterInputs(x=x, w=w, b=b), rows


def quantised_scores(M=4096, E=256, frac=0.3, seed=7):
    """fp32 scores ~ N(0,1); a seeded ``frac`` of rows rounded to multiples of
    1/8 so that tie plateaus straddle the top-k cut."""
    g = gen(seed)
    s = torch.randn(M, E, generator=g)
    rows = torch.rand(M, generator=g) < frac
    s[rows] = torch.round(s[rows] * 8.0) / 8.0
    return s, rows


# -------------------------------------------------------------------- MoE --
@dataclass
class MoEWeights:
    w_router: torch.Tensor   # [E, H] fp32
    w13: torch.Tensor        # [E, 2I, H] bf16 (rows [0,I) gate, [I,2I) up)
    w2: torch.Tensor         # [E, H, I] bf16
    H: int
    E: int
    I: int


QWEN_SHAPE = dict(H=2048, E=128, I=768, top_k=8)
DSV4_SHAPE = dict(H=4096, E=256, I=2048, top_k=8)


def moe_weights(H, E, I, seed=11, std=0.02, unit=False, device="cpu") -> MoEWeights:
    """MoE weights.  Default: all ~ N(0, std); unit=True: W13 ~ N(0,1/sqrt(H)),
    W2 ~ N(0, 1/sqrt(I)), router ~ N(0, 1/sqrt(H))."""
    s13 = 1.0 / math.sqrt(H) if unit else std
    s2 = 1.0 / math.sqrt(I) if unit else std
    sr = 1.0 / math.sqrt(H) if unit else std
    return MoEWeights(
        w_router=normal((E, H), sr, seed + 1, device=device),
        w13=normal((E, 2 * I, H), s13, seed + 2, torch.bfloat16, device=device),
        w2=normal((E, H, I), s2, seed + 3, torch.bfloat16, device=device),
        H=H, E=E, I=I)


def moe_tokens(M, H, seed=21, std=0.02, unit=False, device="cpu"):
    """Token activations x [M, H] bf16."""
    return normal((M, H), 1.0 if unit else std, seed, torch.bfloat16, device=device)


def random_routing(M, E, top_k, seed=31):
    """ids [M,k] int32 with distinct experts per row, wts [M,k] fp32 in (0,1)."""
    g = gen(seed)
    ids = torch.argsort(torch.rand(M, E, generator=g), dim=1)[:, :top_k].to(torch.int32)
    wts = torch.rand(M, top_k, generator=g).to(torch.float32)
    return ids.contiguous(), wts.contiguous()


def skewed_routing(M, E, top_k, hot=4, seed=33):
    """Routing where every row uses the first ``hot`` experts (load skew):
    ragged expert counts with some experts empty."""
    g = gen(seed)
    ids = torch.empty(M, top_k, dtype=torch.int32)
    for m in range(M):
        rest = torch.randperm(E - hot, generator=g)[: top_k - hot] + hot
        ids[m] = torch.cat([torch.arange(hot), rest]).to(torch.int32)[torch.randperm(top_k, generator=g)]
    wts = torch.rand(M, top_k, generator=g).to(torch.float32)
    return ids.contiguous(), wts.contiguous()


def compositions(n_comp=50, n_targets=16, max_batch=4096, seed=41, sizes=None):
    """Co-batch compositions: list of (batch, positions of the targets).

    Batch sizes come from ``sizes`` first, then uniform in [1, max_batch]; a
    batch smaller than the number of targets carries the first ``batch``
    targets.  Target positions are a seeded random subset of the batch."""
    g = gen(seed)
    out = []
    sizes = list(sizes or [])
    for c in range(n_comp):
        B = sizes[c] if c < len(sizes) else int(torch.randint(1, max_batch + 1, (1,), generator=g))
        nt = min(B, n_targets)
        pos = torch.randperm(B, generator=g)[:nt]
        out.append((B, pos))
    return out


def batch_sizes(max_m=4096):
    """1, 8 and 2^n - 1, 2^n, 2^n + 1 for 2^n in [16, max_m], plus max_m."""
    s = {1, 8}
    p = 16
    while p <= max_m:
        s.update({p - 1, p, p + 1})
        p *= 2
    return sorted(v for v in s if v <= max_m)


def unambiguous_rows(r64, k, margin=1e-4):
    """Rows of fp64 scores whose top-k selection cannot be changed by a
    perturbation smaller than `margin`: among the k+1 largest scores every
    adjacent gap is either exactly 0 (an exact tie, decided by index on both
    sides) or at least `margin`.  Used to compare selections made from
    scores computed in different precisions."""
    r = np.asarray(r64, np.float64)
    s = -np.sort(-r, axis=1)[:, : k + 1]
    gaps = s[:, :-1] - s[:, 1:]
    return np.where(np.all((gaps == 0) | (gaps >= margin), axis=1))[0]
