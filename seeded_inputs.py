"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can be fed
from it without sharing code.

Recipe (the pages publish no data; the shapes stand in for the attention
layers of the long-context training runs they describe):

* Q, K, V and dO are i.i.d. N(0, 1), drawn in fp32 by a CPU
  ``torch.Generator`` seeded with ``seed + k`` (k = 0, 1, 2, 3 for Q, K, V,
  dO), shape [B, H, S, D] in *position* (unpermuted) order, then rounded to
  the compute dtype (bf16 round-to-nearest-even) where that is not fp32.
* Sampled rows use ``seed + 4``.
"""
from __future__ import annotations

import torch

_NAMES = ("q", "k", "v", "do")


def _randn(shape, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32)


def attention_inputs(B: int, H: int, S: int, D: int, dtype: torch.dtype = torch.bfloat16,
                     seed: int = 0, with_do: bool = True) -> dict[str, torch.Tensor]:
    """Return CPU tensors q, k, v (and do) of shape [B, H, S, D] in ``dtype``."""
    out = {}
    names = _NAMES if with_do else _NAMES[:3]
    for idx, name in enumerate(names):
        x = _randn((B, H, S, D), seed + idx)
        out[name] = x if dtype == torch.float32 else x.to(dtype)
    return out


def device_inputs(B: int, H: int, S: int, D: int, dtype: torch.dtype, seed: int,
                  device: torch.device, with_do: bool = True) -> dict[str, torch.Tensor]:
    """Same distribution drawn directly on ``device`` (for timing only; the
    parity tests use the CPU draw so the oracle sees the host copy)."""
    out = {}
    names = _NAMES if with_do else _NAMES[:3]
    for idx, name in enumerate(names):
        g = torch.Generator(device=device)
        g.manual_seed(int(seed + idx))
        x = torch.randn((B, H, S, D), generator=g, device=device, dtype=torch.float32)
        out[name] = x if dtype == torch.float32 else x.to(dtype)
    return out


def sample_rows(n: int, B: int, H: int, S: int, seed: int = 0) -> torch.Tensor:
    """n (b, h, position) triples drawn uniformly with the row seed (seed + 4)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed + 4))
    b = torch.randint(0, B, (n,), generator=g)
    h = torch.randint(0, H, (n,), generator=g)
    p = torch.randint(0, S, (n,), generator=g)
    return torch.stack([b, h, p], dim=1)


def sample_tail_keys(n: int, S: int, window: int, seed: int = 0) -> torch.Tensor:
    """n distinct key positions from the last ``window`` positions (row seed)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed + 4))
    w = min(window, S)
    perm = torch.randperm(w, generator=g)[: min(n, w)]
    return torch.sort(S - w + perm).values


def sample_keys(n: int, S: int, seed: int = 0) -> torch.Tensor:
    """n distinct key positions drawn uniformly over [0, S) (row seed), sorted."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed + 4) * 104729 + 3)
    m = min(n, S)
    if S <= 4 * m:
        pick = torch.randperm(S, generator=g)[:m]
    else:  # rejection of repeats keeps memory O(n) for long sequences
        seen = set()
        out = []
        while len(out) < m:
            for x in torch.randint(0, S, (2 * m,), generator=g).tolist():
                if x not in seen:
                    seen.add(x)
                    out.append(x)
                    if len(out) == m:
                        break
        pick = torch.as_tensor(out, dtype=torch.int64)
    return torch.sort(pick).values


def sample_head(B: int, H: int, seed: int = 0) -> tuple[int, int]:
    """One (b, h) chosen with the row seed, for per-head key-row checks."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed + 4) * 7919 + 1)
    b = int(torch.randint(0, B, (1,), generator=g))
    h = int(torch.randint(0, H, (1,), generator=g))
    return b, h
