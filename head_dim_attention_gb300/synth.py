"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic.  Every tensor is drawn on the CPU in float32 from one
``torch.Generator`` seeded with ``seed``, in the fixed order q, k, v, bias, dO,
then cast to the requested dtype, so the same call gives bit-identical inputs
on every host.  Q/K/V/dO are i.i.d. N(0, 1); the bias is an fp32 N(0, 1)
key-position row of shape [1, 1, 1, Nkv] (or [1, 1, Nq, Nkv] when
``bias="query"``).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    bias: torch.Tensor | None
    do: torch.Tensor | None


def make_inputs(B: int, Hq: int, Hkv: int, Nq: int, Nkv: int, D: int, dtype=torch.bfloat16,
                bias: bool | str = False, grad: bool = False, seed: int = 0) -> Inputs:
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(B, Hq, Nq, D, generator=g, dtype=torch.float32).to(dtype)
    k = torch.randn(B, Hkv, Nkv, D, generator=g, dtype=torch.float32).to(dtype)
    v = torch.randn(B, Hkv, Nkv, D, generator=g, dtype=torch.float32).to(dtype)
    b = None
    if bias:
        shape = (1, 1, Nq, Nkv) if bias == "query" else (1, 1, 1, Nkv)
        b = torch.randn(*shape, generator=g, dtype=torch.float32)
    do = torch.randn(B, Hq, Nq, D, generator=g, dtype=torch.float32).to(dtype) if grad else None
    return Inputs(q, k, v, b, do)
