"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws random numbers, so the
CUDA path and the CPU oracle can be fed identical values without sharing code.

Recipe: a CPU ``torch.Generator`` seeded with ``seed`` draws fp32 N(0, 1) values
in the fixed order Q, K, V, dO and then (learnable sink only) the per-head
softmax offset.  Q/K/V/dO are rounded to bf16 (round-to-nearest-even by
``Tensor.to``); the offset stays fp32.  All sequences are full length (no
padding), as in the codelab's and the TransformerEngine example's random
BSHD inputs.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Shape:
    B: int
    S_q: int
    S_kv: int
    H_q: int
    H_kv: int
    d_qk: int
    d_v: int


def make_inputs(shape: Shape, seed: int, *, with_dout: bool = True,
                learnable_offset: bool = False, dtype=torch.bfloat16):
    """Return a dict with q, k, v[, dout][, offset] on the CPU.

    q [B,S_q,H_q,d_qk], k [B,S_kv,H_kv,d_qk], v [B,S_kv,H_kv,d_v], dout like O
    [B,S_q,H_q,d_v], all ``dtype`` (bf16 by default); offset fp32 [H_q].
    """
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    s = shape
    out = {}
    out["q"] = torch.randn((s.B, s.S_q, s.H_q, s.d_qk), generator=g, dtype=torch.float32).to(dtype)
    out["k"] = torch.randn((s.B, s.S_kv, s.H_kv, s.d_qk), generator=g, dtype=torch.float32).to(dtype)
    out["v"] = torch.randn((s.B, s.S_kv, s.H_kv, s.d_v), generator=g, dtype=torch.float32).to(dtype)
    if with_dout:
        out["dout"] = torch.randn((s.B, s.S_q, s.H_q, s.d_v), generator=g, dtype=torch.float32).to(dtype)
    if learnable_offset:
        out["offset"] = torch.randn((s.H_q,), generator=g, dtype=torch.float32)
    return out


def make_bias(shape, seed: int, dtype=torch.bfloat16):
    """An additive attention bias of `shape` ([Bb, Hb, S_q, S_kv]): fp32 N(0, 1) from
    its own CPU generator (seeded `seed`), rounded to bf16."""
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(dtype)
