"""Seeded synthetic inputs for the tensor-parallel MLP block.

This module only draws random tensors; it holds none of the block's
arithmetic, so both the CUDA path and the fp64 oracle can take their inputs
from it without sharing any computation.

Workloads follow the layer shapes named on the source pages:

* GPT-2-medium (355M): hidden 1024, seq 1024 -- "Megatron-LM: Tensor Model
  Parallel" (charles2530.github.io), GPT-2 Training, Table 2.
* Megatron 8.3B: hidden 3072, 72 layers, 8-way model parallel -- same page,
  Scaling Study, Table 1; weights before the residual scaled by 1/sqrt(2N)
  (same page, Training recipe table, "Initialization").
* MT-NLG 530B: hidden 20480, seq 2048, TP 8 -- "MT-NLG 530B deep dive"
  (zzszmyf.github.io), section 4.1 model configuration.

The FFN width is 4h everywhere and T = batch * seq tokens.  Every tensor is
drawn as float32 N(0, std) on the CPU and rounded to bfloat16 (round to
nearest even).  Tensor k of X, A, b1, B, b2, residual, dY (in that order)
and row chunk c of it come from a ``torch.Generator`` seeded with
(seed, k, c), so any subset of the tensors equals the same entries of the
full draw.  A tensor whose std is 0 is all zeros.
"""

from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os
from typing import Dict, Optional

import torch

# Matrices are drawn in row chunks of about this many elements, each chunk
# from its own generator, so that chunks can be drawn in parallel threads and
# the float32 temporaries stay small.  The chunking is part of the stream's
# definition: results depend only on the seed.
_CHUNK_ELEMS = 1 << 24

DRAW_ORDER = ("X", "A", "b1", "B", "b2", "residual", "dY")


@dataclasses.dataclass(frozen=True)
class Workload:
    """One MLP-block problem: T tokens, hidden h, FFN width F, t shards."""

    name: str
    T: int
    h: int
    F: int
    t: int
    std: Dict[str, float]
    seed: int

    @property
    def f(self) -> int:
        return self.F // self.t

    def flops_fwd_bwd(self) -> int:
        """Algorithmic flops of forward + backward: six GEMMs of 2*T*h*F."""
        return 12 * self.T * self.h * self.F

    def shape(self, key: str):
        T, h, F = self.T, self.h, self.F
        return {
            "X": (T, h),
            "A": (h, F),
            "b1": (F,),
            "B": (F, h),
            "b2": (h,),
            "residual": (T, h),
            "dY": (T, h),
        }[key]

    def with_shape(self, T: int, t: Optional[int] = None, name: Optional[str] = None):
        return dataclasses.replace(
            self, T=T, t=self.t if t is None else t, name=name or self.name
        )


def _std(x=1.0, a=0.02, b1=0.0, b=0.02, b2=0.0, res=1.0, dy=1.0):
    return {"X": x, "A": a, "b1": b1, "B": b, "b2": b2, "residual": res, "dY": dy}


# The five workload families.  The seed of family k is 1000 + k.
TINY = Workload("tiny", 128, 256, 1024, 2, _std(b1=0.01, b2=0.01), 1000)
GPT2_MEDIUM = Workload("gpt2-medium", 8192, 1024, 4096, 2, _std(), 1001)
MEGATRON_8_3B = Workload(
    "megatron-8.3b", 8192, 3072, 12288, 8, _std(b=0.02 / math.sqrt(2 * 72)), 1002
)
MTNLG_530B = Workload("mt-nlg-530b", 2048, 20480, 81920, 8, _std(a=0.006, b=0.006), 1003)
SWEEP = Workload("sweep-h4096", 2048, 4096, 16384, 8, _std(), 1004)

SWEEP_TOKENS = (512, 1024, 2048, 4096, 16384)
SWEEP_SHARDS = (1, 2, 4, 8)

WORKLOADS = {w.name: w for w in (TINY, GPT2_MEDIUM, MEGATRON_8_3B, MTNLG_530B, SWEEP)}


def custom(T: int, h: int, F: int, t: int, seed: int, std=None, name="custom") -> Workload:
    """A workload of arbitrary shape with the tiny family's distributions."""
    return Workload(name, T, h, F, t, dict(std or TINY.std), seed)


def _gen(seed: int, k: int, c: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed * 1_000_003 + k * 10_007 + c) & 0x7FFFFFFFFFFFFFFF)
    return g


def _draw(seed: int, k: int, shape, std: float) -> torch.Tensor:
    if std == 0.0:
        return torch.zeros(shape, dtype=torch.bfloat16)
    if len(shape) == 1 or math.prod(shape) <= _CHUNK_ELEMS:
        x = torch.randn(shape, generator=_gen(seed, k, 0), dtype=torch.float32)
        return (x * std).to(torch.bfloat16)
    rows, cols = shape
    out = torch.empty(shape, dtype=torch.bfloat16)
    step = max(1, _CHUNK_ELEMS // cols)

    def chunk(c):
        r0 = c * step
        r1 = min(rows, r0 + step)
        x = torch.randn((r1 - r0, cols), generator=_gen(seed, k, c), dtype=torch.float32)
        out[r0:r1] = (x * std).to(torch.bfloat16)

    n = (rows + step - 1) // step
    with cf.ThreadPoolExecutor(max_workers=min(n, os.cpu_count() or 1)) as ex:
        list(ex.map(chunk, range(n)))
    return out


def make_inputs(w: Workload, keys=DRAW_ORDER) -> Dict[str, torch.Tensor]:
    """Draw the workload's bf16 tensors on the CPU (contiguous, row-major)."""
    return {key: _draw(w.seed, DRAW_ORDER.index(key), w.shape(key), w.std[key]).contiguous()
            for key in DRAW_ORDER if key in keys}


# ------------------------------------------------------- attention block

ATTN_DRAW_ORDER = ("X", "Wqkv", "bqkv", "Wo", "bo", "residual", "dY")
_ATTN_KEY_BASE = 16  # generator key indices of the attention tensors (after the MLP's)


@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """One head-parallel self-attention block: nb sequences of s tokens,
    hidden h, nh heads of d = h / nh, t shards of nh / t heads."""

    name: str
    nb: int
    s: int
    h: int
    nh: int
    t: int
    std: Dict[str, float]
    seed: int

    @property
    def T(self) -> int:
        return self.nb * self.s

    @property
    def d(self) -> int:
        return self.h // self.nh

    def flops_fwd_bwd(self) -> int:
        """Algorithmic flops: the Q/K/V and output projections (2 T h 3h and
        2 T h h forward, twice that backward) and the six products of causal
        attention (S = Q K^T, O = P V; dP, dV, dQ, dK), 2 d flops per visible
        (query, key) pair per head each."""
        pairs = self.nb * self.s * (self.s + 1) // 2
        proj = 3 * (2 * self.T * self.h * 3 * self.h + 2 * self.T * self.h * self.h)
        return proj + 6 * 2 * pairs * self.h

    def shape(self, key: str):
        T, h = self.T, self.h
        return {
            "X": (T, h),
            "Wqkv": (h, 3 * h),
            "bqkv": (3 * h,),
            "Wo": (h, h),
            "bo": (h,),
            "residual": (T, h),
            "dY": (T, h),
        }[key]


def _attn_std(x=1.0, w=0.02, bqkv=0.0, wo=0.02, bo=0.0, res=1.0, dy=1.0):
    return {"X": x, "Wqkv": w, "bqkv": bqkv, "Wo": wo, "bo": bo, "residual": res, "dY": dy}


# Attention shapes of the pages' GPT-2 models ("Megatron-LM: Tensor Model
# Parallel", Table 2: 355M with 16 heads of 64, 2.5B with 20 of 96, 8.3B with
# 24 of 128; sequence length 1024), batch 8 as in the MLP workloads.  The
# output projection sits before the residual, so the 8.3B model scales it by
# 1/sqrt(2 * 72) like B.  The tiny case matches the tiny MLP block's tokens.
ATTN_TINY = AttnWorkload("attn-tiny", 2, 64, 256, 4, 2, _attn_std(bqkv=0.01, bo=0.01), 1100)
ATTN_GPT2_355M = AttnWorkload("attn-gpt2-355m", 8, 1024, 1024, 16, 2, _attn_std(), 1101)
ATTN_GPT2_2_5B = AttnWorkload("attn-gpt2-2.5b", 8, 1024, 1920, 20, 2,
                              _attn_std(wo=0.02 / math.sqrt(2 * 54)), 1102)
ATTN_GPT2_8_3B = AttnWorkload("attn-gpt2-8.3b", 8, 1024, 3072, 24, 8,
                              _attn_std(wo=0.02 / math.sqrt(2 * 72)), 1103)

# MT-NLG 530B's attention: 128 heads of 160 over h = 20480, sequence 2048,
# 8-way tensor parallel ("MT-NLG 530B deep dive", section 4.1), one sequence
# as in the MLP workload, weights N(0, 0.006) as the MLP's.
ATTN_MTNLG_530B = AttnWorkload("attn-mt-nlg-530b", 1, 2048, 20480, 128, 8,
                               _attn_std(w=0.006, wo=0.006), 1104)

ATTN_WORKLOADS = {w.name: w for w in (ATTN_TINY, ATTN_GPT2_355M, ATTN_GPT2_2_5B, ATTN_GPT2_8_3B,
                                      ATTN_MTNLG_530B)}


def attn_custom(nb: int, s: int, h: int, nh: int, t: int, seed: int, std=None,
                name="attn-custom") -> AttnWorkload:
    """An attention block of arbitrary shape with the tiny case's distributions."""
    return AttnWorkload(name, nb, s, h, nh, t, dict(std or ATTN_TINY.std), seed)


def make_attn_inputs(w: AttnWorkload, keys=ATTN_DRAW_ORDER) -> Dict[str, torch.Tensor]:
    """Draw the attention block's bf16 tensors on the CPU (contiguous)."""
    return {key: _draw(w.seed, _ATTN_KEY_BASE + ATTN_DRAW_ORDER.index(key), w.shape(key),
                       w.std[key]).contiguous()
            for key in ATTN_DRAW_ORDER if key in keys}


def sample_indices(n: int, k: int, seed: int) -> torch.Tensor:
    """k distinct sorted indices in [0, n) (always includes n-1, the tail)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    k = min(k, n)
    idx = torch.randperm(n, generator=gen)[:k]
    if k and (n - 1) not in idx.tolist():
        idx[-1] = n - 1
    return torch.sort(idx).values.to(torch.int64)

