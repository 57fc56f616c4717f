"""Seeded synthetic inputs for the fused cascaded-reduction kernels.

This module is shared by the CUDA path (bench, GPU tests) and the CPU oracle;
it imports neither.  It holds random draws, dtype casts and the workload
shapes only: no step of the cascades themselves (no max, no exp, no softmax,
no top-k, no absmax, no quantisation, no GEMM).  Every tensor is a CPU
tensor; callers move it where they need it.

Recipes (one per workload; shapes are those of the five workloads the kernels
are built for):

* attention: Q, K, V ~ N(0, 1) drawn in fp32 from a seeded torch CPU
  generator, then cast to the kernel dtype (round-to-nearest-even for bf16).
* variable-length prefill: per-sequence lengths drawn uniformly from a range
  with a seeded generator; Q, K, V ~ N(0, 1) packed token-major
  [total, H, d] (no padding), with the cumulative lengths as int32.
* latent-KV decode: the query and the latent cache ~ N(0, 1), cast to bf16.
* MoE gate: x and W_gate hold integers drawn uniformly from {-2, ..., 2}, cast
  to bf16 (exact).  W_gate is stored expert-major, [E][D] (the layout of a
  linear layer's weight), so that both GEMM operands are contiguous along D.
* FP8 GEMM: X ~ N(0, 1) with an i.i.d. Bernoulli(0.01) outlier mask whose
  entries are multiplied by 20, cast to bf16.  W ~ N(0, 1) cast to bf16,
  stored [N][K] (each output column's K weights contiguous).  The fused path
  takes W pre-quantised (E4M3 codes with one fp32 scale per output column);
  each side makes that from W with its own per-row absmax quantiser (the
  library's rf_absmax_quant_fp8, the oracle's row_scale and quantise), and
  the tests check that the two agree bit for bit.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal(g: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32)


def _cast(t: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return t.contiguous()
    if dtype == "bf16":
        return t.to(torch.bfloat16).contiguous()
    raise ValueError(f"unknown dtype {dtype!r}")


# ---------------------------------------------------------------- workloads


@dataclass(frozen=True)
class AttnShape:
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    d: int
    dtype: str  # "f32" or "bf16"
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclass(frozen=True)
class MoEShape:
    T: int
    D: int
    E: int
    k: int
    seed: int


@dataclass(frozen=True)
class FP8Shape:
    M: int
    N: int
    K: int
    seed: int
    outlier_p: float = 0.01
    outlier_mult: float = 20.0


# The five named workloads.  Prefill attention has Lq queries per head; decode
# has one query token per (batch, query head), stored as Lq = 1.
TINY_ATTN = AttnShape(B=1, Hq=1, Hkv=1, Lq=64, Lk=256, d=64, dtype="f32", seed=0)
BERT_PREFILL = AttnShape(B=8, Hq=16, Hkv=16, Lq=512, Lk=512, d=64, dtype="bf16", seed=1)
DECODE_2K = AttnShape(B=32, Hq=32, Hkv=8, Lq=1, Lk=2048, d=128, dtype="bf16", seed=2)
DECODE_32K = AttnShape(B=32, Hq=32, Hkv=8, Lq=1, Lk=32768, d=128, dtype="bf16", seed=3)
MOE_GATE = MoEShape(T=8192, D=4096, E=64, k=2, seed=4)
FP8_GEMM = FP8Shape(M=4096, N=4096, K=4096, seed=5)


# ---------------------------------------------------------------- generators


def attention_inputs(shape: AttnShape):
    """Q [B,Hq,Lq,d], K and V [B,Hkv,Lk,d], all ~ N(0,1) in shape.dtype."""
    g = _gen(shape.seed)
    q = _cast(_normal(g, (shape.B, shape.Hq, shape.Lq, shape.d)), shape.dtype)
    k = _cast(_normal(g, (shape.B, shape.Hkv, shape.Lk, shape.d)), shape.dtype)
    v = _cast(_normal(g, (shape.B, shape.Hkv, shape.Lk, shape.d)), shape.dtype)
    return q, k, v


def decode_inputs(shape: AttnShape):
    """Decode layout: Q [B,Hq,d] (one query token), K and V [B,Hkv,Lk,d]."""
    assert shape.Lq == 1
    q, k, v = attention_inputs(shape)
    return q.reshape(shape.B, shape.Hq, shape.d).contiguous(), k, v


@dataclass(frozen=True)
class VarlenShape:
    """A batch of B sequences (query length = key length per sequence) with
    lengths drawn uniformly from [len_lo, len_hi], or given in ``lens``."""
    B: int
    H: int
    d: int
    len_lo: int
    len_hi: int
    dtype: str
    seed: int
    lens: tuple = ()

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# Short sequences (the same number of query rows per head as the BERT-style
# workload) for comparing the incremental and two-pass evaluation orders.
SHORT_PREFILL_256 = AttnShape(B=16, Hq=16, Hkv=16, Lq=256, Lk=256, d=64, dtype="bf16", seed=7)
SHORT_PREFILL_128 = AttnShape(B=32, Hq=16, Hkv=16, Lq=128, Lk=128, d=64, dtype="bf16", seed=8)

# A packed batch of BERT-style sequences of mixed length (no padding).
PREFILL_VARLEN = VarlenShape(B=16, H=16, d=64, len_lo=64, len_hi=1024, dtype="bf16", seed=6)


def varlen_inputs(shape: VarlenShape):
    """q, k, v [total, H, d] and cu_seqlens int32 [B + 1] (queries and keys
    share the lengths)."""
    g = _gen(shape.seed)
    if shape.lens:
        lens = torch.tensor(shape.lens, dtype=torch.int64)
    else:
        lens = torch.randint(shape.len_lo, shape.len_hi + 1, (shape.B,), generator=g)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
    total = int(cu[-1])
    q = _cast(_normal(g, (total, shape.H, shape.d)), shape.dtype)
    k = _cast(_normal(g, (total, shape.H, shape.d)), shape.dtype)
    v = _cast(_normal(g, (total, shape.H, shape.d)), shape.dtype)
    return q, k, v, cu


@dataclass(frozen=True)
class MLAShape:
    """Latent-KV (multi-latent attention) decode: B sequences of Lk cached
    latent rows of d_qk dims (d_v latent dims, which also serve as the
    values, then d_qk - d_v positional dims), Hq query heads, one query token.
    Defaults: the published DeepSeek-V3 attention (128 heads, latent rank
    512, positional width 64) with the softmax scale of its un-absorbed
    192-wide query-key heads."""
    B: int
    Hq: int
    Lk: int
    seed: int
    d_qk: int = 576
    d_v: int = 512
    scale: float = 1.0 / math.sqrt(192.0)


MLA_DECODE = MLAShape(B=64, Hq=128, Lk=4096, seed=9)


def mla_inputs(shape: MLAShape):
    """q [B, Hq, d_qk] and the latent cache ckv [B, Lk, d_qk], both ~ N(0, 1)
    in bf16."""
    g = _gen(shape.seed)
    q = _cast(_normal(g, (shape.B, shape.Hq, shape.d_qk)), "bf16")
    ckv = _cast(_normal(g, (shape.B, shape.Lk, shape.d_qk)), "bf16")
    return q, ckv


def moe_inputs(shape: MoEShape):
    """x [T,D] and W_gate [E,D]: integers uniform in {-2..2}, as bf16."""
    g = _gen(shape.seed)
    x = torch.randint(-2, 3, (shape.T, shape.D), generator=g, dtype=torch.int32)
    w = torch.randint(-2, 3, (shape.E, shape.D), generator=g, dtype=torch.int32)
    return x.to(torch.bfloat16).contiguous(), w.to(torch.bfloat16).contiguous()


def fp8_inputs(shape: FP8Shape):
    """X [M,K] bf16 with outliers; W [N,K] bf16 ~ N(0, 1) (to be quantised
    per row of this layout, i.e. per output column)."""
    g = _gen(shape.seed)
    x = _normal(g, (shape.M, shape.K))
    mask = torch.rand(shape.M, shape.K, generator=g) < shape.outlier_p
    x = torch.where(mask, x * shape.outlier_mult, x).to(torch.bfloat16).contiguous()
    w = _normal(g, (shape.N, shape.K)).to(torch.bfloat16).contiguous()
    return x, w
