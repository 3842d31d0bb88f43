"""Seeded synthetic inputs for the multi-head attention forward pass.

This module only draws numbers: it holds none of the method's arithmetic. The
same host arrays feed the fp64 oracle (widened) and the GPU path (copied), so
both see identical values.

Workload shapes follow the pages' model sizes ("003-Transformer" tutorial,
make_model: d_model=512, h=8, so d_k=64; the Transformer base sizes of the
"Attention Is All You Need" model) and the call forms the pages show:
self-attention self_attn(x, x, x, mask), decoder masked self-attention with the
subsequent mask, and source attention src_attn(x, m, m, src_mask) with the
encoder memory as both key and value ("The Annotated Transformer",
DecoderLayer.forward). Weights are Xavier-uniform, as in the d2l training recipe
(d2l Transformer chapter summary), biases zero; activations are N(0, 1) so that
the scaled scores have unit variance (the sqrt(d_k) rationale of "From RNN to
Attention", part 3). There is no dataset: these synthetic shapes stand in for
the pages' translation data.

Generation order per config (torch CPU generator, seed 20261202 + index):
query, [memory], W_q, b_q, W_k, b_k, W_v, b_v, W_o, b_o, valid_lens.
Values are drawn in fp32; for bf16 workloads they are rounded to bf16 and kept
as fp32 arrays holding bf16-exact values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    dtype: str            # "f32" or "bf16": storage type of inputs, weights and outputs
    B: int
    Lq: int
    Lk: int
    d_model: int
    h: int
    causal: bool
    self_attn: bool       # query, key and value are one tensor
    valid_fixed: tuple | None = None       # fixed key valid lengths
    valid_range: tuple | None = None       # (lo, hi) inclusive uniform key valid lengths
    note: str = ""

    @property
    def d_k(self) -> int:
        return self.d_model // self.h


WORKLOADS = {
    "tiny": Workload("tiny", 0, "f32", 2, 10, 10, 512, 8, False, True, valid_fixed=(10, 7),
                     note="tiny fp32 self-attention, key padding mask, valid lens [10, 7]"),
    "enc": Workload("enc", 1, "bf16", 32, 128, 128, 512, 8, False, True, valid_range=(64, 128),
                    note="encoder self-attention, key padding valid lens U{64..128}"),
    "dec": Workload("dec", 2, "bf16", 32, 256, 256, 512, 8, True, True, valid_range=(128, 256),
                    note="decoder masked self-attention, causal AND key padding U{128..256}"),
    "xattn": Workload("xattn", 3, "bf16", 16, 256, 320, 1024, 16, False, False,
                      valid_range=(160, 320),
                      note="encoder-decoder attention, memory as key and value, padding U{160..320}"),
    "long": Workload("long", 4, "bf16", 4, 8192, 8192, 1024, 16, True, True,
                     note="long-sequence causal self-attention, causal mask only"),
    # wider heads (d_k = 128): the same model width with h = 8
    "long_d128": Workload("long_d128", 5, "bf16", 4, 8192, 8192, 1024, 8, True, True,
                          note="long-sequence causal self-attention with d_k = 128"),
}


@dataclass
class Inputs:
    """Host arrays (numpy fp32, bf16-exact for bf16 workloads)."""
    wl: Workload
    query: np.ndarray
    key: np.ndarray
    value: np.ndarray
    weights: dict = field(default_factory=dict)   # w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o
    valid_lens: np.ndarray | None = None
    dense: np.ndarray | None = None


def round_bf16(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16).to(torch.float32)


def xavier_uniform(g: torch.Generator, fan_out: int, fan_in: int) -> torch.Tensor:
    bound = math.sqrt(6.0 / (fan_in + fan_out))
    return (torch.rand((fan_out, fan_in), generator=g, dtype=torch.float32) * 2.0 - 1.0) * bound


def make_inputs(wl: Workload, *, bias_scale: float = 0.0, seed_offset: int = 0,
                B: int | None = None) -> Inputs:
    """Draw the seeded inputs of workload ``wl``.

    bias_scale > 0 draws biases from U(-bias_scale, bias_scale) instead of zeros
    (exercises the bias epilogue). ``B`` overrides the batch size (used to shard
    a batch across ranks: rank r draws with seed_offset r).
    """
    g = torch.Generator().manual_seed(SEED_BASE + wl.index + 1000 * seed_offset)
    Bn = wl.B if B is None else B
    d = wl.d_model
    q = torch.randn((Bn, wl.Lq, d), generator=g, dtype=torch.float32)
    if wl.self_attn:
        k = v = q
    else:
        k = torch.randn((Bn, wl.Lk, d), generator=g, dtype=torch.float32)
        v = k
    w = {}
    for name in ("q", "k", "v", "o"):
        w["w_" + name] = xavier_uniform(g, d, d)
        if bias_scale > 0:
            w["b_" + name] = (torch.rand((d,), generator=g) * 2.0 - 1.0) * bias_scale
        else:
            w["b_" + name] = torch.zeros((d,), dtype=torch.float32)
    vl = None
    if wl.valid_fixed is not None:
        vl = torch.tensor(list(wl.valid_fixed)[:Bn] + [wl.Lk] * max(0, Bn - len(wl.valid_fixed)),
                          dtype=torch.int32)
    elif wl.valid_range is not None:
        lo, hi = wl.valid_range
        vl = torch.randint(lo, hi + 1, (Bn,), generator=g, dtype=torch.int32)
    if wl.dtype == "bf16":
        q = round_bf16(q)
        k = q if wl.self_attn else round_bf16(k)
        v = k
        w = {n: round_bf16(t) for n, t in w.items()}
    to_np = lambda t: t.contiguous().numpy()
    qn = to_np(q)
    kn = qn if k is q else to_np(k)           # aliasing is kept: self-attention passes one tensor
    return Inputs(wl, qn, kn, kn if v is k else to_np(v),
                  {n: to_np(t) for n, t in w.items()},
                  None if vl is None else vl.numpy())


def random_case(seed: int, B: int, Lq: int, Lk: int, d_model: int, h: int, *,
                dtype: str = "bf16", self_attn: bool = False, kv_alias: bool = True,
                bias_scale: float = 0.1, valid_lens=None, x_scale: float = 1.0) -> Inputs:
    """A seeded case of arbitrary shape (ragged tails, tiny sizes, edge cases)."""
    wl = Workload(f"case{seed}", 0, dtype, B, Lq, Lk, d_model, h, False, self_attn)
    g = torch.Generator().manual_seed(SEED_BASE + 7919 * seed + 17)
    q = torch.randn((B, Lq, d_model), generator=g) * x_scale
    if self_attn:
        assert Lq == Lk
        k = v = q
    else:
        k = torch.randn((B, Lk, d_model), generator=g) * x_scale
        v = k if kv_alias else torch.randn((B, Lk, d_model), generator=g) * x_scale
    w = {}
    for name in ("q", "k", "v", "o"):
        w["w_" + name] = xavier_uniform(g, d_model, d_model)
        w["b_" + name] = (torch.rand((d_model,), generator=g) * 2.0 - 1.0) * bias_scale
    if dtype == "bf16":
        q = round_bf16(q)
        k = q if self_attn else round_bf16(k)
        v = k if (self_attn or kv_alias) else round_bf16(v)
        w = {n: round_bf16(t) for n, t in w.items()}
    vl = None if valid_lens is None else np.asarray(valid_lens, dtype=np.int32)
    qn = q.contiguous().numpy()
    kn = qn if k is q else k.contiguous().numpy()
    vn = kn if v is k else v.contiguous().numpy()
    return Inputs(wl, qn, kn, vn,
                  {n: t.contiguous().numpy() for n, t in w.items()}, vl)


def sample_rows(L: int, n: int, seed: int) -> np.ndarray:
    """n distinct query positions in [0, L), always including 0 and L-1, sorted."""
    rng = np.random.default_rng(SEED_BASE + 31 * seed)
    n = min(n, L)
    inner = rng.choice(np.arange(1, L - 1), size=max(0, n - 2), replace=False) if L > 2 else []
    rows = sorted(set([0, L - 1]) | set(int(x) for x in inner))
    return np.asarray(rows, dtype=np.int32)


@dataclass
class FFNInputs:
    x: np.ndarray
    w_1: np.ndarray
    b_1: np.ndarray
    w_2: np.ndarray
    b_2: np.ndarray
    dtype: str


FFN_WORKLOADS = {
    # the pages' base sizes: d_model 512, d_ff 2048 ("003-Transformer", make_model)
    "ffn_base": dict(B=32, L=256, d_model=512, d_ff=2048),
    # the long workload's width with the same 4x expansion
    "ffn_long": dict(B=4, L=8192, d_model=1024, d_ff=4096),
}


def make_ffn_inputs(B: int, L: int, d_model: int, d_ff: int, *, seed: int = 0, dtype: str = "bf16",
                    bias_scale: float = 0.1) -> FFNInputs:
    """x ~ N(0, 1); W_1 [d_ff, d_model], W_2 [d_model, d_ff] Xavier-uniform; biases U(-s, s)."""
    g = torch.Generator().manual_seed(SEED_BASE + 104729 * (seed + 1))
    x = torch.randn((B, L, d_model), generator=g)
    w1 = xavier_uniform(g, d_ff, d_model)
    b1 = (torch.rand((d_ff,), generator=g) * 2 - 1) * bias_scale
    w2 = xavier_uniform(g, d_model, d_ff)
    b2 = (torch.rand((d_model,), generator=g) * 2 - 1) * bias_scale
    ts = [x, w1, b1, w2, b2]
    if dtype == "bf16":
        ts = [round_bf16(t) for t in ts]
    return FFNInputs(*[t.contiguous().numpy() for t in ts], dtype)


def make_ln_params(d_model: int, *, seed: int = 0, dtype: str = "bf16"):
    """LayerNorm gain U(0.5, 1.5) and bias U(-0.1, 0.1), seeded (numpy fp32, bf16-exact for bf16)."""
    g = torch.Generator().manual_seed(SEED_BASE + 15485863 * (seed + 1))
    a = torch.rand((d_model,), generator=g) + 0.5
    b = (torch.rand((d_model,), generator=g) * 2 - 1) * 0.1
    if dtype == "bf16":
        a, b = round_bf16(a), round_bf16(b)
    return a.contiguous().numpy(), b.contiguous().numpy()
