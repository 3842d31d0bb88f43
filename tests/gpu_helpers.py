"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
on seeded host inputs, and compare against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from transformer_head_scaled_fwd_gb300 import binding

# bf16 I/O with fp32 accumulation: |g - o| <= 1.5e-2 + 2e-2 |o| per element;
# fp32 storage and arithmetic: |g - o| <= 1e-4 + 1e-4 |o|; p_attn row sums within 1e-3 of 1.
TOL = {"bf16": (1.5e-2, 2e-2), "f32": (1e-4, 1e-4)}
ROWSUM_TOL = 1e-3


def to_dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dtype).contiguous()


def run_gpu(inp, *, causal=False, valid_lens=None, dense=None, want_p_attn=False, stages=False):
    """Run mha_forward on inp (workloads.Inputs). Returns (out fp64 numpy, p_attn or None)."""
    wl = inp.wl
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    q = to_dev(inp.query, dt)
    k = q if inp.key is inp.query else to_dev(inp.key, dt)
    v = k if inp.value is inp.key else to_dev(inp.value, dt)
    W = {n: to_dev(a, dt) for n, a in inp.weights.items()}
    B, Lq, d = inp.query.shape
    Lk = inp.key.shape[1]
    h = wl.h
    dtc = binding.MHA_BF16 if wl.dtype == "bf16" else binding.MHA_F32
    ws = torch.empty(binding.workspace_size(dtc, B, Lq, Lk, d, h), dtype=torch.uint8, device="cuda")
    out = torch.empty(B, Lq, d, dtype=dt, device="cuda")
    p = torch.full((B, h, Lq, Lk), float("nan"), device="cuda") if want_p_attn else None
    vl = None if valid_lens is None else torch.as_tensor(np.asarray(valid_lens), dtype=torch.int32).cuda()
    dm = None if dense is None else torch.as_tensor(np.asarray(dense), dtype=torch.uint8).cuda()
    mask = binding.make_mask(causal, vl, dm)
    if stages:
        binding.mha_qkv_projection(q, k, v, W["w_q"], W["b_q"], W["w_k"], W["b_k"], W["w_v"], W["b_v"], h,
                                   workspace=ws)
        binding.mha_attention_core(dtc, B, Lq, Lk, d, h, workspace=ws, mask=mask, p_attn=p)
        binding.mha_output_projection(W["w_o"], W["b_o"], B, Lq, Lk, h, out=out, workspace=ws)
    else:
        binding.mha_forward(q, k, v, W["w_q"], W["b_q"], W["w_k"], W["b_k"], W["w_v"], W["b_v"],
                            W["w_o"], W["b_o"], h, out=out, workspace=ws, mask=mask, p_attn=p)
    torch.cuda.synchronize()
    assert binding.mha_check_device_status(reset=True) == 0, "a pipeline wait gave up"
    o = out.double().cpu().numpy()
    return o, (None if p is None else p.double().cpu().numpy())


def run_oracle(inp, *, causal=False, valid_lens=None, dense=None, rows=None, want_p_attn=False):
    w = inp.weights
    return oracle.mha_forward(inp.query, inp.key, inp.value, w["w_q"], w["b_q"], w["w_k"], w["b_k"],
                              w["w_v"], w["b_v"], w["w_o"], w["b_o"], inp.wl.h, causal=causal,
                              valid_lens=valid_lens, dense=dense, rows=rows, want_p_attn=want_p_attn)


def assert_close(got, ref, kind, what="out"):
    atol, rtol = TOL[kind]
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} elements outside |g-o| <= {atol} + {rtol}|o|; "
            f"worst at {idx}: got {got[idx]!r} oracle {ref[idx]!r}; max abs err {err.max():.3e}")
    return float(err.max())
