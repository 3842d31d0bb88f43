"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

CPU only. Each test would fail for a plausible mistake in the oracle: a dropped
1/sqrt(d_k), a fill added instead of replacing, a transposed weight, a wrong
head split or concat order, an off-by-one causal diagonal, a mask on the wrong
axis.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from transformer_head_scaled_fwd_gb300 import workloads as wlmod

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _weights(d, seed, bias=0.1):
    rng = np.random.default_rng(seed)
    bound = math.sqrt(6.0 / (2 * d))
    w = {}
    for n in "qkvo":
        w["w_" + n] = rng.uniform(-bound, bound, (d, d))
        w["b_" + n] = rng.uniform(-bias, bias, (d,)) if bias else np.zeros(d)
    return w


def _run(q, k, v, w, h, **kw):
    return oracle.mha_forward(q, k, v, w["w_q"], w["b_q"], w["w_k"], w["b_k"], w["w_v"], w["b_v"],
                              w["w_o"], w["b_o"], h, **kw)


# ---------------------------------------------------------------- worked example
def test_thinking_machines_worked_example():
    """Raw scores 112 / 96 at d_k = 64 -> scaled 14 / 12 -> weights 0.8808 / 0.1192."""
    g = json.load(open(os.path.join(GOLDEN, "thinking_machines.json")))
    d, h = g["d_k"], 1
    eye = np.eye(d)
    w = {"w_q": eye, "w_k": eye, "w_v": eye, "w_o": eye,
         "b_q": None, "b_k": None, "b_v": None, "b_o": None}
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1.0
    k = np.zeros((1, 2, d)); k[0, 0, 0] = g["raw_scores"][0]; k[0, 1, 0] = g["raw_scores"][1]
    v = np.zeros((1, 2, d)); v[0, 0, 0] = 1.0; v[0, 1, 1] = 1.0
    out, p = _run(q, k, v, w, h, want_p_attn=True)
    np.testing.assert_allclose(p[0, 0, 0], g["weights"], rtol=0, atol=1e-15)
    expect = np.zeros(d); expect[:2] = g["weights"]
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-15)
    # without the scale the weight on "Machines" would be ~1e-7 (the article's point)
    assert p[0, 0, 0, 1] > 1e3 * g["unscaled_weight_on_machines_max"]


# ---------------------------------------------------------------- causal convention
def test_causal_matches_printed_subsequent_mask():
    rows = [l for l in open(os.path.join(GOLDEN, "subsequent_mask_5.txt")) if not l.startswith("#")]
    printed = np.array([[int(t) for t in l.split()] for l in rows if l.strip()])
    L, d, h = 5, 8, 2
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, L, d))
    w = _weights(d, 4)
    _, p = _run(x, x, x, w, h, causal=True, want_p_attn=True)
    for hh in range(h):
        assert np.all(p[0, hh][printed == 0] == 0.0)
        assert np.all(p[0, hh][printed == 1] > 0.0)
    # row 0 sees only itself: weight exactly 1, so out_0 = W_o (W_v x_0 + b_v) + b_o
    v0 = w["w_v"] @ x[0, 0] + w["b_v"]
    out, _ = _run(x, x, x, w, h, causal=True, want_p_attn=True)
    np.testing.assert_allclose(out[0, 0], w["w_o"] @ v0 + w["b_o"], rtol=0, atol=1e-13)


# ---------------------------------------------------------------- softmax invariants
def test_rows_sum_to_one_and_masked_keys_zero():
    B, Lq, Lk, d, h = 3, 7, 9, 16, 4
    rng = np.random.default_rng(5)
    q = rng.standard_normal((B, Lq, d)); kv = rng.standard_normal((B, Lk, d))
    w = _weights(d, 6)
    vl = [9, 4, 1]
    _, p = _run(q, kv, kv, w, h, valid_lens=vl, want_p_attn=True)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-14)
    for b in range(B):
        assert np.all(p[b, :, :, vl[b]:] < 1e-30)


def test_fully_masked_row_is_uniform_mean_of_values():
    """-1e9 fill on every key makes all scores equal: uniform weights over all L_k keys."""
    B, L, d, h = 2, 6, 16, 4
    rng = np.random.default_rng(7)
    x = rng.standard_normal((B, L, d))
    w = _weights(d, 8)
    out, p = _run(x, x, x, w, h, valid_lens=[0, 3], want_p_attn=True)
    np.testing.assert_allclose(p[0], 1.0 / L, rtol=0, atol=1e-15)
    vmean = (x[0] @ w["w_v"].T + w["b_v"]).mean(0)
    expect = w["w_o"] @ vmean + w["b_o"]
    for i in range(L):
        np.testing.assert_allclose(out[0, i], expect, rtol=0, atol=1e-13)
    # fully masked via the dense mask (broadcast over queries) as well
    dense = np.zeros((B, 1, L), dtype=np.uint8); dense[1, 0, :2] = 1
    out2, p2 = _run(x, x, x, w, h, dense=dense, want_p_attn=True)
    np.testing.assert_allclose(p2[0], 1.0 / L, rtol=0, atol=1e-15)
    assert np.all(p2[1, :, :, 2:] < 1e-30)


def test_single_key_gives_weight_one():
    B, Lq, d, h = 2, 3, 8, 1
    rng = np.random.default_rng(9)
    q = rng.standard_normal((B, Lq, d)); kv = rng.standard_normal((B, 1, d))
    w = _weights(d, 10)
    out, p = _run(q, kv, kv, w, h, want_p_attn=True)
    assert np.all(p == 1.0)
    for b in range(B):
        expect = w["w_o"] @ (w["w_v"] @ kv[b, 0] + w["b_v"]) + w["b_o"]
        for i in range(Lq):
            np.testing.assert_allclose(out[b, i], expect, rtol=0, atol=1e-13)


def test_identical_query_rows_identical_outputs():
    B, L, d, h = 1, 6, 16, 2
    rng = np.random.default_rng(11)
    q = rng.standard_normal((B, L, d)); q[0, 4] = q[0, 1]
    kv = rng.standard_normal((B, 8, d))
    out = _run(q, kv, kv, _weights(d, 12), h)
    np.testing.assert_array_equal(out[0, 4], out[0, 1])


def test_masked_keys_do_not_influence_output():
    B, Lq, Lk, d, h = 2, 5, 8, 16, 4
    rng = np.random.default_rng(13)
    q = rng.standard_normal((B, Lq, d)); kv = rng.standard_normal((B, Lk, d))
    w = _weights(d, 14)
    vl = [5, 8]
    out1 = _run(q, kv, kv, w, h, valid_lens=vl)
    kv2 = kv.copy(); kv2[0, 5:] = 1e3 * rng.standard_normal((3, d))
    out2 = _run(q, kv2, kv2, w, h, valid_lens=vl)
    np.testing.assert_allclose(out1, out2, rtol=0, atol=1e-12)


def test_head_permutation_invariance():
    """Permuting whole heads in W_q/W_k/W_v (rows) and W_o (columns) leaves out unchanged."""
    B, L, d, h = 2, 5, 12, 3
    dk = d // h
    rng = np.random.default_rng(15)
    x = rng.standard_normal((B, L, d))
    w = _weights(d, 16)
    perm = [2, 0, 1]
    idx = np.concatenate([np.arange(p * dk, (p + 1) * dk) for p in perm])
    w2 = dict(w)
    for n in "qkv":
        w2["w_" + n] = w["w_" + n][idx]; w2["b_" + n] = w["b_" + n][idx]
    w2["w_o"] = w["w_o"][:, idx]
    np.testing.assert_allclose(_run(x, x, x, w, h), _run(x, x, x, w2, h), rtol=0, atol=1e-12)
    # but a split across head boundaries (mixing features of two heads) does change it
    idx_bad = np.roll(np.arange(d), 1)
    w3 = dict(w)
    for n in "qkv":
        w3["w_" + n] = w["w_" + n][idx_bad]; w3["b_" + n] = w["b_" + n][idx_bad]
    w3["w_o"] = w["w_o"][:, idx_bad]
    assert np.abs(_run(x, x, x, w, h) - _run(x, x, x, w3, h)).max() > 1e-6


# ---------------------------------------------------------------- library routine
def _torch_mha(q, k, v, w, h, key_padding=None, attn_mask=None):
    d = q.shape[-1]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).double()
    out, _ = torch.nn.functional.multi_head_attention_forward(
        t(q).transpose(0, 1), t(k).transpose(0, 1), t(v).transpose(0, 1), d, h,
        None, torch.cat([t(w["b_q"]), t(w["b_k"]), t(w["b_v"])]), None, None, False, 0.0,
        t(w["w_o"]), t(w["b_o"]), training=False, key_padding_mask=key_padding,
        need_weights=False, attn_mask=attn_mask, use_separate_proj_weight=True,
        q_proj_weight=t(w["w_q"]), k_proj_weight=t(w["w_k"]), v_proj_weight=t(w["w_v"]))
    return out.transpose(0, 1).numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_multi_head_attention(causal):
    """Rows with at least one allowed key: -1e9 fill and -inf masking agree exactly in fp64,
    so PyTorch's own MHA (separate projection weights, [out, in] layout) must match."""
    B, L, d, h = 3, 11, 32, 4
    rng = np.random.default_rng(17 + causal)
    x = rng.standard_normal((B, L, d))
    w = _weights(d, 18)
    vl = np.array([11, 6, 1], dtype=np.int32)
    kpm = torch.from_numpy(np.arange(L)[None, :] >= vl[:, None])
    am = torch.triu(torch.ones(L, L, dtype=torch.bool), diagonal=1) if causal else None
    got = _run(x, x, x, w, h, causal=causal, valid_lens=vl)
    ref = _torch_mha(x, x, x, w, h, key_padding=kpm, attn_mask=am)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_cross_attention_matches_torch():
    B, Lq, Lk, d, h = 2, 4, 9, 16, 2
    rng = np.random.default_rng(19)
    q = rng.standard_normal((B, Lq, d)); m = rng.standard_normal((B, Lk, d))
    w = _weights(d, 20)
    vl = np.array([9, 5], dtype=np.int32)
    kpm = torch.from_numpy(np.arange(Lk)[None, :] >= vl[:, None])
    np.testing.assert_allclose(_run(q, m, m, w, h, valid_lens=vl),
                               _torch_mha(q, m, m, w, h, key_padding=kpm), rtol=0, atol=1e-12)


def test_linear_is_nn_linear_layout():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((3, 5)); W = rng.standard_normal((4, 5)); b = rng.standard_normal(4)
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(W), torch.from_numpy(b))
    np.testing.assert_allclose(oracle.linear(x, W, b), ref.numpy(), rtol=0, atol=1e-14)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("mask", ["none", "pad", "causal", "dense"])
def test_brute_force_tiny(mask):
    """Pure-Python loops on L_q=2, L_k=3 (L_q=L_k=3 for causal), d_model=4, h=2."""
    rng = np.random.default_rng(23)
    B, d, h = 2, 4, 2
    Lq, Lk = (3, 3) if mask == "causal" else (2, 3)
    q = rng.standard_normal((B, Lq, d)); k = rng.standard_normal((B, Lk, d))
    v = rng.standard_normal((B, Lk, d))
    w = _weights(d, 24)
    kw = {}
    if mask == "pad":
        kw["valid_lens"] = [2, 3]
    if mask == "causal":
        kw["causal"] = True
    if mask == "dense":
        kw["dense"] = rng.integers(0, 2, (B, Lq, Lk)).astype(np.uint8)
        kw["dense"][0, 1, :] = 0          # one fully masked row
    ob, pb = brute.mha_forward(q.tolist(), k.tolist(), v.tolist(),
                               *[w[n].tolist() for n in ("w_q", "b_q", "w_k", "b_k", "w_v", "b_v",
                                                          "w_o", "b_o")], h,
                               causal=kw.get("causal", False), valid_lens=kw.get("valid_lens"),
                               dense=None if "dense" not in kw else kw["dense"].tolist())
    oc, pc = _run(q, k, v, w, h, want_p_attn=True, **kw)
    np.testing.assert_allclose(oc, np.array(ob), rtol=0, atol=1e-12)
    np.testing.assert_allclose(pc, np.array(pb), rtol=0, atol=1e-12)


def test_sampled_rows_equal_full_rows():
    B, L, d, h = 2, 13, 16, 4
    rng = np.random.default_rng(25)
    x = rng.standard_normal((B, L, d)); w = _weights(d, 26)
    rows = [0, 4, 12]
    full, pf = _run(x, x, x, w, h, causal=True, valid_lens=[13, 9], want_p_attn=True)
    part, pp = _run(x, x, x, w, h, causal=True, valid_lens=[13, 9], rows=rows, want_p_attn=True)
    np.testing.assert_array_equal(full[:, rows], part)
    np.testing.assert_array_equal(pf[:, :, rows], pp)


def test_rejects_indivisible_heads():
    x = np.zeros((1, 2, 6))
    with pytest.raises(ValueError):
        _run(x, x, x, _weights(6, 1), 4)


# ---------------------------------------------------------------- planted mistakes
def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant mistakes in the brute-force oracle (CPU) and check a pin fails for each."""
    g = json.load(open(os.path.join(GOLDEN, "thinking_machines.json")))
    d = g["d_k"]
    eye = np.eye(d).tolist()
    q = [[[1.0] + [0.0] * (d - 1)]]
    k = [[[g["raw_scores"][0]] + [0.0] * (d - 1), [g["raw_scores"][1]] + [0.0] * (d - 1)]]
    v = [[[1.0] + [0.0] * (d - 1), [0.0, 1.0] + [0.0] * (d - 2)]]

    def weights_of(fn):
        _, p = fn(q, k, v, eye, None, eye, None, eye, None, eye, None, 1)
        return p[0][0][0]

    assert np.allclose(weights_of(brute.mha_forward), g["weights"], atol=1e-15)
    # mistake 1: scale dropped (sqrt(d_k) -> 1)
    monkeypatch.setattr(brute.math, "sqrt", lambda x: 1.0)
    assert not np.allclose(weights_of(brute.mha_forward), g["weights"], atol=1e-3)
    monkeypatch.undo()
    # mistake 2: the causal diagonal excluded (j >= i masked instead of j > i)
    orig = brute.allowed
    monkeypatch.setattr(brute, "allowed",
                        lambda b, i, j, c, vl, dn: orig(b, i, j, c, vl, dn) and not (c and j == i))
    x = np.random.default_rng(1).standard_normal((1, 3, 4)).tolist()
    w = _weights(4, 2)
    wl = [w[n].tolist() for n in ("w_q", "b_q", "w_k", "b_k", "w_v", "b_v", "w_o", "b_o")]
    _, p_bad = brute.mha_forward(x, x, x, *wl, 2, causal=True)
    monkeypatch.undo()
    _, p_ok = brute.mha_forward(x, x, x, *wl, 2, causal=True)
    rows = [l for l in open(os.path.join(GOLDEN, "subsequent_mask_5.txt")) if not l.startswith("#")]
    printed = np.array([[int(t) for t in l.split()] for l in rows if l.strip()])[:3, :3]
    assert np.all((np.array(p_ok[0][0]) > 0) == (printed == 1))
    assert not np.all((np.array(p_bad[0][0]) > 1e-6) == (printed == 1))


def test_workload_generator_is_seeded_and_bf16_exact():
    a = wlmod.make_inputs(wlmod.WORKLOADS["enc"], B=2)
    b = wlmod.make_inputs(wlmod.WORKLOADS["enc"], B=2)
    np.testing.assert_array_equal(a.query, b.query)
    t = torch.from_numpy(a.query)
    assert torch.equal(t, t.to(torch.bfloat16).float())
    assert a.valid_lens.min() >= 64 and a.valid_lens.max() <= 128
