"""Pins of the fp64 LayerNorm and residual-sublayer oracle.

"The Annotated Transformer", LayerNorm: a_2 (x - mean) / (std + eps) + b_2 with
torch's default (unbiased) std; SublayerConnection: x + dropout(sublayer(norm(x))).
"003-Transformer" uses nn.LayerNorm instead (biased variance, eps inside the root)."""
import math

import numpy as np
import torch

import oracle


def test_torch_kind_is_nn_layernorm():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 7, 16)) * 3 + 1
    a, b = rng.standard_normal(16), rng.standard_normal(16)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (16,), torch.from_numpy(a), torch.from_numpy(b),
                                         eps=1e-5)
    np.testing.assert_allclose(oracle.layernorm(x, a, b, 1e-5, oracle.LN_TORCH), ref.numpy(), rtol=0, atol=1e-12)


def test_annotated_kind_uses_unbiased_std():
    """With eps = 0 the two kinds differ exactly by sqrt((d - 1) / d) (unbiased vs biased std)."""
    rng = np.random.default_rng(2)
    d = 12
    x = rng.standard_normal((5, d))
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (d,), eps=0.0).numpy()
    np.testing.assert_allclose(oracle.layernorm(x, None, None, 0.0, oracle.LN_ANNOTATED),
                               ref * math.sqrt((d - 1) / d), rtol=0, atol=1e-12)


def test_annotated_closed_forms():
    # a constant row has x - mean = 0: the output is b_2 exactly
    b = np.arange(4.0)
    np.testing.assert_array_equal(oracle.layernorm(np.full((1, 4), 3.5), None, b, 1e-6, 0)[0], b)
    # [-1, 1]: mean 0, unbiased std sqrt(2): y = x / (sqrt(2) + eps)
    eps = 1e-6
    np.testing.assert_allclose(oracle.layernorm(np.array([[-1.0, 1.0]]), None, None, eps, 0)[0],
                               [-1 / (math.sqrt(2) + eps), 1 / (math.sqrt(2) + eps)], rtol=0, atol=1e-15)


def _mha_weights(d, seed):
    rng = np.random.default_rng(seed)
    bound = math.sqrt(6.0 / (2 * d))
    w = {}
    for n in "qkvo":
        w["w_" + n] = rng.uniform(-bound, bound, (d, d))
        w["b_" + n] = rng.uniform(-0.1, 0.1, d)
    return [w[n] for n in ("w_q", "b_q", "w_k", "b_k", "w_v", "b_v", "w_o", "b_o")]


def test_sublayer_is_residual_plus_attention_of_normed_input():
    rng = np.random.default_rng(3)
    B, L, d, h = 2, 6, 16, 4
    x = rng.standard_normal((B, L, d))
    a, b = rng.uniform(0.5, 1.5, d), rng.uniform(-0.1, 0.1, d)
    ws = _mha_weights(d, 4)
    got = oracle.sublayer_forward(x, a, b, 1e-6, 0, *ws, h, causal=True, valid_lens=[6, 3])
    y = oracle.layernorm(x, a, b, 1e-6, 0)
    ref = x + oracle.mha_forward(y, y, y, *ws, h, causal=True, valid_lens=[6, 3])
    np.testing.assert_array_equal(got, ref)
    # source attention: the memory is not normalised
    m = rng.standard_normal((B, 9, d))
    got2 = oracle.sublayer_forward(x, a, b, 1e-6, 1, *ws, h, memory=m, valid_lens=[9, 4])
    y2 = oracle.layernorm(x, a, b, 1e-6, 1)
    np.testing.assert_array_equal(got2, x + oracle.mha_forward(y2, m, m, *ws, h, valid_lens=[9, 4]))
    # zero output projection: the sublayer is the identity on x (residual only)
    ws0 = list(ws)
    ws0[6] = np.zeros((d, d)); ws0[7] = np.zeros(d)
    np.testing.assert_array_equal(oracle.sublayer_forward(x, a, b, 1e-6, 0, *ws0, h), x)


def _torch_sublayer(x, memory, a, b, eps, ws, h, key_pad):
    """Pre-norm source-attention sublayer composed from library routines in fp64: torch's
    layer_norm (the nn.LayerNorm form) on the query side only, torch's own
    multi_head_attention_forward with the memory as key and value, plus the residual.
    Nothing here calls the oracle."""
    F = torch.nn.functional
    t = lambda v: torch.from_numpy(np.asarray(v, dtype=np.float64))
    w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o = [t(v) for v in ws]
    d = x.shape[-1]
    y = F.layer_norm(t(x), (d,), t(a), t(b), eps=eps)
    out, _ = F.multi_head_attention_forward(
        y.transpose(0, 1), t(memory).transpose(0, 1), t(memory).transpose(0, 1), d, h,
        None, torch.cat([b_q, b_k, b_v]), None, None, False, 0.0, w_o, b_o, training=False,
        key_padding_mask=torch.from_numpy(key_pad), need_weights=False,
        use_separate_proj_weight=True, q_proj_weight=w_q, k_proj_weight=w_k, v_proj_weight=w_v)
    return t(x) + out.transpose(0, 1)


def test_source_attention_sublayer_against_torch_composition():
    """Source attention normalises the decoder input, not the encoder memory
    ("The Annotated Transformer", DecoderLayer: src_attn(x, m, m, src_mask) inside a
    SublayerConnection that applies norm to x only). Pinned against an independent
    composition of torch's fp64 layer_norm and multi_head_attention_forward; a
    normalised memory gives a different result and must fail the same comparison."""
    rng = np.random.default_rng(5)
    B, L, Lm, d, h = 2, 5, 7, 16, 4
    x = rng.standard_normal((B, L, d)) * 2 + 0.5
    m = rng.standard_normal((B, Lm, d)) * 3 - 1.0      # far from normalised
    a, b = rng.uniform(0.5, 1.5, d), rng.uniform(-0.1, 0.1, d)
    ws = _mha_weights(d, 6)
    vl = np.array([7, 4])
    pad = np.arange(Lm)[None, :] >= vl[:, None]       # torch: True = ignore this key
    got = oracle.sublayer_forward(x, a, b, 1e-5, oracle.LN_TORCH, *ws, h, memory=m, valid_lens=vl)
    ref = _torch_sublayer(x, m, a, b, 1e-5, ws, h, pad).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # the planted mistake: normalising the memory too moves the result well off
    m_normed = torch.nn.functional.layer_norm(torch.from_numpy(m), (d,), torch.from_numpy(a),
                                              torch.from_numpy(b), eps=1e-5).numpy()
    wrong = oracle.sublayer_forward(x, a, b, 1e-5, oracle.LN_TORCH, *ws, h, memory=m_normed, valid_lens=vl)
    assert np.abs(wrong - ref).max() > 1e-3
