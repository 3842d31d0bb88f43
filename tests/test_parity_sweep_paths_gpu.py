"""Seeded shape sweeps of the other paths against the fp64 oracle: the position-wise FFN
("003-Transformer" tutorial, feed-forward layer), the pre-norm residual sublayer ("The Annotated
Transformer", SublayerConnection, both LayerNorm forms) and incremental decoding (each new token
attends to every cached token and itself: causal self-attention row by row). Outputs compared on
sampled rows with the same tolerances as the other parity tests."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from transformer_head_scaled_fwd_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu
WN = ("w_q", "b_q", "w_k", "b_k", "w_v", "b_v", "w_o", "b_o")
TOL = {"bf16": (1.5e-2, 2e-2), "f32": (1e-4, 1e-4)}


@pytest.fixture(scope="module")
def bnd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_head_scaled_fwd_gb300 import build as B
    B.build()
    from transformer_head_scaled_fwd_gb300 import binding
    binding.load()
    binding.mha_check_device_status(reset=True)
    return binding


def _check(got, ref, dtype, what="out"):
    atol, rtol = TOL[dtype]
    err = np.abs(got - ref)
    bad = ~(err <= atol + rtol * np.abs(ref))
    assert not bad.any(), f"{what}: {int(bad.sum())} of {err.size} outside tolerance, max abs err {err.max():.3e}"


def _tdt(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


# ------------------------------------------------------------------ FFN
def _ffn_case(i):
    rng = np.random.default_rng(7000 + i)
    dtype = "f32" if i % 4 == 3 else "bf16"
    if dtype == "bf16":
        d = int(rng.choice([64, 192, 512, 1024]))
        d_ff = int(rng.choice([64, 320, 1024, 2048]))
    else:
        d = int(rng.choice([48, 96, 256]))
        d_ff = int(rng.choice([100, 384]))
    B = int(rng.integers(1, 5))
    L = int(rng.choice([1, 5, 77, 128, 129, 300, 600]))
    return dict(i=i, dtype=dtype, B=B, L=L, d=d, d_ff=d_ff)


@pytest.mark.parametrize("c", [_ffn_case(i) for i in range(12)],
                         ids=lambda c: f"{c['dtype']}-B{c['B']}-L{c['L']}-d{c['d']}-ff{c['d_ff']}")
def test_ffn_sweep(bnd, c):
    inp = W.make_ffn_inputs(c["B"], c["L"], c["d"], c["d_ff"], seed=7100 + c["i"], dtype=c["dtype"])
    dt = _tdt(c["dtype"])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dt)
    x = dev(inp.x)
    code = bnd.MHA_BF16 if c["dtype"] == "bf16" else bnd.MHA_F32
    ws = torch.empty(bnd.ffn_workspace_size(code, c["B"], c["L"], c["d"], c["d_ff"]), dtype=torch.uint8,
                     device="cuda")
    out = torch.full_like(x, float("nan"))
    bnd.mha_ffn_forward(x, dev(inp.w_1), dev(inp.b_1), dev(inp.w_2), dev(inp.b_2), out=out, workspace=ws)
    torch.cuda.synchronize()
    assert bnd.mha_check_device_status(reset=True) == 0
    rows = W.sample_rows(c["L"], 32, seed=7200 + c["i"])
    ref = oracle.ffn_forward(inp.x[:, rows], inp.w_1, inp.b_1, inp.w_2, inp.b_2)
    _check(out.double().cpu().numpy()[:, rows], ref, c["dtype"])


# ------------------------------------------------------------------ residual sublayer
def _sub_case(i):
    rng = np.random.default_rng(7300 + i)
    dtype = "f32" if i % 4 == 3 else "bf16"
    d, h = ([(256, 4), (512, 8), (1024, 8), (512, 4)] if dtype == "bf16" else [(96, 3), (256, 4)])[
        int(rng.integers(0, 4 if dtype == "bf16" else 2))]
    B = int(rng.integers(1, 4))
    L = int(rng.choice([1, 33, 128, 200, 300]))
    source = bool(rng.integers(0, 2))
    L_mem = int(rng.choice([1, 40, 129, 257])) if source else 0
    return dict(i=i, dtype=dtype, B=B, L=L, d=d, h=h, source=source, L_mem=L_mem, kind=int(i % 2),
                eps=1e-6 if i % 2 == 0 else 1e-5)


@pytest.mark.parametrize("c", [_sub_case(i) for i in range(10)],
                         ids=lambda c: (f"{c['dtype']}-B{c['B']}-L{c['L']}-d{c['d']}h{c['h']}-"
                                        f"{'source' + str(c['L_mem']) if c['source'] else 'self'}-ln{c['kind']}"))
def test_sublayer_sweep(bnd, c):
    B, L, d, h = c["B"], c["L"], c["d"], c["h"]
    inp = W.random_case(7400 + c["i"], B, L, L, d, h, self_attn=True, dtype=c["dtype"], bias_scale=0.05)
    ln = W.make_ln_params(d, seed=7500 + c["i"], dtype=c["dtype"])
    rng = np.random.default_rng(7600 + c["i"])
    dt = _tdt(c["dtype"])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dt)
    mem = W.random_case(7700 + c["i"], B, c["L_mem"], c["L_mem"], d, h, self_attn=True,
                        dtype=c["dtype"]).query if c["source"] else None
    Lk = c["L_mem"] if c["source"] else L
    vl = [int(v) for v in rng.integers(1, Lk + 1, size=B)]
    causal = not c["source"]
    x = dev(inp.query)
    code = bnd.MHA_BF16 if c["dtype"] == "bf16" else bnd.MHA_F32
    ws = torch.empty(bnd.sublayer_workspace_size(code, B, L, c["L_mem"], d, h), dtype=torch.uint8, device="cuda")
    out = torch.full_like(x, float("nan"))
    vlt = torch.tensor(vl, dtype=torch.int32, device="cuda")
    bnd.mha_sublayer_forward(x, dev(ln[0]), dev(ln[1]), c["eps"], c["kind"], *[dev(inp.weights[n]) for n in WN], h,
                             out=out, workspace=ws, memory=None if mem is None else dev(mem),
                             mask=bnd.make_mask(causal, vlt, None))
    torch.cuda.synchronize()
    assert bnd.mha_check_device_status(reset=True) == 0
    rows = W.sample_rows(L, 24, seed=7800 + c["i"])
    ref = oracle.sublayer_forward(inp.query, ln[0], ln[1], c["eps"], c["kind"], *[inp.weights[n] for n in WN], h,
                                  memory=mem, causal=causal, valid_lens=vl, rows=rows)
    _check(out.double().cpu().numpy()[:, rows], ref, c["dtype"])


# ------------------------------------------------------------------ incremental decoding
def _dec_case(i):
    rng = np.random.default_rng(7900 + i)
    d, h = [(256, 4), (512, 8), (512, 4), (1024, 16), (1024, 8)][int(rng.integers(0, 5))]   # d_k 64 / 128
    B = int(rng.choice([1, 3, 8, 17, 64]))
    T0 = int(rng.choice([0, 1, 63, 200, 700]))
    return dict(i=i, B=B, d=d, h=h, T0=T0, steps=int(rng.integers(1, 4)), L_max=T0 + 8)


@pytest.mark.parametrize("c", [_dec_case(i) for i in range(8)],
                         ids=lambda c: f"B{c['B']}-d{c['d']}h{c['h']}-T0{c['T0']}-steps{c['steps']}")
def test_decode_sweep(bnd, c):
    B, d, h, T0, steps, L_max = c["B"], c["d"], c["h"], c["T0"], c["steps"], c["L_max"]
    T = T0 + steps
    inp = W.random_case(8000 + c["i"], B, T, T, d, h, self_attn=True, bias_scale=0.05)
    rng = np.random.default_rng(8100 + c["i"])
    # ragged histories: sequence b starts decoding after lens[b] <= T0 cached tokens
    lens = [int(v) for v in rng.integers(0, T0 + 1, size=B)] if T0 > 0 else [0] * B
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(torch.bfloat16)
    w = [bf(inp.weights[n]) for n in WN]
    k = torch.zeros(B, h, L_max, d // h, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    if T0 > 0:
        bnd.mha_kv_cache_prefill(bf(inp.query[:, :T0]), w[2], w[3], w[4], w[5], h, k_cache=k, v_cache=v)
    clen = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ws = torch.empty(bnd.decode_workspace_size(B, d, h, L_max), dtype=torch.uint8, device="cuda")
    ww = [inp.weights[n] for n in WN]
    for s in range(steps):
        pos = [lens[b] + s for b in range(B)]
        x_new = np.stack([inp.query[b, pos[b]] for b in range(B)])
        out = torch.full((B, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        bnd.mha_decode_step(bf(x_new), *w, h, k_cache=k, v_cache=v, cache_len=clen, out=out, workspace=ws)
        torch.cuda.synchronize()
        assert bnd.mha_check_device_status(reset=True) == 0
        got = out.double().cpu().numpy()
        for b in sorted({0, B - 1} | {int(v) for v in rng.integers(0, B, size=2)}):   # up to 4 sequences
            xb = inp.query[b:b + 1, :pos[b] + 1]
            ref = oracle.mha_forward(xb, xb, xb, *ww, h, causal=True, rows=[pos[b]])
            _check(got[b], ref[0, 0], "bf16", what=f"step {s} sequence {b}")
    assert clen.cpu().tolist() == [l + steps for l in lens]
