"""A seeded sweep of problem shapes through mha_forward against the fp64 oracle, on
sampled query rows: head widths 8 to 128 in bf16 (tensor-core kernels, the narrow-head
form, the persistent d_k = 128 kernel) and 32 / 64 / 96 in fp32, self and cross
attention with aliased or distinct key / value, every mask kind and their
combinations, sequence lengths on both sides of the tile sizes and of the short-key
instance threshold (1024 keys). Same tolerances as the other parity tests."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from transformer_head_scaled_fwd_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_head_scaled_fwd_gb300 import build as B
    B.build()
    from transformer_head_scaled_fwd_gb300 import binding
    binding.load()
    binding.mha_check_device_status(reset=True)


from gpu_helpers import ROWSUM_TOL, assert_close, run_gpu, run_oracle  # noqa: E402

# (d_model, h) per dtype: bf16 d_k = 8, 16, 32, 64, 128; fp32 d_k = 32, 64, 96
BF16_HEADS = [(512, 64), (256, 16), (512, 16), (256, 4), (512, 8), (1024, 16), (512, 4), (1024, 8), (384, 3)]
F32_HEADS = [(256, 8), (512, 8), (384, 4)]
LENGTHS = [1, 2, 31, 127, 128, 129, 255, 256, 300, 640, 1023, 1025, 1300]


def _case(i):
    rng = np.random.default_rng(9000 + i)
    dtype = "f32" if i % 6 == 5 else "bf16"
    d, h = (F32_HEADS if dtype == "f32" else BF16_HEADS)[int(rng.integers(0, 3 if dtype == "f32" else 9))]
    self_attn = bool(rng.integers(0, 2))
    Lq = int(rng.choice(LENGTHS))
    Lk = Lq if self_attn else int(rng.choice(LENGTHS))
    B = int(rng.integers(1, 4))
    if dtype == "f32":   # keep the fp32 SIMT path small
        Lq, Lk = min(Lq, 300), min(Lk, 300)
        Lk = Lq if self_attn else Lk
    kind = ["none", "causal", "lens", "dense", "causal+lens", "dense+lens"][int(rng.integers(0, 6))]
    if "causal" in kind and not self_attn:
        kind = kind.replace("causal", "lens").replace("lens+lens", "lens")
    return dict(seed=9100 + i, dtype=dtype, B=B, Lq=Lq, Lk=Lk, d=d, h=h, self_attn=self_attn,
                kv_alias=bool(rng.integers(0, 2)), kind=kind,
                p_attn=bool(i % 4 == 0) and B * h * Lq * Lk <= 20_000_000, rng_seed=9200 + i)


def _fixed(i, dtype, B, Lq, Lk, d, h, kind, kv_alias=False, p_attn=False):
    return dict(seed=9500 + i, dtype=dtype, B=B, Lq=Lq, Lk=Lk, d=d, h=h, self_attn=False,
                kv_alias=kv_alias, kind=kind, p_attn=p_attn, rng_seed=9600 + i)


# cross attention far from square: one or a few queries over many keys, many queries
# over a few keys, three heads of 128, and key counts past the short-key threshold
CASES = [_case(i) for i in range(30)] + [
    _fixed(0, "bf16", 2, 1, 1300, 512, 8, "lens", p_attn=True),
    _fixed(1, "bf16", 3, 31, 2100, 384, 3, "dense+lens"),
    _fixed(2, "bf16", 2, 1300, 5, 512, 4, "dense", kv_alias=True),
    _fixed(3, "bf16", 1, 200, 4100, 1024, 8, "none"),
    _fixed(4, "bf16", 2, 129, 2049, 512, 8, "dense+lens", p_attn=True),
    _fixed(5, "f32", 2, 3, 700, 256, 4, "lens", p_attn=True),
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: (f"{c['dtype']}-B{c['B']}-{c['Lq']}x{c['Lk']}-d{c['d']}h{c['h']}-"
                                                     f"{'self' if c['self_attn'] else 'cross'}-{c['kind']}"))
def test_sweep_against_oracle(c):
    inp = W.random_case(c["seed"], c["B"], c["Lq"], c["Lk"], c["d"], c["h"], dtype=c["dtype"],
                        self_attn=c["self_attn"], kv_alias=c["kv_alias"])
    rng = np.random.default_rng(c["rng_seed"])
    kw = {}
    if "causal" in c["kind"]:
        kw["causal"] = True
    if "lens" in c["kind"]:
        kw["valid_lens"] = [int(x) for x in rng.integers(0, c["Lk"] + 1, size=c["B"])]
    if "dense" in c["kind"]:
        mq = c["Lq"] if rng.integers(0, 2) else 1
        kw["dense"] = (rng.random((c["B"], mq, c["Lk"])) < 0.6).astype(np.uint8)
    got, gp = run_gpu(inp, want_p_attn=c["p_attn"], **kw)
    rows = W.sample_rows(c["Lq"], 24, seed=c["rng_seed"])
    ref = run_oracle(inp, rows=rows, **kw)
    assert_close(got[:, rows], ref, c["dtype"])
    if gp is not None:
        np.testing.assert_allclose(gp.sum(-1), 1.0, atol=ROWSUM_TOL)
