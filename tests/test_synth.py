"""The seeded input generator: deterministic, in the documented draw order, N(0, 1)."""
import torch

from head_dim_attention_gb300.synth import make_inputs


def test_same_seed_same_bits():
    a = make_inputs(1, 2, 1, 33, 47, 64, dtype=torch.float16, bias=True, grad=True, seed=5)
    b = make_inputs(1, 2, 1, 33, 47, 64, dtype=torch.float16, bias=True, grad=True, seed=5)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v), (a.bias, b.bias), (a.do, b.do)):
        assert torch.equal(x, y)
    c = make_inputs(1, 2, 1, 33, 47, 64, dtype=torch.float16, bias=True, grad=True, seed=6)
    assert not torch.equal(a.q, c.q)


def test_shapes_dtypes_and_bias_forms():
    x = make_inputs(2, 4, 2, 5, 7, 64, dtype=torch.bfloat16, bias="query", grad=True)
    assert x.q.shape == (2, 4, 5, 64) and x.k.shape == (2, 2, 7, 64) and x.v.shape == (2, 2, 7, 64)
    assert x.do.shape == (2, 4, 5, 64)
    assert x.q.dtype == x.k.dtype == x.v.dtype == x.do.dtype == torch.bfloat16
    assert x.bias.shape == (1, 1, 5, 7) and x.bias.dtype == torch.float32
    y = make_inputs(1, 1, 1, 5, 7, 64, bias=True)
    assert y.bias.shape == (1, 1, 1, 7) and y.do is None
    assert make_inputs(1, 1, 1, 5, 7, 64).bias is None


def test_draw_order_q_k_v_bias_do():
    # one generator, drawn in the order q, k, v, bias, dO, each in float32 then cast
    B, Hq, Hkv, Nq, Nkv, D = 1, 2, 1, 3, 4, 64
    x = make_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype=torch.float16, bias=True, grad=True, seed=11)
    g = torch.Generator("cpu").manual_seed(11)
    want = [torch.randn(B, Hq, Nq, D, generator=g), torch.randn(B, Hkv, Nkv, D, generator=g),
            torch.randn(B, Hkv, Nkv, D, generator=g), torch.randn(1, 1, 1, Nkv, generator=g),
            torch.randn(B, Hq, Nq, D, generator=g)]
    got = [x.q, x.k, x.v, x.bias, x.do]
    for w, t in zip(want, got):
        assert torch.equal(w.to(t.dtype), t)


def test_standard_normal_moments():
    x = make_inputs(1, 1, 1, 256, 256, 512, dtype=torch.float32, seed=0)
    v = torch.cat([x.q.flatten(), x.k.flatten(), x.v.flatten()]).double()
    n = v.numel()
    assert abs(v.mean().item()) < 5 / n ** 0.5
    assert abs(v.var().item() - 1.0) < 10 * (2 / n) ** 0.5
