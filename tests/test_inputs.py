"""The seeded input recipe shared by the tests and the bench (CPU only)."""
import torch

from sliding_window_attention_prefill_gb300 import inputs


def test_same_seed_same_bits_and_seeds_differ():
    a = inputs.prefill_inputs(1, 64, 4, 2, 32, seed=5)
    b = inputs.prefill_inputs(1, 64, 4, 2, 32, seed=5)
    c = inputs.prefill_inputs(1, 64, 4, 2, 32, seed=6)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert not torch.equal(a[0], c[0])


def test_sink_rows_are_exactly_eight_times_the_plain_draw():
    for dt in (torch.bfloat16, torch.float16):
        q0, k0, v0 = inputs.prefill_inputs(2, 40, 4, 2, 32, seed=3, dtype=dt)
        q1, k1, v1 = inputs.prefill_inputs(2, 40, 4, 2, 32, seed=3, sink_rows=4, dtype=dt)
        assert k1.dtype == dt
        assert torch.equal(q0, q1) and torch.equal(v0, v1)
        assert torch.equal(k1[:, 4:], k0[:, 4:])
        # a power of two: exact in both 16-bit types at these magnitudes
        assert torch.equal(k1[:, :4].float(), 8.0 * k0[:, :4].float())


def test_standard_normal_rounded_to_16_bits():
    g = inputs.generator(0)
    x = inputs.normal_bf16((1 << 20,), g)
    assert x.dtype == torch.bfloat16
    f = x.float()
    assert abs(f.mean().item()) < 5e-3 and abs(f.std().item() - 1.0) < 5e-3
    # the draw is float32 N(0,1) rounded once to bf16
    g2 = inputs.generator(0)
    ref = torch.randn(1 << 20, generator=g2, dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(x, ref)


def test_decode_stream_shapes():
    kp, vp, ks, vs, qs = inputs.decode_stream(3, 8, 2, 16, prompt=10, steps=4, seed=1)
    assert kp.shape == (3, 10, 2, 16) and vp.shape == (3, 10, 2, 16)
    assert ks.shape == (4, 3, 1, 2, 16) and vs.shape == (4, 3, 1, 2, 16)
    assert qs.shape == (4, 3, 8, 16)
