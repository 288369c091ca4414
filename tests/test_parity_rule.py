"""The tolerance rule for 16-bit outputs averaged from large values
(tests/parity.py), pinned to the formats and to the rounding steps it is
derived from: bf16 keeps 7 stored mantissa bits, fp16 10."""
import numpy as np
import pytest
import torch

from .parity import abs_values, assert_close_16, bounds_16, scale_16_bits


def _emulated_16bit_attention(scores, v, dtype):
    """softmax(scores) . v with the weights rounded to the 16-bit type before
    the product and the output rounded at the end (the GPU path's roundings);
    everything else in float64.  Returns (out, exact, A)."""
    s = torch.from_numpy(scores)
    p = torch.exp(s - s.max(dim=-1, keepdim=True).values)
    l = p.sum(dim=-1, keepdim=True)
    vv = torch.from_numpy(v)
    exact = (p @ vv) / l
    pr = p.to(dtype).double()
    out = ((pr @ vv) / l).to(dtype).double()
    a = (p @ vv.abs()) / l
    return out.numpy(), exact.numpy(), a.numpy()


@pytest.mark.parametrize("dtype,name", [(torch.bfloat16, "bf16"), (torch.float16, "f16")])
@pytest.mark.parametrize("v_scale,s_scale", [(1.0, 1.0), (16.0, 16.0), (64.0, 4.0)])
def test_rule_holds_for_the_rounding_it_is_derived_from(dtype, name, v_scale, s_scale):
    rng = np.random.default_rng(int(v_scale + s_scale))
    scores = rng.normal(0, s_scale, size=(64, 300))
    v = torch.from_numpy(rng.normal(0, v_scale, size=(300, 128))).to(dtype).double().numpy()
    out, exact, a = _emulated_16bit_attention(scores, v, dtype)
    lse = np.zeros(64)
    assert_close_16(out, lse, exact, lse, a, name)
    # an error of 2^-(m-2) A (four times the allowed one) on one element fails
    m = 7 if name == "bf16" else 10
    bad = out.copy()
    i = np.unravel_index(np.argmax(a), a.shape)
    bad[i] += max(4 * 2.0 ** -m * a[i], 4e-2)
    with pytest.raises(AssertionError):
        assert_close_16(bad, lse, exact, lse, a, name)


def test_values_of_order_one_keep_the_stated_bars():
    # bf16: 2^-7 A stays at or below 1e-2 for A up to 1.28; fp16: up to 10.24
    bound, large = bounds_16(np.full(10, 1.2), "bf16")
    assert np.all(bound == 1e-2) and not large.any()
    bound, large = bounds_16(np.full(10, 16.0), "bf16")
    assert np.all(bound == 16.0 / 128) and large.all()
    bound, large = bounds_16(np.array([8.0, 16.0]), "f16")
    assert bound.tolist() == [1e-2, 16.0 / 1024] and large.tolist() == [False, True]


def test_sign_clearing_and_power_of_two_scaling_are_exact():
    x = torch.randn(1000).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    back = torch.from_numpy(abs_values(bits).view(np.int16)).view(torch.bfloat16)
    assert torch.equal(back, x.abs())
    up = scale_16_bits(bits, 16.0)
    assert torch.equal(torch.from_numpy(up.view(np.int16)).view(torch.bfloat16), x * 16)
