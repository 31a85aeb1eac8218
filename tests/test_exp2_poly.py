"""The FMA-pipe exponential used for part of the forward softmax.

CPU: the committed float32 coefficients meet the error bound of their
relative-minimax fit on [0, 1).  GPU: the device routine (range split +
polynomial + exponent add) matches the exact 2^x within that bound plus
float32 rounding, over the whole argument range the softmax uses."""
import numpy as np
import pytest

from attention_tiled_fwd_gb300 import exp2_poly_fit


def test_committed_coefficients_meet_their_bound():
    assert exp2_poly_fit.max_rel_error(exp2_poly_fit.COEFFS) <= exp2_poly_fit.MAX_REL_ERR * 1.001


def test_fit_reproduces_committed_coefficients():
    c, e = exp2_poly_fit.remez()
    np.testing.assert_allclose(np.float32(c), np.float32(exp2_poly_fit.COEFFS), rtol=2e-7)
    assert e <= exp2_poly_fit.MAX_REL_ERR


@pytest.mark.gpu
def test_device_exp2_matches_exact_power_of_two():
    import torch
    from helpers import cuda_or_skip
    from attention_tiled_fwd_gb300 import _native
    dev = cuda_or_skip()
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.linspace(-125.0, 8.0, 400001), -125.0 + 133.0 * torch.rand(200000, generator=g),
                   torch.tensor([-125.0, -1e-7, 0.0, 1e-7, 0.5, 1.0, 7.999, 8.0])]).float()
    xd = x.to(dev)
    yd = torch.empty_like(xd)
    _native.check(_native.load().fa_selftest_exp2(xd.data_ptr(), yd.data_ptr(), xd.numel(), None), "exp2")
    torch.cuda.synchronize()
    exact = np.exp2(x.double().numpy())
    rel = np.abs(yd.double().cpu().numpy() / exact - 1.0)
    assert rel.max() <= exp2_poly_fit.MAX_REL_ERR + 4e-7, rel.max()
