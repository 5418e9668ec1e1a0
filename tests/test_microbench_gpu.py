"""The instruction probes' FMA-pipe exp2 meets the accuracy its description
states: relative error at most 7.5e-5 against the exact 2^x (float64) over
x in [-125, 0], the range the softmax exponents take; CUDA's exp2f is
evaluated beside it on the same inputs for comparison."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_exp2_poly_relative_error_bound():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_forward_mbarrier_gb300 import microbench

    x = np.concatenate([np.linspace(-125.0, 0.0, 1 << 20), -np.arange(0, 126, 0.5)]).astype(np.float32)
    y_poly, y_exp2f = microbench.exp2_poly_values(x)
    exact = np.exp2(x.astype(np.float64))
    rel_poly = np.abs(y_poly - exact) / exact
    rel_exp2f = np.abs(y_exp2f - exact) / exact
    assert rel_poly.max() <= 7.5e-5, rel_poly.max()
    assert rel_exp2f.max() <= 1e-6, rel_exp2f.max()
