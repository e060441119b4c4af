"""The derived GPU tolerances (tests/tolerance.py) rest on closed-form
activation slopes; check them against central differences of the oracle's
activations, and the activation values against the oracle's."""
import numpy as np

from oracle import layer as L
from tests import tolerance as tol


def test_activation_slopes_match_central_differences():
    g = np.concatenate([np.linspace(-12, 12, 4001), [-1e-3, 0.0, 1e-3]])
    h = 1e-6
    for kind, f in ((0, L.silu), (1, L.gelu_tanh)):
        act, slope, ev = tol._act_slope_eval(g, kind)
        assert np.allclose(act, f(g), rtol=1e-15, atol=1e-300)
        fd = (f(g + h) - f(g - h)) / (2 * h)
        assert np.allclose(slope, np.abs(fd), rtol=1e-6, atol=1e-8)
        assert (ev >= 0).all() and np.isfinite(ev).all()
    # gelu_tanh's evaluation bound covers a few fp32 roundings of the value
    _, _, ev = tol._act_slope_eval(g, 1)
    act = L.gelu_tanh(g)
    assert (ev >= 4 * tol.U32 * np.abs(act)).all()
