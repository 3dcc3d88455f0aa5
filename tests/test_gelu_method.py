"""The epilogues' GELU: Abramowitz & Stegun 7.1.26 erf (CPU check of the transcription).

The formula is evaluated in float32 the way the kernels evaluate it and compared
with the exact erf GELU (scipy, float64); the published bound |erf error| <=
1.5e-7 gives |GELU error| <= 0.5 * 1.5e-7 * |x| plus float32 rounding.
"""
import numpy as np
from scipy.special import erf


def gelu_as7126_f32(x):
    """float32, in the kernels' order: constants folded (p/sqrt2, log2(e)/2, the 1/2 of Phi)."""
    x = x.astype(np.float32)
    p_s = np.float32(0.3275911 * 0.7071067811865476)
    h = [np.float32(0.5 * v) for v in (0.254829592, -0.284496736, 1.421413741, -1.453152027, 1.061405429)]
    ax = np.abs(x)
    t = np.float32(1) / (p_s * ax + np.float32(1))
    half_erfc = t * ((((h[4] * t + h[3]) * t + h[2]) * t + h[1]) * t + h[0]) * \
        np.exp2((x * x) * np.float32(-0.7213475204444817))
    return x * np.where(x >= 0, np.float32(1) - half_erfc, half_erfc)


def test_gelu_as7126_error_bound():
    x = np.linspace(-12, 12, 200001).astype(np.float64)
    exact = 0.5 * x * (1 + erf(x / np.sqrt(2)))
    got = gelu_as7126_f32(x).astype(np.float64)
    err = np.abs(got - exact)
    bound = 0.5 * 1.5e-7 * np.abs(x) + 4 * np.finfo(np.float32).eps * np.abs(exact) + 1e-12
    assert np.all(err <= bound), float(np.max(err / bound))
    assert np.max(err) < 1e-6
