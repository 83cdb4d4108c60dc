"""Quantization signal-to-noise ratio (MOSS blog, section 2).

Test infrastructure only (see ``oracle/__init__``).

SNR is the power of the signal over the power of the quantization error,
reported in dB: ``10 * log10(sum x**2 / sum (x - x_hat)**2)``.  The blog
notes that equation (4) writes the ratio and its dB form on one line; the two
are separate steps here.  The RMS normalisation of section 3 divides both sums
by n, which cancels.

Pins (``tests/test_oracle_snr.py``): an exactly representable tensor gives
+inf; a constant signal with a known +-delta error gives -20*log10(delta).
"""
from __future__ import annotations

import numpy as np


def snr_db(x, x_hat) -> float:
    x = np.asarray(x, dtype=np.float64)
    d = x - np.asarray(x_hat, dtype=np.float64)
    sig = float(np.sum(x * x))
    noise = float(np.sum(d * d))
    if noise == 0.0:
        return float("inf")
    return 10.0 * np.log10(sig / noise)
