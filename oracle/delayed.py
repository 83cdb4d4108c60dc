"""Delayed scaling with an amax history (Flax guide, sections 2.3 and 5.1).

Test infrastructure only (see ``oracle/__init__``).

State per quantized tensor: an fp32 history of length L (1024 in the guide,
initialised to zeros) and an fp32 scale (initialised to 1.0) -- section 5.1.

One use of the state (``in_q``, section 2.3), in the guide's order:

1. ``new_scale`` is computed from the max of the history as it stands (the
   previous steps' amaxes): ``amax_from_history = max(history)``.
2. the input is quantized with ``new_scale``.
3. the history takes the current input's amax: ``roll(history, -1)`` then
   element 0 is overwritten with it (``compute_amax_history``).

``compute_scale`` is not printed on the page; it says the algorithm follows
Transformer Engine's ``update_fp8_metas`` and keeps the old scale when the
history max is zero or not finite.  Plain reading adopted (consistent with the
page's ``scale = amax / MAX``): ``new_scale = fl32(max / MAX)`` when
``max > 0`` and finite, else the old scale.

Pins (``tests/test_oracle_delayed.py``): the ``fp32_max_grad`` worked example
of section 5.3 (one push of 3.0 into a zero history gives ``[3, 0, ..., 0]``
and the scale stays 1.0); a hand recomputation of 16 steps with a plain Python
list; the sliding-window property.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .formats import fmt_of
from .quantize import amax, quantize_with_scale

F32 = np.float32


@dataclass
class DelayedState:
    history: np.ndarray  # float32 [L]
    scale: np.float32

    @staticmethod
    def initial(length: int = 1024) -> "DelayedState":
        return DelayedState(np.zeros(length, dtype=F32), F32(1.0))

    def copy(self) -> "DelayedState":
        return DelayedState(self.history.copy(), F32(self.scale))


def compute_scale(amax_from_history, old_scale, fmt) -> np.float32:
    f = fmt_of(fmt)
    m = F32(amax_from_history)
    if np.isfinite(m) and m > 0:
        return F32(m / F32(f.max))
    return F32(old_scale)


def compute_amax_history(current_amax, history) -> np.ndarray:
    new = np.roll(np.asarray(history, dtype=F32), -1)
    new[0] = F32(current_amax)
    return new


def update_meta(x, fmt, state: DelayedState):
    """(new_scale, new_history) for input x -- ``update_fp8_meta``."""
    new_scale = compute_scale(np.max(state.history), state.scale, fmt)
    new_hist = compute_amax_history(amax(x), state.history)
    return new_scale, new_hist


def in_q(x, fmt, state: DelayedState):
    """Quantize x with the delayed scale; returns (codes, scale_used, new_state)."""
    new_scale, new_hist = update_meta(x, fmt, state)
    q = quantize_with_scale(x, new_scale, fmt)
    return q, new_scale, DelayedState(new_hist, new_scale)
