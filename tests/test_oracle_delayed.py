"""Pins for the delayed-scaling state machine (oracle/delayed.py).

Evidence: the worked example the Flax guide prints in section 5.3, the history
layout that follows from the guide's printed ``compute_amax_history`` code
(roll by -1, then overwrite element 0), and a hand recomputation with a plain
Python list of amaxes.
"""
import numpy as np

import workloads
from golden.fixtures import load
from oracle import delayed as D
from oracle import quantize as Q

EX = load("fp32_max_grad_example.txt")
CONST = load("format_constants.txt")
F32 = np.float32


def test_worked_example_fp32_max_grad():
    L = int(CONST["amax_history_length"])
    st = D.DelayedState.initial(L)
    assert st.scale == CONST["initial_scale"] and not st.history.any()
    outs = []
    for v in EX["inputs"]:
        _, scale_used, new = D.in_q(np.array([v], F32), "e4m3", st)
        outs.append(new)
    mx_hist = np.maximum(outs[0].history, outs[1].history)
    mx_scale = max(outs[0].scale, outs[1].scale)
    assert mx_scale == EX["max_scale"]
    assert mx_hist[0] == EX["max_history_head"] and np.all(mx_hist[1:] == EX["history_tail"])
    sum_hist = outs[0].history + outs[1].history
    assert outs[0].scale + outs[1].scale == EX["sum_scale"]
    assert sum_hist[0] == EX["sum_history_head"] and np.all(sum_hist[1:] == EX["history_tail"])


def test_history_layout_from_printed_code():
    # roll(-1) then [0] = new: pushes a1, a2, a3 into 4 zeros -> [a3, 0, a1, a2]
    h = np.zeros(4, F32)
    for a in (1.0, 2.0, 3.0):
        h = D.compute_amax_history(a, h)
    assert list(h) == [3.0, 0.0, 1.0, 2.0]
    h = D.compute_amax_history(4.0, h)
    h = D.compute_amax_history(5.0, h)
    assert list(h) == [5.0, 2.0, 3.0, 4.0]


def test_sixteen_steps_hand_recomputed():
    L = 4
    st = D.DelayedState.initial(L)
    seen = []          # every amax pushed so far, oldest first
    expected_scale = 1.0
    for t in range(16):
        x = workloads.normal((8, 8), 2.0 ** ((t * 5) % 7 - 3), seed=100 + t).numpy()
        if t == 6:
            x[:] = 0.0  # an all-zero input step
        window = seen[-L:]
        m = max(window) if window else 0.0
        if m > 0:
            expected_scale = float(np.float32(np.float32(m) / np.float32(448.0)))
        q, scale_used, st = D.in_q(x, "e4m3", st)
        assert scale_used == expected_scale
        assert np.array_equal(q, Q.quantize_with_scale(x, F32(expected_scale), "e4m3"))
        seen.append(float(np.max(np.abs(x))))
        assert st.history[0] == seen[-1]
        window = seen[-L:]
        assert sorted(st.history) == sorted(window + [0.0] * (L - len(window)))
        assert float(np.max(st.history)) == max(seen[-L:])


def test_keeps_scale_on_zero_or_nonfinite_history():
    st = D.DelayedState(np.zeros(8, F32), F32(0.25))
    _, s, _ = D.in_q(np.ones(3, F32), "e4m3", st)
    assert s == F32(0.25)
    h = np.zeros(8, F32)
    h[3] = np.inf
    _, s, _ = D.in_q(np.ones(3, F32), "e4m3", D.DelayedState(h, F32(0.5)))
    assert s == F32(0.5)
    h[3] = np.nan
    _, s, _ = D.in_q(np.ones(3, F32), "e4m3", D.DelayedState(h, F32(0.5)))
    assert s == F32(0.5)


def test_window_forgets_after_L_pushes():
    L = 8
    h = np.zeros(L, F32)
    h = D.compute_amax_history(1000.0, h)
    for _ in range(L - 1):
        h = D.compute_amax_history(1.0, h)
    assert np.max(h) == 1000.0
    h = D.compute_amax_history(1.0, h)
    assert np.max(h) == 1.0
