"""Pins for the oracle's FIFO window (CPU only).

"Reflex: Real-Time VLA Control through Streaming Inference", §III "System
architecture": each tick enqueues the newest frame and evicts the oldest; the
window holds N frames.  Closed form: after T pushes of ids 0..T-1 the window
is ids max(0, T-N) .. T-1 in order, and a push evicts exactly when T > N.
"""
import os

import pytest

from oracle.ring import FrameWindow

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("N", [1, 2, 3, 4, 8, 32])
def test_window_closed_form(N):
    w = FrameWindow(N)
    assert w.window() == [] and w.valid == 0
    for T in range(1, 3 * N + 2):
        ev = w.push(T - 1)
        assert ev == (1 if T > N else 0)
        assert w.window() == list(range(max(0, T - N), T))
        assert w.valid == min(T, N)


def test_window_golden_n3():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "fifo_window_N3.txt"))
            if l.strip() and not l.startswith("#")]
    w = FrameWindow(3)
    for r in rows:
        T = int(r[0])
        if T == 0:
            assert w.window() == []
            continue
        ev = w.push(T - 1)
        assert ev == int(r[1])
        assert w.window() == [int(x) for x in r[2].split(",")]


def test_window_rejects_zero_frames():
    with pytest.raises(ValueError):
        FrameWindow(0)
