"""Logical model of the sliding observation window (test infrastructure only).

"Reflex: Real-Time VLA Control through Streaming Inference", §III "System
architecture", ring-buffer partitions: the sliding history is a FIFO queue of
N observations; every step enqueues the newest frame and evicts the oldest.
§V "Key implementation": ``add_new_prefix()`` adds the new observation tokens
and returns the eviction count; ``evict_source_prefix()`` removes the oldest
frame's tokens from all layers.

The window is kept as a plain Python list in logical order, oldest first.
"""
from __future__ import annotations

from typing import Any, List


class FrameWindow:
    """FIFO of at most ``N`` frames.  Frames are opaque objects."""

    def __init__(self, N: int):
        if N < 1:
            raise ValueError("window needs N >= 1 frames")
        self.N = N
        self.frames: List[Any] = []

    def push(self, frame: Any) -> int:
        """Enqueue the newest frame; evict the oldest if the window overflows.

        Returns the number of frames evicted (0 or 1), the count that
        ``add_new_prefix()`` reports.
        """
        self.frames.append(frame)
        if len(self.frames) > self.N:
            self.frames.pop(0)
            return 1
        return 0

    def window(self) -> List[Any]:
        """Frames currently in the window, oldest first."""
        return list(self.frames)

    @property
    def valid(self) -> int:
        return len(self.frames)
