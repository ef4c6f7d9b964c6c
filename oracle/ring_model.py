"""StreamingLLM-style draft cache model -- TEST INFRASTRUCTURE ONLY.

The draft cache of "Windowed-MTP: Removing the Full-Context Draft-KV Tax at
Million-Token Context" (Abstract) keeps the attention sinks and a sliding
window of recent entries; everything older is dropped ("reclaimed via a
compact ring buffer").  This module states that behaviour with textbook
containers -- a list that keeps the first S positions ever appended and a
``collections.deque(maxlen=W)`` that keeps the W most recent later ones -- so
that it shares nothing with the slot arithmetic of the CUDA ring buffer.

It answers two questions the tests ask:
  * which positions does the draft cache hold after positions 0..p were
    appended one at a time (the draft's key set at query position p);
  * after a rollback to a shorter length, which of the held positions are
    still valid.
"""
from __future__ import annotations

from collections import deque


class StreamingCache:
    def __init__(self, sink: int, window: int):
        if sink < 0 or window < 1:
            raise ValueError("sink >= 0 and window >= 1 required")
        self.sink = sink
        self.window = window
        self.sinks: list[int] = []
        self.recent: deque[int] = deque(maxlen=window)
        self.n_seen = 0

    def append(self, pos: int) -> None:
        """Append the entry of position ``pos`` (positions arrive in order)."""
        if pos != self.n_seen:
            raise ValueError("positions must be appended in order")
        if len(self.sinks) < self.sink:
            self.sinks.append(pos)
        else:
            self.recent.append(pos)
        self.n_seen += 1

    def held(self) -> list[int]:
        """Positions currently held, ascending."""
        return sorted(self.sinks + list(self.recent))

    def rollback(self, new_len: int) -> None:
        """Forget positions >= new_len (speculative entries that were rejected)."""
        if new_len > self.n_seen or new_len < 0:
            raise ValueError("rollback beyond the appended length")
        self.sinks = [p for p in self.sinks if p < new_len]
        kept = [p for p in self.recent if p < new_len]
        self.recent = deque(kept, maxlen=self.window)
        self.n_seen = new_len


def held_after(sink: int, window: int, n: int) -> list[int]:
    """Positions held after appending positions 0..n-1 in order."""
    c = StreamingCache(sink, window)
    for p in range(n):
        c.append(p)
    return c.held()
