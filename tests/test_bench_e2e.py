"""bench.py's end-to-end loop with two steps in flight (CPU, fake CUDA streams).

Every step uploads its inputs, runs the library and downloads its result.
With two buffer slots, step i's upload may not overwrite slot i % 2 before
step i - 2's compute has read it, and step i's compute may not overwrite the
slot's result before step i - 2's download has read it.  The fakes record
every wait and record in program order, so the test checks exactly these
dependencies and that each operation runs on its own stream.
"""
import contextlib
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class FakeEvent:
    n = 0

    def __init__(self, enable_timing=False):
        FakeEvent.n += 1
        self.id = FakeEvent.n
        self.recorded_by = None  # the op label this event marks

    def record(self, stream=None):
        log.append(("record", self.id, stream.name))
        self.recorded_by = current_op[0]

    def elapsed_time(self, other):
        return 1.0


class FakeStream:
    def __init__(self, name=None):
        FakeStream.count = getattr(FakeStream, "count", 0) + 1
        self.name = name or f"side{FakeStream.count}"

    def wait_event(self, ev):
        log.append(("wait", self.name, ev.recorded_by))


log = []
current_op = [None]
current_stream = [None]


def test_two_steps_in_flight_order(monkeypatch):
    log.clear()
    monkeypatch.setattr(torch.cuda, "Stream", lambda: FakeStream())
    monkeypatch.setattr(torch.cuda, "Event", FakeEvent)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda: None)

    @contextlib.contextmanager
    def on(stream):
        prev = current_stream[0]
        current_stream[0] = stream
        yield
        current_stream[0] = prev

    monkeypatch.setattr(torch.cuda, "stream", on)
    ops = []

    def op(kind):
        def f(sl):
            i = sum(1 for o in ops if o[0] == kind)
            ops.append((kind, i, sl, current_stream[0].name))
            current_op[0] = (kind, i)
        return f

    main = FakeStream("main")
    n = 6
    ms = bench.pipelined_e2e(n, op("up"), op("compute"), op("down"), main)
    assert ms == 1.0 / n
    # every step ran all three operations, on three distinct streams, slots alternating
    for kind in ("up", "compute", "down"):
        steps = [o for o in ops if o[0] == kind]
        assert [o[1] for o in steps] == list(range(n))
        assert [o[2] for o in steps] == [i % 2 for i in range(n)]
    streams = {kind: {o[3] for o in ops if o[0] == kind} for kind in ("up", "compute", "down")}
    assert streams["compute"] == {"main"}
    assert len(streams["up"] | streams["down"] | streams["compute"]) == 3
    # the waits: the stream of each op waits on the events that order it
    waits = [(w[1], w[2]) for w in log if w[0] == "wait"]
    up_s, down_s = streams["up"].pop(), streams["down"].pop()
    for i in range(n):
        assert ("main", ("up", i)) in waits                  # compute i after upload i
        assert (down_s, ("compute", i)) in waits             # download i after compute i
        if i >= 2:
            assert (up_s, ("compute", i - 2)) in waits       # slot inputs free again
            assert ("main", ("down", i - 2)) in waits        # slot result read
    # no upload waits on a compute it does not overwrite
    assert (up_s, ("compute", n - 1)) not in waits
