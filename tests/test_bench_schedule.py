"""The bench's graph schedule (host logic, no GPU): exactly --steps steps are
replayed, and step i uses weight copy i mod copies however many steps one
graph holds."""
from __future__ import annotations

import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def expand(schedule, S, copies):
    """The weight copy of every step the schedule runs, in order."""
    steps = []
    for kind, c in schedule:
        if kind == "multi":
            steps += [(c * S + s) % copies for s in range(S)]
        else:
            steps.append(c)
    return steps


@pytest.mark.parametrize("n", [0, 1, 3, 9, 10, 11, 29, 50, 3000, 3001])
@pytest.mark.parametrize("S", [1, 2, 3, 10])
@pytest.mark.parametrize("copies", [1, 3])
def test_graph_schedule_runs_exactly_n_steps_in_copy_order(n, S, copies):
    sched = bench.graph_schedule(n, S, copies)
    assert expand(sched, S, copies) == [i % copies for i in range(n)]
    assert sum(1 for kind, _ in sched if kind == "multi") == (n // S if S > 1 else 0)
