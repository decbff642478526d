"""The 8-lane reduce-scatter of the Gated DeltaNet scan, restated on the CPU
(no GPU): each of a row's 8 threads holds partial output dots of 8 tokens;
three butterfly steps (exchange with the lanes 4, 2 and 1 apart, keeping the
upper or lower half of the remaining tokens by that lane bit) leave lane L
with the full sum for token L."""
import numpy as np


def reduce_scatter(po):
    """po [8 lanes][8 tokens] -> [8 lanes], statement by statement as in the
    kernel: in the step with lane distance d (4, 2, 1) and h = d remaining
    tokens kept, lane tc sends po[i] if (tc & d) else po[i + h], keeps
    po[i + h] if (tc & d) else po[i], and adds what its partner tc ^ d sent."""
    po = [list(row) for row in po]
    for d in (4, 2, 1):
        h = d
        send = [[row[i] if (tc & d) else row[i + h] for i in range(h)] for tc, row in enumerate(po)]
        keep = [[row[i + h] if (tc & d) else row[i] for i in range(h)] for tc, row in enumerate(po)]
        po = [[keep[tc][i] + send[tc ^ d][i] for i in range(h)] for tc in range(8)]
    return [row[0] for row in po]


def test_reduce_scatter_gives_each_lane_its_token():
    rng = np.random.default_rng(3)
    for _ in range(20):
        po = rng.integers(-1000, 1000, size=(8, 8))   # integers: exact sums
        got = reduce_scatter(po.tolist())
        assert got == po.sum(axis=0).tolist()
