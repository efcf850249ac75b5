"""Host-side pieces of the benchmark that need no GPU."""

import pytest

import bench


@pytest.mark.parametrize("layers", [1, 2, 5, 21, 32, 100])
def test_copy_runs_cover_the_layers_in_order(layers):
    runs = bench.copy_runs(layers)
    assert runs[0] == (0, 1)
    assert runs[-1][1] == layers
    for (a, b), (c, _) in zip(runs, runs[1:]):
        assert b == c and a < b
    # each full run is four times the one before it
    sizes = [b - a for a, b in runs]
    for s0, s1 in zip(sizes[:-2], sizes[1:-1]):
        assert s1 == 4 * s0


def test_copy_runs_of_the_llama_step():
    assert bench.copy_runs(32) == [(0, 1), (1, 5), (5, 21), (21, 32)]
