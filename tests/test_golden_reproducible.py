"""The stored golden rows (tests/golden/) are what the oracle computes from the seeded
generator now: two small sweep points are regenerated with the committed script's own
code path and must match the stored text line for line (sums of squares and norms in
hex).  A change to the oracle's arithmetic, the generator or a workload recipe that is
not followed by regenerating the files fails here."""
import pytest

from synth import workloads as W
from tests.golden import make_golden as golden


@pytest.mark.parametrize("point", [(1 << 20, 2, 2), ((1 << 20) + 1, 16, 2)])
def test_golden_rows_reproduce(point):
    name = W.sweep_name(*point)
    with open(golden.golden_path(name), encoding="utf-8") as f:
        stored = [line.strip() for line in f if line.strip() and not line.startswith("#")]
    assert len(stored) == W.by_name(name).steps >= 2
    assert golden.golden_rows(name, procs=2) == stored
