"""Host-side arithmetic of bench.py that feeds reported numbers (no GPU)."""
import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_pair_tests_counts_the_27_cells():
    """The neighbour query's work: for every particle, the particles of the
    cells around its own (clipped at the grid's faces), by brute force."""
    bench = _bench()
    rng = np.random.default_rng(3)
    for dims in ((5, 4, 3), (1, 1, 1), (7, 1, 2)):
        gx, gy, gz = dims
        c = rng.integers(0, 5, size=gx * gy * gz).astype(np.uint32)
        want = 0
        for z in range(gz):
            for y in range(gy):
                for x in range(gx):
                    around = sum(int(c[X + gx * (Y + gy * Z)])
                                 for Z in range(z - 1, z + 2) for Y in range(y - 1, y + 2) for X in range(x - 1, x + 2)
                                 if 0 <= X < gx and 0 <= Y < gy and 0 <= Z < gz)
                    want += int(c[x + gx * (y + gy * z)]) * around
        assert bench.pair_tests(c, dims) == want, dims
