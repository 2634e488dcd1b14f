"""GPU parity of the Morton (Z-curve) cell order ("Reordenar por celda y la
coalescencia de memoria", §El orden de las celdas) against the oracle built
with the same order: the fused build and the per-step entry points, cubic
grids (the shift-and-mask spread) and unequal power-of-two sides (the bit
deposit), and the neighbour density walked over a Morton grid."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_matches_oracle, gpu_build, to_u32
from test_next_gpu import _density_case
from uniform_grid_particle_gb300 import scenes

pytestmark = pytest.mark.gpu

MORTON = 1


@pytest.fixture(scope="module")
def ug():
    from uniform_grid_particle_gb300 import ugrid

    ugrid.lib()
    return ugrid


def _rows(n, dims, cs, origin, seed, margin=0.3):
    rng = np.random.default_rng(seed)
    lo = np.array(origin, np.float64) - margin
    hi = np.array(origin, np.float64) + np.array(dims) * float(cs) + margin
    rows = np.zeros((n, 8), np.float32)
    rows[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
    rows[:, 3] = 1.0
    rows[:, 7] = (0.5 + rng.random(n)).astype(np.float32)
    return rows


def _check(ug, o, rows, dims, origin, cs, stable):
    p = ug.make_params(rows.shape[0], dims, origin, cs, order=MORTON)
    flags = ug.GRID_STABLE if stable else 0
    got = gpu_build(ug, rows, dims, origin, cs, flags, params=p)
    ref = o.build(rows, dims, origin, cs, order=MORTON)
    assert_matches_oracle(o, rows, got, ref, stable)
    return got, ref


@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
@pytest.mark.parametrize("name", ["tiny", "headline", "contention"])
def test_scene_build_morton(ug, oracle_lib, name, stable):
    s = scenes.SCENES[name]
    _check(ug, oracle_lib, s.particles(), s.dims, s.origin, s.cell_size, stable)


UNEQUAL = [
    (50_000, (8, 32, 4)),
    (16_385, (64, 2, 16)),
    (33, (1, 1, 1)),
    (1, (2, 2, 2)),
    (100_000, (1, 1, 1024)),
    (200_000, (256, 128, 64)),
    (70_000, (2048, 2, 1)),
]


@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
@pytest.mark.parametrize("n,dims", UNEQUAL, ids=[f"{n}-{d[0]}x{d[1]}x{d[2]}" for n, d in UNEQUAL])
def test_unequal_sides(ug, oracle_lib, n, dims, stable):
    cs = np.float32(0.25)
    origin = (np.float32(-1.0), np.float32(0.5), np.float32(2.0))
    _check(ug, oracle_lib, _rows(n, dims, cs, origin, seed=n + dims[0]), dims, origin, cs, stable)


def test_largest_cubic_spread(ug, oracle_lib):
    """1024^3 cells: the widest grid the ten-bit spread serves."""
    dims, cs, origin = (1024, 1024, 1024), np.float32(1.0 / 64), (np.float32(-8.0),) * 3
    _check(ug, oracle_lib, _rows(300_000, dims, cs, origin, seed=3, margin=0.05), dims, origin, cs, False)


def test_morton_count_entry_point(ug, oracle_lib):
    """grid_count alone writes celdaDe and conteos in Morton order."""
    s = scenes.SCENES["headline"]
    rows = s.particles()
    p = ug.make_params(s.n, s.dims, s.origin, s.cell_size, order=MORTON)
    ref = oracle_lib.build(rows, s.dims, s.origin, s.cell_size, order=MORTON)
    conteos = torch.zeros(s.cells, dtype=torch.int32, device="cuda")
    celda = torch.empty(s.n, dtype=torch.int32, device="cuda")
    ug.grid_count(torch.from_numpy(rows).cuda(), conteos, celda, p)
    assert np.array_equal(to_u32(celda), ref["celdaDe"])
    assert np.array_equal(to_u32(conteos), ref["conteos"])


def test_morton_is_a_relabelling_of_linear(ug):
    """On the device too, the Morton build holds the linear build's cells
    under new labels: same counts, same members (stable mode)."""
    s = scenes.SCENES["headline"]
    rows = s.particles()
    lin = gpu_build(ug, rows, s.dims, s.origin, s.cell_size, ug.GRID_STABLE)
    p = ug.make_params(s.n, s.dims, s.origin, s.cell_size, order=MORTON)
    mor = gpu_build(ug, rows, s.dims, s.origin, s.cell_size, ug.GRID_STABLE, params=p)
    # cell of each particle in both labellings gives the relabelling
    relabel = np.full(s.cells, -1, np.int64)
    relabel[lin["celdaDe"]] = mor["celdaDe"]
    occupied = lin["conteos"] > 0
    assert np.array_equal(mor["conteos"][relabel[occupied]], lin["conteos"][occupied])
    assert int(mor["conteos"].sum()) == s.n
    for c in np.nonzero(occupied)[0][:: max(1, occupied.sum() // 2000)]:
        a = lin["ordenado"][lin["inicios"][c]:lin["inicios"][c + 1]]
        m = relabel[c]
        b = mor["ordenado"][mor["inicios"][m]:mor["inicios"][m + 1]]
        assert np.array_equal(a, b)


@pytest.mark.parametrize("name,h_frac", [("tiny", 1.0), ("headline", 1.0), ("headline", 0.6)])
def test_density_morton(ug, oracle_lib, name, h_frac):
    s = scenes.SCENES[name]
    _density_case(ug, oracle_lib, s.particles(), s.dims, s.origin, s.cell_size, s.cell_size * h_frac, order=MORTON)


def test_density_morton_unequal_sides(ug, oracle_lib):
    """~25 particles per cell on a 32x16x8 grid (the deposit path), with
    particles beyond the domain clamped into the boundary cells."""
    dims, cs = (32, 16, 8), np.float32(0.5)
    origin = (np.float32(-6.0), np.float32(-5.0), np.float32(-4.25))
    rows = _rows(100_000, dims, cs, origin, seed=22)
    _density_case(ug, oracle_lib, rows, dims, origin, cs, cs, order=MORTON)
