"""GPU parity on seeded random shapes: particle counts from 1 to 400,000 on a
log scale, grids of any sides (up to 4 M cells), both cell orders where the
sides allow Morton, both build modes, positions spread over the grid and
somewhat past it (clamped), and a share of the particles crowded into a few
cells.  Each case goes through grid_build, so every plan it chooses (cluster,
one-CTA, sparse, bucketed, fused) meets cases near its limits; all are
compared element by element with the oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_matches_oracle, gpu_build

pytestmark = pytest.mark.gpu

CASES = 200


@pytest.fixture(scope="module")
def ug():
    from uniform_grid_particle_gb300 import build, ugrid

    build.build()
    assert torch.cuda.is_available()
    return ugrid


def _case(seed: int):
    rng = np.random.default_rng(1000 + seed)
    n = int(np.exp(rng.uniform(0.0, np.log(400_000))))
    morton = rng.random() < 0.3
    if morton:
        dims = tuple(int(2 ** rng.integers(0, 8)) for _ in range(3))
    else:
        dims = tuple(int(np.exp(rng.uniform(0.0, np.log(300)))) for _ in range(3))
    while dims[0] * dims[1] * dims[2] > 4_000_000:
        dims = tuple(max(1, d // 2) for d in dims)
    cs = np.float32(rng.uniform(0.01, 0.5))
    origin = tuple(np.float32(v) for v in rng.uniform(-3.0, 3.0, 3))
    lo = np.array(origin, np.float64) - float(cs)
    hi = np.array(origin, np.float64) + np.array(dims) * float(cs) + float(cs)
    rows = np.zeros((n, 8), np.float32)
    rows[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
    rows[:, 3:] = rng.random((n, 5)).astype(np.float32)
    crowd = int(n * rng.uniform(0.0, 0.3)) if rng.random() < 0.5 else 0
    if crowd:
        spots = rng.integers(0, n, size=3)
        pick = rng.integers(0, n, size=crowd)
        rows[pick, :3] = rows[spots[rng.integers(0, 3, size=crowd)], :3]
    stable = bool(rng.random() < 0.5)
    return n, dims, origin, cs, rows, stable, 1 if morton else 0


@pytest.mark.parametrize("seed", range(CASES))
def test_random_shape(ug, oracle_lib, seed):
    n, dims, origin, cs, rows, stable, order = _case(seed)
    p = ug.make_params(n, dims, origin, cs, order=order)
    got = gpu_build(ug, rows, dims, origin, cs, ug.GRID_STABLE if stable else 0, params=p)
    ref = oracle_lib.build(rows, dims, origin, cs, order=order)
    assert_matches_oracle(oracle_lib, rows, got, ref, stable)


@pytest.mark.parametrize("seed", range(0, CASES, 4))
def test_random_shape_phase_by_phase(ug, oracle_lib, seed):
    """The pages' chain one entry point at a time (clear, count, scan,
    scatter in both modes, reorder) on the same random shapes."""
    o = oracle_lib
    n, dims, origin, cs, rows, _, order = _case(seed)
    C = dims[0] * dims[1] * dims[2]
    p = ug.make_params(n, dims, origin, cs, order=order)
    ref = o.build(rows, dims, origin, cs, order=order)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()  # noqa: E731
    u32 = lambda t: t.cpu().numpy().view(np.uint32)  # noqa: E731
    origen = torch.from_numpy(rows).cuda()
    ws = torch.zeros(ug.grid_workspace_bytes(p, ug.GRID_STABLE), dtype=torch.uint8, device="cuda")

    conteos = torch.full((C,), 5, dtype=torch.int32, device="cuda")
    celda = torch.empty(n, dtype=torch.int32, device="cuda")
    ug.grid_clear(conteos, p)
    ug.grid_count(origen, conteos, celda, p)
    assert np.array_equal(u32(celda), ref["celdaDe"])
    assert np.array_equal(u32(conteos), ref["conteos"])

    inicios = torch.empty(C + 1, dtype=torch.int32, device="cuda")
    ug.grid_scan(conteos, inicios, ws, p)
    assert ug.grid_status(ws) == 0
    assert np.array_equal(u32(inicios), ref["inicios"])

    cursor = torch.zeros(C, dtype=torch.int32, device="cuda")
    ordenado = torch.empty(n, dtype=torch.int32, device="cuda")
    ug.grid_scatter(celda, inicios, cursor, ordenado, ws, p)
    assert ug.grid_status(ws) == 0
    assert np.array_equal(u32(cursor), ref["conteos"])
    assert np.array_equal(o.canonicalise(ref["inicios"], u32(ordenado)), ref["ordenado"])
    cursor.zero_()
    ug.grid_scatter(celda, inicios, cursor, ordenado, ws, p, flags=ug.GRID_STABLE)
    assert ug.grid_status(ws) == 0
    assert np.array_equal(u32(ordenado), ref["ordenado"])

    destino = torch.empty_like(origen)
    ug.grid_reorder(ordenado, origen, destino, ws, p)
    assert ug.grid_status(ws) == 0
    assert np.array_equal(destino.cpu().numpy().view(np.uint32), ref["destino"].view(np.uint32))
