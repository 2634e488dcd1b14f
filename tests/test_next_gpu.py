"""Rows beyond the core build: overflow diagnostics and the multi-array gather,
through the C ABI, against the CPU oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import gpu_build, to_u32
from uniform_grid_particle_gb300 import scenes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ug():
    from uniform_grid_particle_gb300 import build, ugrid

    build.build()
    return ugrid


@pytest.mark.parametrize("name", ["headline", "contention", "tiny"])
@pytest.mark.parametrize("capacidad", [1, 4, 64, 100_000])
def test_diagnostics_match_oracle(ug, oracle_lib, name, capacidad):
    s = scenes.SCENES[name]
    rows = s.particles()
    got = gpu_build(ug, rows, s.dims, s.origin, s.cell_size)
    p = ug.make_params(s.n, s.dims, s.origin, s.cell_size)
    diag = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    conteos = torch.from_numpy(got["conteos"].view(np.int32)).cuda()
    want = oracle_lib.diagnostics(oracle_lib.cell_index(rows, s.dims, s.origin, s.cell_size), s.cells, capacidad)
    for _ in range(2):  # a second call on the same diag array gives the same numbers
        ug.grid_diagnostics(conteos, diag, p, capacidad)
        assert tuple(int(v) for v in to_u32(diag)) == want


def test_diagnostics_ragged_cells(ug, oracle_lib):
    dims = (7, 11, 13)                       # 1001 cells: not a multiple of 4
    rng = np.random.default_rng(3)
    celda = rng.integers(0, 1001, 50_000, dtype=np.uint32)
    celda[:3000] = 1000                      # the last cell, in the tail of the vector loop
    conteos = np.bincount(celda, minlength=1001).astype(np.uint32)
    p = ug.make_params(celda.size, dims, (0, 0, 0), 1.0)
    diag = torch.empty(2, dtype=torch.int32, device="cuda")
    ug.grid_diagnostics(torch.from_numpy(conteos.view(np.int32)).cuda(), diag, p, 64)
    assert tuple(int(v) for v in to_u32(diag)) == oracle_lib.diagnostics(celda, 1001, 64)


def test_reorder_many_matches_oracle(ug, oracle_lib):
    s = scenes.SCENES["headline"]
    rows = s.particles()
    got = gpu_build(ug, rows, s.dims, s.origin, s.cell_size)
    ordenado = got["ordenado"]
    n = s.n
    rng = np.random.default_rng(9)
    aspecto = rng.integers(0, 2**32, (n, 8), dtype=np.uint64).astype(np.uint32)     # color, tam, semilla, _r
    wide = rng.integers(0, 2**32, (n, 12), dtype=np.uint64).astype(np.uint32)       # 48-byte records
    narrow = rng.integers(0, 2**32, (n, 4), dtype=np.uint64).astype(np.uint32)      # 16-byte records
    hosts = [rows, aspecto, wide, narrow]
    srcs = [torch.from_numpy(h).cuda() for h in hosts]
    dsts = [torch.empty_like(t) for t in srcs]
    p = ug.make_params(n, s.dims, s.origin, s.cell_size)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    ug.grid_reorder_many(torch.from_numpy(ordenado.view(np.int32)).cuda(), list(zip(srcs, dsts)), ws, p)
    assert ug.grid_status(ws) == 0
    for h, d in zip(hosts, dsts):
        want = oracle_lib.reorder_records(ordenado, h)
        assert np.array_equal(d.cpu().numpy().view(np.uint8), want.view(np.uint8))
    # the particle array matches the build's own gather
    assert np.array_equal(dsts[0].cpu().numpy().view(np.uint32), got["destino"].view(np.uint32))


# Record widths (in u32 words) of each call: the TMA form serves records of
# at most 64 bytes (128-byte slots up to 32 bytes, 256-byte slots above), the
# plain kernel wider ones.
MANY_CASES = [
    (1, [4]), (3, [4, 4]), (5, [8, 4]), (127, [4, 12]), (128, [16]), (129, [4, 4, 4, 4]),
    (4099, [12, 16]), (100_003, [4, 4]), (100_003, [8, 16, 12]), (65_536, [20, 4]),
    (20_001, [64]), (300_000, [4, 8]),
]


@pytest.mark.parametrize("n,widths", MANY_CASES)
def test_reorder_many_shapes(ug, oracle_lib, n, widths):
    rng = np.random.default_rng(n + len(widths))
    # Random stretches and stretches already in order, so that chunks take
    # both the gathered and the plain-load paths.
    ordenado = rng.permutation(n).astype(np.uint32)
    for lo in range(0, n, 4096):
        if rng.random() < 0.3:
            ordenado[lo:lo + 1000] = np.sort(ordenado[lo:lo + 1000])
    hosts = [rng.integers(0, 2**32, (n, w), dtype=np.uint64).astype(np.uint32) for w in widths]
    srcs = [torch.from_numpy(h).cuda() for h in hosts]
    dsts = [torch.full_like(t, 0x7f7f7f7f) for t in srcs]
    p = ug.make_params(n, (8, 8, 8), (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    ug.grid_reorder_many(torch.from_numpy(ordenado.view(np.int32)).cuda(), list(zip(srcs, dsts)), ws, p)
    assert ug.grid_status(ws) == 0
    for h, d in zip(hosts, dsts):
        assert np.array_equal(d.cpu().numpy(), oracle_lib.reorder_records(ordenado, h))


@pytest.mark.parametrize("widths", [[12, 16], [4, 4, 4]])
def test_reorder_many_bad_index_in_gathered_chunks(ug, oracle_lib, widths):
    """Out-of-range indices inside chunks that would otherwise be gathered by
    TMA (random order), in arrays of 48/64 and of 16 bytes: those chunks are
    copied with plain loads, the bad records skipped, the rest exact."""
    n = 70_001
    rng = np.random.default_rng(31)
    ordenado = rng.permutation(n).astype(np.uint32)
    bad = np.array([0, 4097, 33_333, n - 1])
    ordenado[bad] = n + np.arange(bad.size, dtype=np.uint32)
    hosts = [rng.integers(0, 2**32, (n, w), dtype=np.uint64).astype(np.uint32) for w in widths]
    srcs = [torch.from_numpy(h).cuda() for h in hosts]
    dsts = [torch.zeros_like(t) for t in srcs]
    p = ug.make_params(n, (8, 8, 8), (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    ug.grid_reorder_many(torch.from_numpy(ordenado.view(np.int32)).cuda(), list(zip(srcs, dsts)), ws, p)
    assert ug.grid_status(ws) == 4
    ok = np.ones(n, bool)
    ok[bad] = False
    for h, d in zip(hosts, dsts):
        got = d.cpu().numpy()
        assert (got[bad] == 0).all(), "bad records are not written"
        assert np.array_equal(got[ok], oracle_lib.reorder_records(ordenado[ok], h))


def test_reorder_many_identity_order(ug, oracle_lib):
    """An ordenado already in order: every chunk takes the plain-load copy."""
    n = 123_457
    rng = np.random.default_rng(32)
    ordenado = np.arange(n, dtype=np.uint32)
    hosts = [rng.integers(0, 2**32, (n, w), dtype=np.uint64).astype(np.uint32) for w in (4, 12)]
    srcs = [torch.from_numpy(h).cuda() for h in hosts]
    dsts = [torch.zeros_like(t) for t in srcs]
    p = ug.make_params(n, (8, 8, 8), (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    ug.grid_reorder_many(torch.from_numpy(ordenado.view(np.int32)).cuda(), list(zip(srcs, dsts)), ws, p)
    assert ug.grid_status(ws) == 0
    for h, d in zip(hosts, dsts):
        assert np.array_equal(d.cpu().numpy(), oracle_lib.reorder_records(ordenado, h))


def test_reorder_many_rejects_index_out_of_range(ug):
    n = 2000
    p = ug.make_params(n, (4, 4, 4), (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    ordenado = torch.randperm(n, device="cuda").int()
    ordenado[5] = n
    a, b = torch.randn(n, 8, device="cuda"), torch.randn(n, 4, device="cuda")
    da, db = torch.zeros_like(a), torch.zeros_like(b)
    ug.grid_reorder_many(ordenado, [(a, da), (b, db)], ws, p)
    assert ug.grid_status(ws) == 4
    assert (da[5] == 0).all() and (db[5] == 0).all()
    ok = torch.arange(n, device="cuda") != 5
    assert torch.equal(da[ok], a[ordenado[ok].long()]) and torch.equal(db[ok], b[ordenado[ok].long()])


def _density_case(ug, oracle_lib, rows, dims, origin, cs, h, order=0):
    """GPU density through both access paths against the float64 oracle.

    Tolerance: each term's fp32 error is at most a few ulps of h^2 inside
    (h^2 - r^2)^3, i.e. ~3e-7 m h^6; over ~100 terms plus the fp32 running sum
    (~100 * 2^-24 relative) that stays below 1e-4 * (rho + m_max h^6).  Terms
    whose inclusion fp32 and float64 decide differently have r^2 within a few
    ulps of h^2 and are ~1e-19 m h^6."""
    n = rows.shape[0]
    p = ug.make_params(n, dims, origin, cs, order=order)
    got = gpu_build(ug, rows, dims, origin, cs, params=p)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    inicios = torch.from_numpy(got["inicios"].view(np.int32)).cuda()
    ordenado = torch.from_numpy(got["ordenado"].view(np.int32)).cuda()
    rho_sorted = torch.empty(n, dtype=torch.float32, device="cuda")
    rho_indirect = torch.empty(n, dtype=torch.float32, device="cuda")
    ug.grid_density(torch.from_numpy(got["destino"]).cuda(), inicios, rho_sorted, ws, p, h)
    ug.grid_density(torch.from_numpy(rows).cuda(), inicios, rho_indirect, ws, p, h, ordenado=ordenado)
    assert ug.grid_status(ws) == 0
    a, b = rho_sorted.cpu().numpy(), rho_indirect.cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), "both paths add the same terms in the same order"
    ref = oracle_lib.density(rows, dims, origin, cs, got["inicios"], got["ordenado"], h, order=order)
    by_particle = np.empty(n, np.float64)
    by_particle[got["ordenado"]] = a
    scale = float(rows[:, 7].max()) * float(h) ** 6 if n else 0.0
    err = np.abs(by_particle - ref)
    assert np.all(err <= 1e-4 * (ref + scale)), f"max error {err.max()} (rho up to {ref.max()})"
    return ref


@pytest.mark.parametrize("name,h_frac", [("tiny", 1.0), ("headline", 1.0), ("headline", 0.6), ("contention", 1.0)])
def test_density_matches_oracle(ug, oracle_lib, name, h_frac):
    s = scenes.SCENES[name]
    _density_case(ug, oracle_lib, s.particles(), s.dims, s.origin, s.cell_size, s.cell_size * h_frac)


def test_density_sph_like(ug, oracle_lib):
    """~25 particles per cell and ~100 neighbours within h, on a non-cubic grid
    with particles outside the domain (clamped into the boundary cells)."""
    rng = np.random.default_rng(21)
    n, dims, cs = 200_000, (24, 20, 17), np.float32(0.5)
    origin = (np.float32(-6.0), np.float32(-5.0), np.float32(-4.25))
    lo = np.array(origin, np.float64) - 0.3
    hi = np.array(origin, np.float64) + np.array(dims) * float(cs) + 0.3
    rows = np.zeros((n, 8), np.float32)
    rows[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
    rows[:, 3] = 1.0
    rows[:, 7] = (0.5 + rng.random(n)).astype(np.float32)
    ref = _density_case(ug, oracle_lib, rows, dims, origin, cs, cs)
    assert float(np.median(ref)) > 0.0


def test_density_empty_scene(ug):
    p = ug.make_params(0, (4, 4, 4), (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    inicios = torch.zeros(65, dtype=torch.int32, device="cuda")
    ug.grid_density(None, inicios, torch.empty(0, device="cuda"), ws, p, 1.0)
    assert ug.grid_status(ws) == 0


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("h_frac", [1.0, 0.7])
def test_density_stale_grid(ug, oracle_lib, order, h_frac):
    """A grid built before the particles moved ("Construir el índice…", §La
    dispersión: the query walks the cells the grid lists).  Each particle
    walks the 27 cells around the cell of its current position, and a
    candidate counts where the grid lists it, at its current position: the
    reading the oracle follows (pinned against all pairs with that membership
    rule).  About 12 particles per cell, so the tiles serve most runs and the
    moved particles take the per-particle walk."""
    rng = np.random.default_rng(40 + order)
    dims, cs = (32, 32, 32), np.float32(0.3125)
    origin = (np.float32(-5.0), np.float32(-5.0), np.float32(-5.0))
    n = 12 * dims[0] * dims[1] * dims[2]
    lo = np.array(origin, np.float64)
    hi = lo + np.array(dims) * float(cs)
    before = np.zeros((n, 8), np.float32)
    before[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
    before[:, 3] = 1.0
    before[:, 7] = (0.5 + rng.random(n)).astype(np.float32)
    after = before.copy()
    moving = rng.random(n) < 0.3
    after[moving, :3] += (rng.uniform(-0.45, 0.45, (int(moving.sum()), 3)) * cs).astype(np.float32)
    p = ug.make_params(n, dims, origin, cs, order=order)
    got = gpu_build(ug, before, dims, origin, cs, params=p)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    inicios = torch.from_numpy(got["inicios"].view(np.int32)).cuda()
    ordenado = torch.from_numpy(got["ordenado"].view(np.int32)).cuda()
    h = float(cs) * h_frac
    rho_sorted = torch.empty(n, dtype=torch.float32, device="cuda")
    rho_indirect = torch.empty(n, dtype=torch.float32, device="cuda")
    # the records in the grid's order, at their current positions
    ug.grid_density(torch.from_numpy(after[got["ordenado"]]).cuda(), inicios, rho_sorted, ws, p, h)
    ug.grid_density(torch.from_numpy(after).cuda(), inicios, rho_indirect, ws, p, h, ordenado=ordenado)
    assert ug.grid_status(ws) == 0
    a, b = rho_sorted.cpu().numpy(), rho_indirect.cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), "both paths add the same terms in the same order"
    ref = oracle_lib.density(after, dims, origin, cs, got["inicios"], got["ordenado"], h, order=order)
    by_particle = np.empty(n, np.float64)
    by_particle[got["ordenado"]] = a
    scale = float(after[:, 7].max()) * h ** 6
    err = np.abs(by_particle - ref)
    assert np.all(err <= 1e-4 * (ref + scale)), f"max error {err.max()} (rho up to {ref.max()})"
    # the moved particles really left their cells
    now = oracle_lib.cell_index(after, dims, origin, cs, order=order)
    assert int(np.sum(now != got["celdaDe"])) > n // 20


@pytest.mark.parametrize("order", [0, 1])
def test_density_dense_cells(ug, oracle_lib, order):
    """50 particles per cell, near the top of the 20-60 per cell that
    "Contar partículas por celda" (§La contención) calls healthy, on a grid
    with power-of-two sides (so it also builds in Morton order)."""
    rng = np.random.default_rng(50 + order)
    dims, cs = (32, 32, 16), np.float32(0.25)
    origin = (np.float32(-4.0), np.float32(-4.0), np.float32(-2.0))
    n = 50 * dims[0] * dims[1] * dims[2]
    lo = np.array(origin, np.float64)
    hi = lo + np.array(dims) * float(cs)
    rows = np.zeros((n, 8), np.float32)
    rows[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
    rows[:, 3] = 1.0
    rows[:, 7] = (0.5 + rng.random(n)).astype(np.float32)
    ref = _density_case(ug, oracle_lib, rows, dims, origin, cs, cs, order=order)
    assert float(np.median(ref)) > 0.0
