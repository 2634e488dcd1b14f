"""CUDA path (through the C ABI) against the CPU oracle, element by element."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_matches_oracle, gpu_build, special_rows, to_u32
from uniform_grid_particle_gb300 import scenes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ug():
    from uniform_grid_particle_gb300 import build, ugrid

    build.build()
    assert torch.cuda.is_available()
    return ugrid


def _check(ug, o, rows, dims, origin, cs, stable):
    flags = ug.GRID_STABLE if stable else 0
    got = gpu_build(ug, rows, dims, origin, cs, flags)
    ref = o.build(rows, dims, origin, cs)
    assert_matches_oracle(o, rows, got, ref, stable)
    return got


# ---------------------------------------------------------------- the workloads

@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
@pytest.mark.parametrize("name", ["tiny", "scan_dominated", "headline", "contention", "stress"])
def test_scene_build(ug, oracle_lib, name, stable):
    s = scenes.SCENES[name]
    rows = s.particles()
    _check(ug, oracle_lib, rows, s.dims, s.origin, s.cell_size, stable)


def test_contention_unshuffled(ug, oracle_lib):
    rows = scenes.contention_particles(1_000_000, 99, 128, shuffle=False)
    _check(ug, oracle_lib, rows, (128,) * 3, (-5.0,) * 3, 0.078125, False)
    _check(ug, oracle_lib, rows, (128,) * 3, (-5.0,) * 3, 0.078125, True)


# ---------------------------------------------------------------- ragged shapes

RAGGED = [(1, (17, 19, 23)), (33, (17, 19, 23)), (1023, (5, 3, 2)), (1025, (17, 19, 23)),
          (4096 * 3 + 77, (17, 19, 23)), (100_003, (31, 7, 61)), (65_537, (1, 1, 1)),
          (250_000, (64, 1, 9))]


@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
@pytest.mark.parametrize("n,dims", RAGGED, ids=[f"{n}-{d[0]}x{d[1]}x{d[2]}" for n, d in RAGGED])
def test_ragged(ug, oracle_lib, n, dims, stable):
    origin = (np.float32(-1.3), np.float32(2.2), np.float32(0.7))
    cs = np.float32(0.37)
    rng = np.random.default_rng(n)
    lo = np.array(origin, np.float64) - 0.5
    hi = np.array(origin, np.float64) + np.array(dims) * float(cs) + 0.5
    rows = np.zeros((n, 8), np.float32)
    rows[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
    rows[:, 3:] = rng.random((n, 5)).astype(np.float32)
    _check(ug, oracle_lib, rows, dims, origin, cs, stable)


# ---------------------------------------------------------------- small scenes (one-CTA build)

SMALL = [(8192, (32, 16, 16)), (8193, (32, 16, 16)), (8192, (3, 2731, 1)), (5000, (20, 20, 20)),
         (7, (1, 1, 1)), (8192, (1, 1, 1)), (3000, (7, 5, 3))]


@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
@pytest.mark.parametrize("n,dims", SMALL, ids=[f"{n}-{d[0]}x{d[1]}x{d[2]}" for n, d in SMALL])
def test_small_scene_limits(ug, oracle_lib, n, dims, stable):
    """Scenes at, just past and far inside the one-CTA build's limits (8192
    particles, 8192 cells): 8192 cells, 8193 particles, 8193 cells, a cell
    count that is not a multiple of eight, every particle in one cell."""
    origin = (np.float32(-0.9), np.float32(0.4), np.float32(-2.1))
    cs = np.float32(0.25)
    rng = np.random.default_rng(n + dims[0])
    lo = np.array(origin, np.float64) - 0.3
    hi = np.array(origin, np.float64) + np.array(dims) * float(cs) + 0.3
    rows = np.zeros((n, 8), np.float32)
    rows[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
    rows[:, 3:] = rng.random((n, 5)).astype(np.float32)
    _check(ug, oracle_lib, rows, dims, origin, cs, stable)


CLUSTER = [(32_768, (64, 64, 32)), (32_769, (64, 64, 32)), (30_000, (50, 50, 50)), (20_000, (128, 1000, 1)),
           (12_345, (131_073, 1, 1)), (20_000, (16, 16, 16))]


@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
@pytest.mark.parametrize("n,dims", CLUSTER, ids=[f"{n}-{d[0]}x{d[1]}x{d[2]}" for n, d in CLUSTER])
def test_cluster_scene_limits(ug, oracle_lib, n, dims, stable):
    """Scenes at and just past the cluster build's limits (32,768 particles,
    131,072 cells), and inside them."""
    origin = (np.float32(-0.5), np.float32(-0.25), np.float32(0.0))
    cs = np.float32(0.125)
    rng = np.random.default_rng(n + dims[1])
    lo = np.array(origin, np.float64) - 0.2
    hi = np.array(origin, np.float64) + np.array(dims) * float(cs) + 0.2
    rows = np.zeros((n, 8), np.float32)
    rows[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
    rows[:, 3:] = rng.random((n, 5)).astype(np.float32)
    _check(ug, oracle_lib, rows, dims, origin, cs, stable)


@pytest.mark.parametrize("n", [8192, 32_768])
def test_cluster_scene_one_cell(ug, oracle_lib, n):
    """Every particle on one cell of a small grid: the cluster build's warps
    take their slots with one remote atomic per warp."""
    rows = scenes.single_cell_particles(n, 9, (0.3, 0.3, 0.3))
    for stable in (False, True):
        got = _check(ug, oracle_lib, rows, (16,) * 3, (-5.0,) * 3, 0.625, stable)
        if stable:
            assert np.array_equal(got["ordenado"], np.arange(n, dtype=np.uint32))


@pytest.mark.parametrize("crowd", [33, 1024, 1025, 6000])
def test_small_scene_long_segments(ug, oracle_lib, crowd):
    """A small scene with one crowded cell among scattered particles: the
    one-CTA build's stable mode sorts segments longer than 32 with the whole
    CTA."""
    rng = np.random.default_rng(crowd)
    base = scenes.uniform_particles(8000 - crowd, 41)
    rows = np.concatenate([base, base[:crowd].copy()])
    rows[-crowd:, :3] = np.float32(0.1)
    rows = rows[rng.permutation(rows.shape[0])]
    for stable in (True, False):
        _check(ug, oracle_lib, rows, (16,) * 3, (-5.0,) * 3, 0.625, stable)


# ---------------------------------------------------------------- sparse grids (single-barrier build)

SPARSE = [(5_000, (97, 89, 13)), (20_000, (256, 256, 3)), (100_000, (128, 128, 128)),
          (200_000, (256, 256, 256)), (250_000, (1024, 1024, 3)), (300_001, (512, 512, 9)),
          (9_000, (200, 100, 50))]


@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
@pytest.mark.parametrize("n,dims", SPARSE, ids=[f"{n}-{d[0]}x{d[1]}x{d[2]}" for n, d in SPARSE])
def test_sparse_grids(ug, oracle_lib, n, dims, stable):
    """At least four cells per particle: buckets of one window and of several
    (256^3 over the CTAs is about 55,000 cells a bucket, 1024 x 1024 x 3 about
    10,000), ragged sides."""
    origin = (np.float32(-3.1), np.float32(0.6), np.float32(-0.2))
    cs = np.float32(0.05)
    rng = np.random.default_rng(n + 7)
    lo = np.array(origin, np.float64) - 0.2
    hi = np.array(origin, np.float64) + np.array(dims) * float(cs) + 0.2
    rows = np.zeros((n, 8), np.float32)
    rows[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
    rows[:, 3:] = rng.random((n, 5)).astype(np.float32)
    _check(ug, oracle_lib, rows, dims, origin, cs, stable)


@pytest.mark.parametrize("crowd", [5_000, 12_000, 40_000])
def test_sparse_grid_crowded_bucket(ug, oracle_lib, crowd):
    """A sparse grid whose crowded cell puts more particles in one bucket than
    a CTA holds: that bucket streams its pairs (and, in stable mode, sorts the
    crowded segment in shared memory or by radix)."""
    rng = np.random.default_rng(crowd)
    base = scenes.uniform_particles(100_000 - crowd, 43)
    rows = np.concatenate([base, base[:crowd].copy()])
    rows[-crowd:, :3] = np.float32(1.01)
    rows[-crowd // 3:, :3] = np.float32(1.09)  # a second crowded cell next to it
    rows = rows[rng.permutation(rows.shape[0])]
    for stable in (True, False):
        _check(ug, oracle_lib, rows, (128,) * 3, (-5.0,) * 3, 0.078125, stable)


def test_sparse_grid_morton(ug, oracle_lib):
    rows = scenes.uniform_particles(150_000, 47)
    p = ug.make_params(rows.shape[0], (128,) * 3, (-5.0,) * 3, 0.078125, order=ug.GRID_ORDER_MORTON)
    ref = oracle_lib.build(rows, (128,) * 3, (-5.0,) * 3, 0.078125, order=1)
    for stable in (False, True):
        got = gpu_build(ug, rows, (128,) * 3, (-5.0,) * 3, 0.078125, ug.GRID_STABLE if stable else 0, params=p)
        assert_matches_oracle(oracle_lib, rows, got, ref, stable)


# ---------------------------------------------------------------- cell-index edge cases

@pytest.mark.parametrize("dims,cs", [((16,) * 3, 0.625), ((128,) * 3, 0.078125), ((256,) * 3, 0.0390625),
                                     ((37, 11, 5), 0.1), ((9, 40, 13), 0.3)])
def test_faces_ulps_and_specials(ug, oracle_lib, dims, cs):
    origin = (np.float32(-5.0), np.float32(-1.7), np.float32(3.3))
    rows = special_rows(dims, origin, np.float32(cs), seed=dims[0])
    _check(ug, oracle_lib, rows, dims, origin, np.float32(cs), False)


# ---------------------------------------------------------------- degenerate cases

def test_empty_scene(ug, oracle_lib):
    rows = np.zeros((0, 8), np.float32)
    got = gpu_build(ug, rows, (8, 8, 8), (0, 0, 0), 1.0)
    assert got["status"] == 0
    assert not got["conteos"].any() and not got["inicios"].any() and got["inicios"].size == 513


def test_single_cell_grid(ug, oracle_lib):
    rows = scenes.uniform_particles(70_001, 3)
    _check(ug, oracle_lib, rows, (1, 1, 1), (-5, -5, -5), 10.0, False)
    _check(ug, oracle_lib, rows, (1, 1, 1), (-5, -5, -5), 10.0, True)


@pytest.mark.parametrize("n", [2, 33, 10_000, 16_384, 16_385, 1_000_000])
def test_all_particles_in_one_cell(ug, oracle_lib, n):
    """Every particle on one cell centre: maximal contention, one long segment
    (register, shared-memory and radix tiers of the stable sort)."""
    rows = scenes.single_cell_particles(n, 5, (0.0390625,) * 3)
    got = _check(ug, oracle_lib, rows, (128,) * 3, (-5.0,) * 3, 0.078125, True)
    assert np.array_equal(got["ordenado"], np.arange(n, dtype=np.uint32))
    _check(ug, oracle_lib, rows, (128,) * 3, (-5.0,) * 3, 0.078125, False)


def test_large_grid(ug, oracle_lib):
    """512^3 cells: 32768 scan tiles in one look-back chain."""
    rows = scenes.uniform_particles(2_000_000, 17)
    _check(ug, oracle_lib, rows, (512,) * 3, (-5.0,) * 3, np.float32(10 / 512), False)


def test_stable_mode_is_deterministic(ug, oracle_lib):
    s = scenes.SCENES["contention"]
    rows = s.particles()
    a = gpu_build(ug, rows, s.dims, s.origin, s.cell_size, ug.GRID_STABLE)
    b = gpu_build(ug, rows, s.dims, s.origin, s.cell_size, ug.GRID_STABLE)
    assert np.array_equal(a["ordenado"], b["ordenado"])
    assert np.array_equal(a["destino"].view(np.uint32), b["destino"].view(np.uint32))


@pytest.mark.parametrize("crowd", [33, 200, 2000], ids=["crowd33", "crowd200", "crowd2000"])
def test_stable_crowded_cell_inside_a_bucket(ug, oracle_lib, crowd):
    """A cell of more than 32 particles whose bucket still fits one CTA: the
    bucketed build sorts that segment with the CTA's shared-memory bitonic
    sort (shorter ones in registers).  The crowd is interleaved with the rest
    so its particle indices are scattered."""
    rng = np.random.default_rng(crowd)
    base = scenes.uniform_particles(100_000, 31)
    rows = np.concatenate([base, base[:crowd].copy()])
    rows[-crowd:, :3] = np.float32(0.01)  # all in the cell holding (0.01, 0.01, 0.01)
    rows = rows[rng.permutation(rows.shape[0])]
    for stable in (True, False):
        _check(ug, oracle_lib, rows, (128,) * 3, (-5.0,) * 3, 0.078125, stable)


@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
@pytest.mark.parametrize("name", ["headline", "scan_dominated", "contention"])
def test_input_already_in_cell_order(ug, oracle_lib, name, stable):
    """A second build from the first build's destino: equal keys arrive in
    runs, which takes the shared-memory counters' run-length path."""
    s = scenes.SCENES[name]
    first = gpu_build(ug, s.particles(), s.dims, s.origin, s.cell_size)
    rows = np.ascontiguousarray(first["destino"])
    _check(ug, oracle_lib, rows, s.dims, s.origin, s.cell_size, stable)


def test_one_workspace_for_many_sizes(ug, oracle_lib):
    """A workspace sized for the largest call serves smaller ones (fewer
    particles, fewer cells, stable or not) in any order: the arrays that must
    be zero between calls sit where every size finds them."""
    big = ug.make_params(1_000_000, (128,) * 3, (-5.0,) * 3, 0.078125)
    ws = torch.zeros(ug.grid_workspace_bytes(big, ug.GRID_STABLE), dtype=torch.uint8, device="cuda")
    cases = [
        (1_000_000, (128,) * 3, 0, 1), (300_000, (128,) * 3, 0, 2), (1_000_000, (128,) * 3, ug.GRID_STABLE, 3),
        (50_000, (64,) * 3, 0, 4), (1_000_000, (16,) * 3, 0, 5), (777_777, (100, 128, 90), ug.GRID_STABLE, 6),
        (1_000_000, (128,) * 3, 0, 7),
    ]
    for n, dims, flags, seed in cases:
        cs = np.float32(10.0 / dims[0])
        rows = scenes.uniform_particles(n, 1000 + seed)
        p = ug.make_params(n, dims, (-5.0,) * 3, cs)
        b = ug.GridBuffers.allocate(p, flags)
        b.ws = ws
        got = gpu_build(ug, rows, dims, (-5.0,) * 3, cs, flags, bufs=b, params=p)
        ref = oracle_lib.build(rows, dims, (-5.0,) * 3, cs)
        assert_matches_oracle(oracle_lib, rows, got, ref, flags != 0)


@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
def test_build_from_host_memory(ug, oracle_lib, stable):
    """grid_build_host: pinned host records in, destino and inicios back in
    pinned host memory, all on one stream."""
    s = scenes.SCENES["headline"]
    rows = s.particles()
    flags = ug.GRID_STABLE if stable else 0
    p = ug.make_params(s.n, s.dims, s.origin, s.cell_size)
    b = ug.GridBuffers.allocate(p, flags)
    host_in = torch.from_numpy(rows).pin_memory()
    host_dest = torch.empty((s.n, 8), dtype=torch.float32).pin_memory()
    host_inicios = torch.empty(s.cells + 1, dtype=torch.int32).pin_memory()
    dev_in = torch.empty((s.n, 8), dtype=torch.float32, device="cuda")
    ug.grid_build_host(host_in, host_dest, host_inicios, dev_in, b.destino, b.conteos, b.celdaDe, b.inicios,
                       b.ordenado, b.ws, p, flags)
    torch.cuda.synchronize()
    got = {"status": ug.grid_status(b.ws), "conteos": to_u32(b.conteos), "celdaDe": to_u32(b.celdaDe),
           "inicios": host_inicios.numpy().view(np.uint32), "ordenado": to_u32(b.ordenado),
           "destino": host_dest.numpy()}
    assert_matches_oracle(oracle_lib, rows, got, oracle_lib.build(rows, s.dims, s.origin, s.cell_size), stable)


# ---------------------------------------------------------------- one entry point at a time

def test_phases_one_by_one(ug, oracle_lib):
    o = oracle_lib
    s = scenes.SCENES["headline"]
    rows = s.particles()
    n, dims, C = s.n, s.dims, s.cells
    p = ug.make_params(n, dims, s.origin, s.cell_size)
    ref = o.build(rows, dims, s.origin, s.cell_size)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()  # noqa: E731
    origen = torch.from_numpy(rows).cuda()
    ws = torch.zeros(ug.grid_workspace_bytes(p, ug.GRID_STABLE), dtype=torch.uint8, device="cuda")

    conteos = torch.full((C,), 7, dtype=torch.int32, device="cuda")
    celda = torch.empty(n, dtype=torch.int32, device="cuda")
    ug.grid_clear(conteos, p)
    assert not conteos.any()
    ug.grid_count(origen, conteos, celda, p)
    assert np.array_equal(to_u32(celda), ref["celdaDe"])
    assert np.array_equal(to_u32(conteos), ref["conteos"])

    inicios = torch.empty(C + 1, dtype=torch.int32, device="cuda")
    ug.grid_scan(dev(ref["conteos"]), inicios, ws, p)
    assert np.array_equal(to_u32(inicios), ref["inicios"])

    cursor = torch.zeros(C, dtype=torch.int32, device="cuda")
    ordenado = torch.empty(n, dtype=torch.int32, device="cuda")
    ug.grid_scatter(dev(ref["celdaDe"]), dev(ref["inicios"]), cursor, ordenado, ws, p)
    assert ug.grid_status(ws) == 0
    assert np.array_equal(to_u32(cursor), ref["conteos"]), "cursor ends at the histogram"
    assert np.array_equal(o.canonicalise(ref["inicios"], to_u32(ordenado)), ref["ordenado"])

    cursor.zero_()
    ug.grid_scatter(dev(ref["celdaDe"]), dev(ref["inicios"]), cursor, ordenado, ws, p, flags=ug.GRID_STABLE)
    assert ug.grid_status(ws) == 0
    assert np.array_equal(to_u32(ordenado), ref["ordenado"])

    destino = torch.empty_like(origen)
    ug.grid_reorder(dev(ref["ordenado"]), origen, destino, ws, p)
    assert ug.grid_status(ws) == 0
    assert np.array_equal(destino.cpu().numpy().view(np.uint32), ref["destino"].view(np.uint32))


@pytest.mark.parametrize("n", [1, 3, 127, 128, 129, 1023, 4097, 131073, 1_000_003])
def test_reorder_sizes(ug, oracle_lib, n):
    """grid_reorder alone over ragged sizes (partial chunks of 128 records,
    partial groups of four) and an index list with repeats, against the
    oracle's gather."""
    rng = np.random.default_rng(n)
    rows = rng.standard_normal((n, 8)).astype(np.float32)
    ordenado = rng.permutation(n).astype(np.uint32)
    if n > 10:
        ordenado[rng.integers(0, n, n // 10)] = rng.integers(0, n, n // 10)  # some indices repeat
    p = ug.make_params(n, (4, 4, 4), (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    origen = torch.from_numpy(rows).cuda()
    destino = torch.full_like(origen, float("nan"))
    ug.grid_reorder(torch.from_numpy(ordenado.view(np.int32)).cuda(), origen, destino, ws, p)
    torch.cuda.synchronize()
    assert ug.grid_status(ws) == 0
    assert np.array_equal(destino.cpu().numpy().view(np.uint32), oracle_lib.reorder(ordenado, rows).view(np.uint32))


@pytest.mark.parametrize("n", [1, 129, 4096, 1_000_003])
def test_reorder_runs(ug, oracle_lib, n):
    """An ordenado made of runs of consecutive indices (input already in
    cell order, with a few stretches out of order), against the oracle."""
    rng = np.random.default_rng(n + 7)
    rows = rng.standard_normal((n, 8)).astype(np.float32)
    ordenado = np.arange(n, dtype=np.uint32)
    for _ in range(min(20, n // 64)):
        a = int(rng.integers(0, n - 32))
        ordenado[a:a + 32] = ordenado[a:a + 32][::-1].copy()
    p = ug.make_params(n, (4, 4, 4), (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    origen = torch.from_numpy(rows).cuda()
    destino = torch.full_like(origen, float("nan"))
    ug.grid_reorder(torch.from_numpy(ordenado.view(np.int32)).cuda(), origen, destino, ws, p)
    torch.cuda.synchronize()
    assert ug.grid_status(ws) == 0
    assert np.array_equal(destino.cpu().numpy().view(np.uint32), oracle_lib.reorder(ordenado, rows).view(np.uint32))


def test_scan_large_counts(ug, oracle_lib):
    """Counts up to 1000 per cell (totals near 2^31) over a ragged cell count."""
    C = 2_097_152 + 1234
    rng = np.random.default_rng(4)
    conteos = rng.integers(0, 1000, C, dtype=np.uint32)
    p = ug.make_params(int(conteos.sum()) & 0xFFFFFFFF, (C, 1, 1), (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    inicios = torch.empty(C + 1, dtype=torch.int32, device="cuda")
    for _ in range(3):   # the workspace is reusable call after call
        ug.grid_scan(torch.from_numpy(conteos.view(np.int32)).cuda(), inicios, ws, p)
        assert np.array_equal(to_u32(inicios), oracle_lib.exclusive_scan(conteos))
    assert ug.grid_status(ws) == 0


# Scenes of a few million particles: more buckets than CTAs, so every CTA
# places several buckets in phase D, and skewed ones whose crowded buckets
# take the atomic fallback; at grid sizes that need no more than a few seconds
# of oracle time.
LARGE = [
    ("uniform", 4_194_304, (160, 160, 160)),
    ("skewed", 2_500_000, (128, 128, 128)),
    ("one_cell_heavy", 1_500_000, (64, 64, 64)),
]


def _large_rows(kind: str, n: int, dims) -> np.ndarray:
    if kind == "uniform":
        rows = scenes.uniform_particles(n, 0xC0FFEE)
    elif kind == "skewed":
        rows = scenes.contention_particles(n, 0xC0FFEF, dims[0])
    else:
        # a third of the particles on one cell centre, the rest uniform
        rows = scenes.uniform_particles(n, 0xC0FFF0)
        centre = np.float32(-5.0 + (dims[0] // 3 + 0.5) * (10.0 / dims[0]))
        rows[: n // 3, :3] = centre
    return rows


@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
@pytest.mark.parametrize("kind,n,dims", LARGE, ids=[g[0] for g in LARGE])
def test_large_scenes(ug, oracle_lib, kind, n, dims, stable):
    rows = _large_rows(kind, n, dims)
    cs = float(np.float32(10.0 / dims[0]))
    origin = (-5.0, -5.0, -5.0)
    ref = oracle_lib.build(rows, dims, origin, cs)
    flags = ug.GRID_STABLE if stable else 0
    got = gpu_build(ug, rows, dims, origin, cs, flags=flags)
    assert_matches_oracle(oracle_lib, rows, got, ref, stable)
