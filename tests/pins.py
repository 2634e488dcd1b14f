"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code.

Every ``pin_*`` function takes an ``oracle.Oracle`` (the real library or a
planted mutant) and raises ``AssertionError`` on a mismatch.  The sources of
truth are:

* the pages' worked example of the exclusive scan (``golden/scan_worked_example.txt``);
* a hand-evaluated table of the linear cell index (``golden/linear_cell_index.txt``);
* exact rational arithmetic (``fractions.Fraction``) for floor((p - o) / cellSize);
* closed forms for special positions (cell centres and faces, the domain's
  edges, out-of-domain values, NaN and infinities);
* independent library routines for whole steps: ``numpy.bincount`` (histogram),
  ``numpy.cumsum`` (scan), a stable ``numpy.argsort`` (scatter), numpy fancy
  indexing (gather);
* a pure-Python brute force on tiny inputs;
* for the Morton order, a hand-interleaved table (``golden/morton_cell_index.txt``),
  bijection and aligned-block contiguity, and the XOR comparison of two cells
  (a definition of the Z-curve order that builds no code).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
F32 = np.float32


def read_golden(name: str) -> list[list[str]]:
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _rows_at(points) -> np.ndarray:
    pts = np.asarray(points, dtype=np.float32).reshape(-1, 3)
    rows = np.zeros((pts.shape[0], 8), dtype=np.float32)
    rows[:, :3] = pts
    rows[:, 3] = 1.0
    rows[:, 7] = 1.0
    return rows


# ---------------------------------------------------------------- cell index

def pin_cell_index_special_positions(o) -> None:
    """Closed forms at the three grid resolutions of the workloads."""
    for dims in (16, 128, 256):
        cs = F32(10.0 / dims)
        stride = (1, dims, dims * dims)
        d3 = (dims, dims, dims)
        org = (-5.0, -5.0, -5.0)
        k = np.arange(dims, dtype=np.float64)
        centres = (F32(-5.0) + ((k + 0.5) * float(cs)).astype(np.float32)).astype(np.float32)
        faces = (-5.0 + k * float(cs)).astype(np.float32)
        assert np.all(centres.astype(np.float64) == -5.0 + (k + 0.5) * float(cs)), "centres not exact"
        assert np.all(faces.astype(np.float64) == -5.0 + k * float(cs)), "faces not exact"
        for axis in range(3):
            for values, what in ((centres, "centre"), (faces, "lower face")):
                pts = np.zeros((dims, 3), dtype=np.float32)
                pts[:] = F32(-5.0)            # other axes at the origin -> coordinate 0
                pts[:, axis] = values
                got = o.cell_index(_rows_at(pts), d3, org, cs)
                want = np.arange(dims, dtype=np.uint32) * np.uint32(stride[axis])
                assert np.array_equal(got, want), f"{what} of every cell, axis {axis}, dims {dims}"
        top = dims - 1
        below5 = np.nextafter(F32(5.0), F32(0.0))
        cases = [
            ((-5.0, -5.0, -5.0), (0, 0, 0)),            # the origin itself
            ((below5, below5, below5), (top, top, top)),  # largest fp32 below the upper edge
            ((5.0, 5.0, 5.0), (top, top, top)),          # the upper edge: clamped
            ((-8.0, 0.0, 8.0), (0, dims // 2, top)),    # outside on both sides
            ((-5.0000005, -5.0, -5.0), (0, 0, 0)),      # just below the origin
            ((math.nan, 8.0, -math.inf), (0, top, 0)),  # NaN -> 0, -inf -> 0
            ((math.inf, math.nan, 1e30), (top, 0, top)),
            ((-1e30, -0.0, 0.0), (0, dims // 2, dims // 2)),
        ]
        pts = [c[0] for c in cases]
        got = o.cell_index(_rows_at(pts), d3, org, cs)
        for (p, xyz), g in zip(cases, got):
            want = xyz[0] + xyz[1] * dims + xyz[2] * dims * dims
            assert int(g) == want, f"position {p} at dims {dims}: got {int(g)}, want {want}"


def _exact_axis(p: float, o: float, cs: float, dim: int) -> int | None:
    """Clamped floor((p - o) / cs) in exact rationals; None when p is within the
    fp32 rounding band of a cell face (there the fp32 evaluation may differ)."""
    r = (Fraction(p) - Fraction(o)) / Fraction(cs)
    f = math.floor(r)
    band = abs(r) * Fraction(1, 1 << 20) + Fraction(1, 1 << 40)
    if r - f < band or (f + 1) - r < band:
        return None
    return min(max(f, 0), dim - 1)


def pin_cell_index_exact_rationals(o, samples: int = 4000, seed: int = 11) -> None:
    """fp32 evaluation agrees with the exact rational cell away from faces."""
    rng = np.random.default_rng(seed)
    dims = (7, 11, 13)
    origin = (F32(-3.25), F32(1.5), F32(-0.375))
    cs = F32(0.8)
    lo = np.array(origin, dtype=np.float64) - 2.0
    hi = lo + 4.0 + np.array(dims) * float(cs)
    pts = (lo + (hi - lo) * rng.random((samples, 3))).astype(np.float32)
    got = o.cell_index(_rows_at(pts), dims, origin, cs)
    checked = 0
    for i in range(samples):
        xyz = [_exact_axis(float(pts[i, d]), float(origin[d]), float(cs), dims[d]) for d in range(3)]
        if any(v is None for v in xyz):
            continue
        checked += 1
        want = xyz[0] + xyz[1] * dims[0] + xyz[2] * dims[0] * dims[1]
        assert int(got[i]) == want, f"particle {pts[i]}: got {int(got[i])}, exact {want}"
    assert checked > samples * 0.99, "too many samples fell in the rounding band"


def pin_linear_index_table(o) -> None:
    """Hand-evaluated x + y*GX + z*GX*GY on a 3x5x7 grid with an offset origin."""
    dims, origin, cs = (3, 5, 7), (1.0, -2.0, 3.0), 0.5
    table = [tuple(int(v) for v in r) for r in read_golden("linear_cell_index.txt")]
    pts = [(origin[0] + (x + 0.5) * cs, origin[1] + (y + 0.5) * cs, origin[2] + (z + 0.5) * cs)
           for x, y, z, _ in table]
    got = o.cell_index(_rows_at(pts), dims, origin, cs)
    for (x, y, z, idx), g in zip(table, got):
        assert int(g) == idx, f"cell ({x},{y},{z}): got {int(g)}, table says {idx}"


# ---------------------------------------------------------------- histogram

def pin_histogram(o, seed: int = 5) -> None:
    rng = np.random.default_rng(seed)
    for n, cells in ((0, 1), (1, 1), (1000, 7), (20000, 4096), (5000, 100000)):
        celda = rng.integers(0, cells, n, dtype=np.uint32)
        got = o.histogram(celda, cells)
        assert np.array_equal(got, np.bincount(celda, minlength=cells).astype(np.uint32))
        assert int(got.sum(dtype=np.uint64)) == n
    one = np.full(777, 3, dtype=np.uint32)
    got = o.histogram(one, 9)
    assert got[3] == 777 and got.sum() == 777


# ---------------------------------------------------------------- scan

def pin_scan_worked_example(o) -> None:
    g = {r[0]: np.array([int(v) for v in r[1:]], dtype=np.uint32) for r in read_golden("scan_worked_example.txt")}
    got = o.exclusive_scan(g["conteos"])
    assert np.array_equal(got, g["inicios"]), f"scan of {g['conteos']}: {got}"
    assert np.array_equal(got[1:], g["finales"])
    assert got[1] == got[2], "empty cell 1 starts where it ends"


def pin_scan_cumsum(o, seed: int = 6) -> None:
    rng = np.random.default_rng(seed)
    for cells in (1, 2, 31, 4096, 100001):
        conteos = rng.integers(0, 50, cells, dtype=np.uint32)
        conteos[rng.random(cells) < 0.5] = 0
        got = o.exclusive_scan(conteos)
        want = np.concatenate([[0], np.cumsum(conteos, dtype=np.uint64)]).astype(np.uint32)
        assert np.array_equal(got, want)
        assert np.all(np.diff(got.astype(np.int64)) >= 0)
        assert int(got[-1]) == int(conteos.sum(dtype=np.uint64))


# ---------------------------------------------------------------- scatter

def pin_scatter_stable_sort(o, seed: int = 7) -> None:
    rng = np.random.default_rng(seed)
    for n, cells in ((0, 3), (1, 1), (64, 27), (5000, 50), (30000, 70000)):
        celda = rng.integers(0, cells, n, dtype=np.uint32)
        inicios = np.concatenate([[0], np.cumsum(np.bincount(celda, minlength=cells))]).astype(np.uint32)
        got = o.scatter(celda, inicios)
        want = np.argsort(celda, kind="stable").astype(np.uint32)
        assert np.array_equal(got, want), "scatter is not the stable counting sort"
        assert np.array_equal(np.sort(got), np.arange(n, dtype=np.uint32)), "not a permutation"
        for c in rng.integers(0, cells, min(cells, 50)):
            seg = got[inicios[c]:inicios[c + 1]]
            assert np.all(celda[seg] == c), "particle outside its cell's segment"


# ---------------------------------------------------------------- gather

def pin_reorder_gather(o, seed: int = 8) -> None:
    rng = np.random.default_rng(seed)
    for n in (0, 1, 333, 10000):
        bits = rng.integers(0, 2**32, (n, 8), dtype=np.uint64).astype(np.uint32)
        origen = bits.view(np.float32)                      # arbitrary bytes, NaN payloads included
        ordenado = rng.permutation(n).astype(np.uint32)
        got = o.reorder(ordenado, origen)
        assert np.array_equal(got.view(np.uint32), bits[ordenado]), "destino[k] != origen[ordenado[k]]"


# ---------------------------------------------------------------- whole chain

def _brute_force(cells_xyz, dims):
    """Pure-Python definition of the build for particles placed at cell centres."""
    gx, gy, gz = dims
    cell = []
    for x, y, z in cells_xyz:
        x = min(max(x, 0), gx - 1)
        y = min(max(y, 0), gy - 1)
        z = min(max(z, 0), gz - 1)
        cell.append(x + gx * (y + gy * z))
    count = [0] * (gx * gy * gz)
    for c in cell:
        count[c] += 1
    start = [0]
    for v in count:
        start.append(start[-1] + v)
    order = sorted(range(len(cell)), key=lambda i: cell[i])   # Python's sort is stable
    return cell, count, start, order


def pin_build_brute_force(o, seeds: int = 200) -> None:
    for s in range(seeds):
        rng = np.random.default_rng(1000 + s)
        dims = tuple(int(v) for v in rng.integers(1, 5, 3))
        n = int(rng.integers(0, 65))
        cs = 0.75
        origin = (float(rng.integers(-4, 4)) * 0.5,) * 3
        xyz = [(int(rng.integers(-2, dims[0] + 2)), int(rng.integers(-2, dims[1] + 2)),
                int(rng.integers(-2, dims[2] + 2))) for _ in range(n)]
        pts = [tuple(origin[d] + (xyz[i][d] + 0.5) * cs for d in range(3)) for i in range(n)]
        rows = _rows_at(pts) if n else np.zeros((0, 8), dtype=np.float32)
        rows[:, 3] = rng.random(n).astype(np.float32)      # distinct payloads to follow the records
        rows[:, 7] = np.arange(n, dtype=np.float32)
        out = o.build(rows, dims, origin, cs)
        cell, count, start, order = _brute_force(xyz, dims)
        assert out["celdaDe"].tolist() == cell, f"seed {s}: celdaDe"
        assert out["conteos"].tolist() == count, f"seed {s}: conteos"
        assert out["inicios"].tolist() == start, f"seed {s}: inicios"
        assert out["ordenado"].tolist() == order, f"seed {s}: ordenado"
        assert np.array_equal(out["destino"].view(np.uint32), rows[order].view(np.uint32)), f"seed {s}: destino"


def pin_build_degenerate(o) -> None:
    """Empty scene; every particle in one cell; one cell only."""
    out = o.build(np.zeros((0, 8), np.float32), (4, 4, 4), (0, 0, 0), 1.0)
    assert not out["conteos"].any() and not out["inicios"].any()
    rows = _rows_at([(2.5, 1.5, 3.5)] * 500)
    out = o.build(rows, (4, 4, 4), (0, 0, 0), 1.0)
    c = 2 + 4 * 1 + 16 * 3
    assert out["conteos"][c] == 500 and out["conteos"].sum() == 500
    assert np.array_equal(out["ordenado"], np.arange(500, dtype=np.uint32))
    assert int(out["inicios"][c]) == 0 and int(out["inicios"][c + 1]) == 500 and int(out["inicios"][-1]) == 500
    out = o.build(_rows_at([(-9, 0, 9), (1, 1, 1)]), (1, 1, 1), (0, 0, 0), 2.0)
    assert out["celdaDe"].tolist() == [0, 0] and out["inicios"].tolist() == [0, 2]


def pin_canonicalise(o, seed: int = 9) -> None:
    rng = np.random.default_rng(seed)
    celda = rng.integers(0, 40, 3000, dtype=np.uint32)
    inicios = np.concatenate([[0], np.cumsum(np.bincount(celda, minlength=40))]).astype(np.uint32)
    stable = np.argsort(celda, kind="stable").astype(np.uint32)
    shuffled = stable.copy()
    for c in range(40):
        seg = shuffled[inicios[c]:inicios[c + 1]]
        rng.shuffle(seg)
    assert not np.array_equal(shuffled, stable)
    assert np.array_equal(o.canonicalise(inicios, shuffled), stable)
    # Hand example with segments of every short length: empty, one, a reversed
    # pair, three out of order, and a pair already in order.
    inicios = np.array([0, 0, 1, 3, 6, 8], dtype=np.uint32)
    ordenado = np.array([5, 9, 2, 7, 4, 1, 0, 3], dtype=np.uint32)
    assert o.canonicalise(inicios, ordenado).tolist() == [5, 2, 9, 1, 4, 7, 0, 3]


def pin_reorder_records(o, seed: int = 13) -> None:
    """Any record size: numpy fancy indexing; 32-byte records: the same as the
    particle gather."""
    rng = np.random.default_rng(seed)
    for n in (0, 1, 777):
        perm = rng.permutation(n).astype(np.uint32)
        for rb in (16, 32, 48, 256):
            recs = rng.integers(0, 256, (n, rb), dtype=np.uint8)
            assert np.array_equal(o.reorder_records(perm, recs), recs[perm]), f"record size {rb}"
        parts = rng.random((n, 8), dtype=np.float32)
        assert np.array_equal(o.reorder_records(perm, parts), o.reorder(perm, parts))


# ---------------------------------------------------------------- neighbour density

def _brute_density(rows, h):
    """All pairs, float64 from the fp32 records: sum_j m_j (h^2 - r^2)^3 over r < h."""
    pos = rows[:, :3].astype(np.float64)
    m = rows[:, 7].astype(np.float64)
    out = np.zeros(rows.shape[0])
    for i in range(rows.shape[0]):
        e = pos - pos[i]
        r2 = e[:, 0] * e[:, 0] + e[:, 1] * e[:, 1] + e[:, 2] * e[:, 2]
        t = np.where(r2 < h * h, h * h - r2, 0.0)
        out[i] = float(np.sum(m * t * t * t))
    return out


def pin_density_brute_force(o, seed: int = 14) -> None:
    """The 27-cell walk finds exactly the neighbours an all-pairs search finds,
    inside the domain and beyond it (clamped particles), on non-cubic grids."""
    rng = np.random.default_rng(seed)
    for dims, cs, n in (((6, 4, 5), 0.5, 900), ((3, 3, 3), 1.0, 400), ((10, 1, 7), 0.25, 700)):
        origin = (-1.0, 0.5, 2.0)
        lo = np.array(origin) - 0.6
        hi = np.array(origin) + np.array(dims) * cs + 0.6
        rows = np.zeros((n, 8), np.float32)
        rows[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
        rows[:, 7] = (0.5 + rng.random(n)).astype(np.float32)
        ref = o.build(rows, dims, origin, cs)
        for h in (cs, 0.7 * cs):
            got = o.density(rows, dims, origin, cs, ref["inicios"], ref["ordenado"], h)
            want = _brute_density(rows, h)
            assert np.allclose(got, want, rtol=1e-12, atol=1e-300), f"dims {dims} h {h}"


def pin_density_stale_grid(o, seed: int = 15) -> None:
    """A grid built before the particles moved: each particle walks the 27
    cells around the cell of its current position, and a candidate counts
    where the grid lists it (its cell at build time), at its current position.
    Brute force over all pairs with that membership rule."""
    rng = np.random.default_rng(seed)
    for order in (0, 1):
        dims, origin, cs, n = (4, 4, 4), (-1.0, 0.5, 2.0), 0.5, 600
        lo, hi = np.array(origin), np.array(origin) + np.array(dims) * cs
        before = np.zeros((n, 8), np.float32)
        before[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
        before[:, 7] = (0.5 + rng.random(n)).astype(np.float32)
        after = before.copy()
        after[:, :3] += (rng.uniform(-0.4, 0.4, (n, 3)) * cs).astype(np.float32)
        grid = o.build(before, dims, origin, cs, order=order)
        now = o.build(after, dims, origin, cs, order=order)
        # cell coordinates from the cell index of each order
        code_xyz = {}
        for z in range(dims[2]):
            for y in range(dims[1]):
                for x in range(dims[0]):
                    c = x + dims[0] * (y + dims[1] * z) if order == 0 else o.morton_cell(x, y, z, dims)
                    code_xyz[c] = np.array((x, y, z))
        listed = np.array([code_xyz[int(c)] for c in grid["celdaDe"]])
        current = np.array([code_xyz[int(c)] for c in now["celdaDe"]])
        moved = int(np.sum(np.any(listed != current, axis=1)))
        assert moved > n // 4, "the displacement moves a good share of the particles"
        pos, m = after[:, :3].astype(np.float64), after[:, 7].astype(np.float64)
        for h in (cs, 0.7 * cs):
            want = np.zeros(n)
            for i in range(n):
                near = np.all(np.abs(listed - current[i]) <= 1, axis=1)
                e = pos[near] - pos[i]
                r2 = e[:, 0] * e[:, 0] + e[:, 1] * e[:, 1] + e[:, 2] * e[:, 2]
                t = np.where(r2 < h * h, h * h - r2, 0.0)
                want[i] = float(np.sum(m[near] * t * t * t))
            got = o.density(after, dims, origin, cs, grid["inicios"], grid["ordenado"], h, order=order)
            assert np.allclose(got, want, rtol=1e-12, atol=1e-300), f"order {order} h {h}"


def pin_density_closed_forms(o) -> None:
    dims, origin, cs, h = (8, 8, 8), (0.0, 0.0, 0.0), 1.0, 1.0
    # one particle alone: its own mass times h^6
    rows = _rows_at([(3.5, 3.5, 3.5)])
    rows[:, 7] = 2.0
    ref = o.build(rows, dims, origin, cs)
    assert o.density(rows, dims, origin, cs, ref["inicios"], ref["ordenado"], h)[0] == 2.0
    # two particles 0.5 apart across a cell face: each gets its own term plus
    # the other's mass times (h^2 - 0.25)^3
    rows = _rows_at([(3.75, 4.0, 4.0), (4.25, 4.0, 4.0)])
    rows[:, 7] = [1.0, 3.0]
    ref = o.build(rows, dims, origin, cs)
    got = o.density(rows, dims, origin, cs, ref["inicios"], ref["ordenado"], h)
    assert got.tolist() == [1.0 + 3.0 * 0.75 ** 3, 3.0 + 1.0 * 0.75 ** 3]
    # exactly h apart: not a neighbour
    rows = _rows_at([(3.5, 4.5, 4.0), (4.5, 4.5, 4.0)])
    ref = o.build(rows, dims, origin, cs)
    assert o.density(rows, dims, origin, cs, ref["inicios"], ref["ordenado"], h).tolist() == [1.0, 1.0]


# ---------------------------------------------------------------- diagnostics

def pin_diagnostics(o, seed: int = 12) -> None:
    """Hand-evaluated cases, then the closed forms maxPorCelda = max(conteos)
    and desbordes = sum over cells of max(0, conteos - capacidad)."""
    for row in read_golden("overflow_diagnostics.txt"):
        text = " ".join(row)
        cap_s, cells_s, want_s = [part.strip() for part in text.split(";")]
        celda = np.array([int(v) for v in cells_s.split()], dtype=np.uint32)
        want = tuple(int(v) for v in want_s.split())
        cells = int(celda.max()) + 1 if celda.size else 1
        assert o.diagnostics(celda, cells, int(cap_s)) == want, f"{text}"
    rng = np.random.default_rng(seed)
    for n, cells, cap in ((5000, 40, 64), (20000, 100, 150), (3000, 5000, 1), (0, 7, 64)):
        celda = rng.integers(0, cells, n, dtype=np.uint32)
        counts = np.bincount(celda, minlength=cells).astype(np.int64)
        want = (int(counts.max()) if n else 0, int(np.maximum(counts - cap, 0).sum()))
        assert o.diagnostics(celda, cells, cap) == want


# ---------------------------------------------------------------- Morton order

def _centres(dims, origin, cs, cells_xyz):
    return _rows_at([(origin[0] + (x + 0.5) * cs, origin[1] + (y + 0.5) * cs, origin[2] + (z + 0.5) * cs)
                     for x, y, z in cells_xyz])


def _all_cells(dims):
    gx, gy, gz = dims
    return [(x, y, z) for z in range(gz) for y in range(gy) for x in range(gx)]


def pin_morton_index_table(o) -> None:
    """Hand-interleaved Morton codes on cubic and unequal power-of-two grids,
    through the exported helper and through the cell index of cell centres."""
    origin, cs = (-1.0, 2.0, 0.5), 0.25
    for row in read_golden("morton_cell_index.txt"):
        gx, gy, gz, x, y, z, idx = (int(v) for v in row)
        assert o.morton_cell(x, y, z, (gx, gy, gz)) == idx, f"{row}"
        got = o.cell_index(_centres((gx, gy, gz), origin, cs, [(x, y, z)]), (gx, gy, gz), origin, cs, order=1)
        assert int(got[0]) == idx, f"cell index of {row}: {int(got[0])}"


def pin_morton_bijection_and_blocks(o) -> None:
    """The Morton index is a bijection onto [0, cells), and every aligned
    2^k x 2^k x 2^k block of a cubic grid (2x2x2 blocks on every grid whose
    sides are all >= 2) holds one contiguous range of codes starting at a
    multiple of its size: the locality the page wants from the Z-curve."""
    origin, cs = (0.0, 0.0, 0.0), 1.0
    for dims in ((4, 4, 4), (8, 2, 4), (16, 8, 2), (1, 8, 4), (2, 1, 1), (16, 16, 16), (32, 4, 8)):
        cells = _all_cells(dims)
        codes = o.cell_index(_centres(dims, origin, cs, cells), dims, origin, cs, order=1).astype(np.int64)
        assert np.array_equal(np.sort(codes), np.arange(len(cells))), f"not a bijection on {dims}"
        xyz = np.array(cells, dtype=np.int64)
        sides = [1]
        if min(dims) >= 2:
            sides.append(2)
        if dims[0] == dims[1] == dims[2]:
            sides = [1 << k for k in range(int(math.log2(dims[0])) + 1)]
        for side in sides:
            key = (xyz[:, 0] // side) + dims[0] * ((xyz[:, 1] // side) + dims[1] * (xyz[:, 2] // side))
            for b in np.unique(key):
                block = np.sort(codes[key == b])
                size = side ** 3
                assert block.size == size and block[0] % size == 0 and block[-1] - block[0] == size - 1, (
                    f"{side}-block {b} of {dims} is not contiguous: {block[:4]}..")


def _zorder_less(a, b) -> int:
    """Comparison of two cells by the most significant differing bit of any
    coordinate (Chan's XOR test): the axis whose XOR has the highest bit
    decides, z outranking y outranking x at equal bit position.  This is the
    order of the Z-curve on a cubic grid, stated without building a code."""
    rank = max(((a[k] ^ b[k]).bit_length(), k) for k in (0, 1, 2))
    if rank[0] == 0:
        return 0
    k = rank[1]
    return -1 if a[k] < b[k] else 1


def pin_morton_matches_xor_comparator(o) -> None:
    """On cubic grids the Morton order of the cells is the order given by the
    XOR comparison, a definition that never interleaves bits."""
    import functools
    origin, cs = (0.0, 0.0, 0.0), 1.0
    for dims in ((8, 8, 8), (16, 16, 16)):
        cells = _all_cells(dims)
        codes = o.cell_index(_centres(dims, origin, cs, cells), dims, origin, cs, order=1)
        by_code = [cells[i] for i in np.argsort(codes, kind="stable")]
        by_xor = sorted(cells, key=functools.cmp_to_key(_zorder_less))
        assert by_code == by_xor, f"Morton order differs from the XOR comparison on {dims}"


def pin_build_orders_agree(o, seed: int = 15) -> None:
    """A build in Morton order is the linear build with its cells relabelled:
    the same particles fall in the same physical cell, every cell keeps its
    count and its members, and the neighbour density does not depend on the
    order (same neighbour sets; sums compared to rounding)."""
    rng = np.random.default_rng(seed)
    for dims, cs, n in (((8, 4, 16), 0.5, 3000), ((4, 4, 4), 1.0, 600), ((2, 8, 1), 0.75, 300)):
        origin = (-0.3, 1.0, 0.2)
        lo = np.array(origin) - 0.4
        hi = np.array(origin) + np.array(dims) * cs + 0.4
        rows = np.zeros((n, 8), np.float32)
        rows[:, :3] = (lo + (hi - lo) * rng.random((n, 3))).astype(np.float32)
        rows[:, 7] = (0.5 + rng.random(n)).astype(np.float32)
        lin = o.build(rows, dims, origin, cs, order=0)
        mor = o.build(rows, dims, origin, cs, order=1)
        cells = _all_cells(dims)
        relabel = o.cell_index(_centres(dims, origin, cs, cells), dims, origin, cs, order=1)
        assert np.array_equal(relabel[lin["celdaDe"]], mor["celdaDe"]), f"celdaDe differs on {dims}"
        assert np.array_equal(mor["conteos"][relabel], lin["conteos"]), f"conteos differ on {dims}"
        for c_lin, c_mor in enumerate(relabel):
            a = lin["ordenado"][lin["inicios"][c_lin]:lin["inicios"][c_lin + 1]]
            b = mor["ordenado"][mor["inicios"][c_mor]:mor["inicios"][c_mor + 1]]
            assert np.array_equal(a, b), f"members of cell {c_lin} differ on {dims}"
        for h in (cs, 0.6 * cs):
            d_lin = o.density(rows, dims, origin, cs, lin["inicios"], lin["ordenado"], h, order=0)
            d_mor = o.density(rows, dims, origin, cs, mor["inicios"], mor["ordenado"], h, order=1)
            assert np.allclose(d_mor, d_lin, rtol=1e-12, atol=0.0), f"density depends on the order ({dims}, h={h})"
            assert np.allclose(d_mor, _brute_density(rows, h), rtol=1e-12, atol=1e-300)


ALL_PINS = [
    pin_cell_index_special_positions,
    pin_linear_index_table,
    pin_cell_index_exact_rationals,
    pin_histogram,
    pin_scan_worked_example,
    pin_scan_cumsum,
    pin_scatter_stable_sort,
    pin_reorder_gather,
    pin_build_degenerate,
    pin_build_brute_force,
    pin_canonicalise,
    pin_diagnostics,
    pin_reorder_records,
    pin_density_closed_forms,
    pin_density_brute_force,
    pin_density_stale_grid,
    pin_morton_index_table,
    pin_morton_bijection_and_blocks,
    pin_morton_matches_xor_comparator,
    pin_build_orders_agree,
]


def run_all(o) -> None:
    for pin in ALL_PINS:
        pin(o)
