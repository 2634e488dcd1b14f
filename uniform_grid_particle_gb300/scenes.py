"""Seeded synthetic particle scenes for the uniform-grid build.

This module only draws inputs: it holds none of the grid arithmetic (no cell
index, no histogram, no scan, no scatter, no gather), so both the CUDA path
and the CPU oracle can be fed from it without sharing any of the method.

Particle record: the 32-byte ``Particula {pos: vec3f, vida: f32, vel: vec3f,
masa: f32}`` of "El estado de las partículas en storage buffers"
(§La estructura y su alineación), stored as float32 ``[N, 8]`` rows:
pos.x, pos.y, pos.z, vida, vel.x, vel.y, vel.z, masa.

Field distributions follow the JavaScript initialiser of that section:
pos uniform in [-5, 5)^3, vida uniform in [1, 4), vel = 0, masa uniform in
[0.5, 1.5).  The random source is numpy's PCG64 bit generator (its raw 64-bit
stream is stable across numpy versions); every float is built here from the
raw words, so no numpy distribution routine is involved.

Scenes (grid origin (-5,-5,-5), cellSize = 10 / dims, exact in fp32):

=============== =========== ========== =========================================
name            N           dims       structure
=============== =========== ========== =========================================
tiny            4,096       16^3       uniform
scan_dominated  100,000     128^3      uniform (the scan over cells dominates)
headline        1,000,000   128^3      uniform
contention      1,000,000   128^3      98 % N(0, 1)^3, 1 % on one cell centre
                                       (cell (64,64,64)), 1 % uniform in
                                       [-8, 8)^3 (mostly outside: clamped);
                                       shuffled
stress          16,777,216  256^3      uniform; built 10 times, ping-pong
sph             5,242,880   64^3       uniform; 20 per cell, ~84 neighbours
                                       within one cell size, records (168 MB)
                                       above L2: for the neighbour query
sph_dense       13,107,200  64^3       uniform; 50 per cell (the dense
                                       neighbour query), records 420 MB
=============== =========== ========== =========================================
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

FLOATS_PER_PARTICLE = 8
RECORD_BYTES = 32

# Offsets of the fields in a row of the float32 [N, 8] view.
POS = slice(0, 3)
VIDA = 3
VEL = slice(4, 7)
MASA = 7

_U24 = 1.0 / float(1 << 24)


@dataclasses.dataclass(frozen=True)
class Scene:
    """One synthetic workload: geometry plus the particle count and recipe."""

    name: str
    n: int
    dims: tuple[int, int, int]
    origin: tuple[float, float, float] = (-5.0, -5.0, -5.0)
    extent: float = 10.0
    kind: str = "uniform"        # "uniform" | "contention"
    builds: int = 1              # consecutive builds with origen/destino swapped
    seed_index: int = 0

    @property
    def cells(self) -> int:
        return self.dims[0] * self.dims[1] * self.dims[2]

    @property
    def cell_size(self) -> float:
        # 10/16, 10/128, 10/256 are exact in fp32; the value is returned as the
        # fp32 number it denotes.
        assert self.dims[0] == self.dims[1] == self.dims[2]
        return float(np.float32(self.extent / self.dims[0]))

    @property
    def seed(self) -> int:
        return 0x5EED0000 + self.seed_index

    def particles(self) -> np.ndarray:
        """float32 [N, 8] particle rows (pos, vida, vel, masa), seeded."""
        if self.kind == "uniform":
            return uniform_particles(self.n, self.seed)
        if self.kind == "contention":
            return contention_particles(self.n, self.seed, self.dims[0])
        raise ValueError(self.kind)


SCENES: dict[str, Scene] = {
    s.name: s
    for s in (
        Scene("tiny", 4096, (16, 16, 16), seed_index=0),
        Scene("scan_dominated", 100_000, (128, 128, 128), seed_index=1),
        Scene("headline", 1_000_000, (128, 128, 128), seed_index=2),
        Scene("contention", 1_000_000, (128, 128, 128), kind="contention", seed_index=3),
        Scene("stress", 16_777_216, (256, 256, 256), builds=10, seed_index=4),
        # 20 particles per cell, so about 84 within one cell size: the cell
        # occupancy of "Contar partículas por celda" (§Elegir bien el tamaño de
        # celda) and the SPH neighbour count of "Reordenar por celda…" (§Qué
        # cuesta la indirección).  Power-of-two sides, so it also builds in
        # Morton order.
        Scene("sph", 5_242_880, (64, 64, 64), seed_index=5),
        # 50 particles per cell, near the top of the 20-60 per cell that
        # "Contar partículas por celda" calls healthy: the dense neighbour
        # query.  Records 420 MB, above L2.
        Scene("sph_dense", 13_107_200, (64, 64, 64), seed_index=6),
    )
}


def _raw(rng: np.random.PCG64, count: int) -> np.ndarray:
    return rng.random_raw(count).astype(np.uint64, copy=False)


def _unit(raw: np.ndarray) -> np.ndarray:
    """[0, 1) doubles with 24 random bits: (raw >> 40) * 2^-24."""
    return (raw >> np.uint64(40)).astype(np.float64) * _U24


def _uniform_f32(raw: np.ndarray, lo: float, hi: float) -> np.ndarray:
    """lo + (hi - lo) * u computed in double, rounded to fp32, kept below hi."""
    v = (lo + (hi - lo) * _unit(raw)).astype(np.float32)
    below = np.nextafter(np.float32(hi), np.float32(lo))
    return np.where(v >= np.float32(hi), below, v).astype(np.float32)


def _fill_common(rows: np.ndarray, rng: np.random.PCG64) -> None:
    """vida U[1,4), vel 0, masa U[0.5,1.5) — two draws per particle."""
    n = rows.shape[0]
    raw = _raw(rng, 2 * n).reshape(n, 2)
    rows[:, VIDA] = _uniform_f32(raw[:, 0], 1.0, 4.0)
    rows[:, VEL] = 0.0
    rows[:, MASA] = _uniform_f32(raw[:, 1], 0.5, 1.5)


def uniform_particles(n: int, seed: int, lo: float = -5.0, hi: float = 5.0) -> np.ndarray:
    """N particles with pos uniform in [lo, hi)^3 (three draws each)."""
    rng = np.random.PCG64(seed)
    rows = np.zeros((n, FLOATS_PER_PARTICLE), dtype=np.float32)
    raw = _raw(rng, 3 * n).reshape(n, 3)
    for d in range(3):
        rows[:, d] = _uniform_f32(raw[:, d], lo, hi)
    _fill_common(rows, rng)
    return rows


def _gaussian_f32(rng: np.random.PCG64, count: int, sigma: float = 1.0) -> np.ndarray:
    """Box-Muller in double from u1 in (0, 1], u2 in [0, 1), rounded to fp32."""
    pairs = (count + 1) // 2
    raw = _raw(rng, 2 * pairs).reshape(pairs, 2)
    u1 = 1.0 - _unit(raw[:, 0])                    # (0, 1]
    u2 = _unit(raw[:, 1])
    r = np.sqrt(-2.0 * np.log(u1)) * sigma
    z = np.stack([r * np.cos(2.0 * math.pi * u2), r * np.sin(2.0 * math.pi * u2)], axis=1)
    return z.reshape(-1)[:count].astype(np.float32)


def random_permutation(n: int, rng: np.random.PCG64) -> np.ndarray:
    """A seeded permutation of 0..n-1: stable argsort of n raw 64-bit draws."""
    return np.argsort(_raw(rng, n), kind="stable")


def contention_particles(n: int, seed: int, dims: int, shuffle: bool = True) -> np.ndarray:
    """98 % N(0,1)^3 around the domain centre, 1 % on one cell centre, 1 % in [-8,8)^3.

    The hot cell is the one whose lower corner is the domain centre: with the
    grid over [-5, 5)^3 that is cell (dims/2, dims/2, dims/2), whose centre is
    -5 + (dims/2 + 1/2) * 10/dims (0.0390625 at 128^3, exact in fp32).
    """
    rng = np.random.PCG64(seed)
    hot = n // 100
    wide = n // 100
    gauss = n - hot - wide
    rows = np.zeros((n, FLOATS_PER_PARTICLE), dtype=np.float32)
    g = _gaussian_f32(rng, 3 * gauss).reshape(gauss, 3)
    rows[:gauss, POS] = g
    centre = np.float32(-5.0 + (dims // 2 + 0.5) * (10.0 / dims))
    rows[gauss:gauss + hot, POS] = centre
    raw = _raw(rng, 3 * wide).reshape(wide, 3)
    for d in range(3):
        rows[gauss + hot:, d] = _uniform_f32(raw[:, d], -8.0, 8.0)
    _fill_common(rows, rng)
    if shuffle:
        rows = rows[random_permutation(n, rng)]
    return np.ascontiguousarray(rows)


def single_cell_particles(n: int, seed: int, point: tuple[float, float, float]) -> np.ndarray:
    """Degenerate scene: every particle at the same position."""
    rows = uniform_particles(n, seed)
    rows[:, POS] = np.asarray(point, dtype=np.float32)
    return rows

