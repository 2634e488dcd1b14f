"""Seeded scene generator: determinism, shapes and the stated distributions (no GPU)."""
import numpy as np

from uniform_grid_particle_gb300 import scenes


def test_uniform_scene_fields_and_determinism():
    a = scenes.uniform_particles(50_000, 123)
    b = scenes.uniform_particles(50_000, 123)
    assert a.dtype == np.float32 and a.shape == (50_000, 8) and a.flags.c_contiguous
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert not np.array_equal(a, scenes.uniform_particles(50_000, 124))
    pos = a[:, scenes.POS]
    assert pos.min() >= -5.0 and pos.max() < 5.0
    assert abs(float(pos.mean())) < 0.05
    assert a[:, scenes.VIDA].min() >= 1.0 and a[:, scenes.VIDA].max() < 4.0
    assert not a[:, scenes.VEL].any()
    assert a[:, scenes.MASA].min() >= 0.5 and a[:, scenes.MASA].max() < 1.5


def test_contention_scene_structure():
    n = 100_000
    rows = scenes.contention_particles(n, 7, 128)
    pos = rows[:, scenes.POS]
    centre = np.float32(0.0390625)
    hot = np.all(pos == centre, axis=1)
    assert hot.sum() == n // 100
    # hot particles are spread through the array, not in one block
    idx = np.nonzero(hot)[0]
    assert idx.min() < n // 10 and idx.max() > n - n // 10
    outside = np.any(np.abs(pos) >= 5.0, axis=1)
    assert 0.5 * (n // 100) < outside.sum() < 1.2 * (n // 100)
    gauss = pos[~hot & ~np.any(np.abs(pos) > 5.0, axis=1)]
    assert abs(float(gauss.std()) - 1.0) < 0.05


def test_scene_table():
    s = scenes.SCENES
    assert [s[k].n for k in ("tiny", "scan_dominated", "headline", "contention", "stress")] == \
        [4096, 100_000, 1_000_000, 1_000_000, 16_777_216]
    assert s["headline"].cells == 128 ** 3 and s["stress"].cells == 256 ** 3
    assert s["tiny"].cell_size == 0.625 and s["headline"].cell_size == 0.078125
    assert s["stress"].cell_size == 0.0390625 and s["stress"].builds == 10
