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


def test_build_kernel_labels_follow_the_library_limits():
    """bench.py names the kernel a scene's build launches from the plan
    limits of grid_build; those limits live in the library's internal header,
    so a change there must show up here."""
    import re

    hdr = open(os.path.join(ROOT, "uniform_grid_particle_gb300", "csrc", "ugrid_internal.cuh")).read()

    def const(name):
        return int(re.search(rf"constexpr \w+ {name} = (\d+);", hdr).group(1))

    bench = _bench()
    cl_n, cl_c = const("kClusterMaxParticles"), const("kClusterMaxCells")
    sm_n, sm_c = const("kSmallMaxParticles"), const("kSmallMaxCells")
    per_cta, cells_per = const("kSparseMaxParticlesPerCta"), const("kSparseCellsPerParticle")
    sms = 152
    k = bench.build_kernel
    assert k(cl_n, cl_c, False, sms) == "build_cluster_kernel"
    assert k(cl_n + 1, cl_c, False, sms) != "build_cluster_kernel"
    assert k(cl_n, cl_c + 1, False, sms) != "build_cluster_kernel"
    assert k(sm_n, sm_c, True, sms) == "build_small_kernel<true>"
    assert k(sm_n + 1, sm_c, True, sms) != "build_small_kernel<true>"
    n = 2 * sms * per_cta
    assert k(n, cells_per * n, False, sms) == "build_sparse_kernel<false>"
    assert k(n + 1, cells_per * (n + 1), False, sms) == "build_bucketed_kernel<false>"
    assert k(n, cells_per * n - 1, True, sms) == "build_bucketed_kernel<true>"
    assert k(1_000_000, 128 ** 3, False, sms) == "build_bucketed_kernel<false>"


def test_algorithmic_bytes_of_the_headline_step():
    """The roofline's byte count for one build of 1,000,000 particles on 128^3
    cells: two clears of the counters, the count (16 bytes of each record read,
    celdaDe written), the scan (counts read, C + 1 starts written), the scatter
    (celdaDe, a start and ordenado per particle) and the gather (ordenado, the
    32-byte record read and written)."""
    bench = _bench()
    n, cells = 1_000_000, 128 ** 3
    alg = bench.algorithmic_bytes(n, cells)
    want = {"clear": 4 * cells, "count": 20 * n, "scan": 8 * cells + 4, "clear_cursor": 4 * cells,
            "scatter": 12 * n, "gather": 68 * n}
    assert alg == want
    assert sum(alg.values()) == 133_554_436


def test_committed_traffic_is_used_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    """A DRAM-traffic line counts only while the hash of the kernel's sources
    matches; a changed source, or a kernel with no line, reports None."""
    import hashlib

    bench = _bench()
    sources = ["reorder.cu"]
    h = hashlib.sha256()
    with open(os.path.join(ROOT, "uniform_grid_particle_gb300", "csrc", "reorder.cu"), "rb") as fh:
        h.update(fh.read())
    good = tmp_path / "good.txt"
    good.write_text(f"# comment\nreorder.cu {h.hexdigest()} 12345\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(good))
    assert bench.kernel_traffic(sources) == 12345.0
    stale = tmp_path / "stale.txt"
    stale.write_text("reorder.cu " + "0" * 64 + " 12345\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(stale))
    assert bench.kernel_traffic(sources) is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(good))
    assert bench.kernel_traffic(["scan.cu"]) is None


def test_roofline_entry_arithmetic():
    """achieved = algorithmic bytes / step time; frac = achieved / peak; the
    committed traffic only for the headline scene's non-stable kernel."""
    bench = _bench()
    e = bench.roofline_entry(0, 133_554_436, 0.0395, 6763.3, "measured")
    assert abs(e["achieved"] - 133_554_436 / 39.5e-6 / 1e9) < 1e-9
    assert abs(e["frac"] - e["achieved"] / 6763.3) < 1e-12
    assert e["bound"] == "hbm" and e["unit"] == "GB/s" and e["kernel"] == "build_bucketed_kernel<false>"
    assert bench.roofline_entry(1, 133_554_436, 0.0417, 6763.3, "measured")["traffic"] is None
    other = bench.roofline_entry(0, 43_554_436, 0.0195, 6763.3, "measured", scene_name="scan_dominated",
                                 kernel="build_sparse_kernel<false>")
    assert other["traffic"] is None and other["kernel"] == "build_sparse_kernel<false>"
