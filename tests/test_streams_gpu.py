"""Several builds in flight at once on separate streams, through
grid_build_host (pinned host records in, destino and inicios back), each with
its own device arrays and workspace: one scene per build plan (cluster,
sparse, bucketed, its atomic fallback), every result compared with the
oracle.  The library keeps per-device launch settings across calls; this
checks that concurrent calls on several streams do not disturb one another."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_matches_oracle
from uniform_grid_particle_gb300 import scenes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ug():
    from uniform_grid_particle_gb300 import build, ugrid

    build.build()
    assert torch.cuda.is_available()
    return ugrid


@pytest.mark.parametrize("rounds", [1, 3])
def test_scenes_on_several_streams(ug, oracle_lib, rounds):
    names = ["tiny", "scan_dominated", "headline", "contention"]
    jobs = []
    for k, name in enumerate(names * rounds):
        s = scenes.SCENES[name]
        stable = k % 2 == 1
        flags = ug.GRID_STABLE if stable else 0
        p = ug.make_params(s.n, s.dims, s.origin, s.cell_size)
        rows = s.particles()
        b = ug.GridBuffers.allocate(p, flags)
        job = {"scene": s, "rows": rows, "stable": stable, "p": p, "b": b, "stream": torch.cuda.Stream(),
               "host_in": torch.from_numpy(rows).pin_memory(),
               "host_dest": torch.empty((s.n, 8), dtype=torch.float32).pin_memory(),
               "host_inicios": torch.empty(s.cells + 1, dtype=torch.int32).pin_memory(),
               "dev_in": torch.empty((s.n, 8), dtype=torch.float32, device="cuda")}
        jobs.append(job)
    torch.cuda.synchronize()
    for j in jobs:  # every build enqueued before any is waited for
        b = j["b"]
        ug.grid_build_host(j["host_in"], j["host_dest"], j["host_inicios"], j["dev_in"], b.destino, b.conteos,
                           b.celdaDe, b.inicios, b.ordenado, b.ws, j["p"], ug.GRID_STABLE if j["stable"] else 0,
                           j["stream"])
    torch.cuda.synchronize()
    for j in jobs:
        s, b = j["scene"], j["b"]
        u32 = lambda t: t.cpu().numpy().view(np.uint32)  # noqa: E731
        got = {"status": ug.grid_status(b.ws), "conteos": u32(b.conteos), "celdaDe": u32(b.celdaDe),
               "inicios": j["host_inicios"].numpy().view(np.uint32), "ordenado": u32(b.ordenado),
               "destino": j["host_dest"].numpy()}
        ref = oracle_lib.build(j["rows"], s.dims, s.origin, s.cell_size)
        assert_matches_oracle(oracle_lib, j["rows"], got, ref, j["stable"])
