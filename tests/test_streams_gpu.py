"""Work in flight at once on separate streams, each call with its own device
arrays and workspace, every result compared with the oracle.  Builds go
through grid_build_host (pinned host records in, destino and inicios back),
one scene per build plan (cluster, sparse, bucketed, its atomic fallback);
multi-array gathers cover both forms of grid_reorder_many.  The library keeps
per-device launch settings across calls; this checks that concurrent calls
on several streams do not disturb one another."""
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


def test_multi_array_gathers_on_several_streams(ug, oracle_lib):
    """grid_reorder_many calls of both TMA slot sizes (records up to 32 bytes,
    and up to 64) and of the plain kernel (a wider record), all in flight at
    once on their own streams, each against the oracle."""
    widths = [[4, 4], [12, 8], [20], [16, 4, 4], [4], [8, 12]]
    jobs = []
    for k, w in enumerate(widths):
        n = 50_000 + 977 * k
        rng = np.random.default_rng(70 + k)
        ordenado = rng.permutation(n).astype(np.uint32)
        hosts = [rng.integers(0, 2**32, (n, c), dtype=np.uint64).astype(np.uint32) for c in w]
        p = ug.make_params(n, (8, 8, 8), (0, 0, 0), 1.0)
        jobs.append({"ordenado": ordenado, "hosts": hosts, "p": p, "stream": torch.cuda.Stream(),
                     "dev_ord": torch.from_numpy(ordenado.view(np.int32)).cuda(),
                     "srcs": [torch.from_numpy(h).cuda() for h in hosts],
                     "ws": torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")})
        jobs[-1]["dsts"] = [torch.empty_like(t) for t in jobs[-1]["srcs"]]
    torch.cuda.synchronize()
    for j in jobs:
        ug.grid_reorder_many(j["dev_ord"], list(zip(j["srcs"], j["dsts"])), j["ws"], j["p"], j["stream"])
    torch.cuda.synchronize()
    for j in jobs:
        assert ug.grid_status(j["ws"]) == 0
        for h, d in zip(j["hosts"], j["dsts"]):
            assert np.array_equal(d.cpu().numpy(), oracle_lib.reorder_records(j["ordenado"], h))
